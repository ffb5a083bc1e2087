/*
 * fp8bs.h -- C ABI of libfp8bs.so: FP8 quantization and scaled FP8 GEMM on one
 * NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (page title, section):
 *   "07 -- The FP8 Family: E4M3, E5M2, and Per-Block Scaling" ("The two
 *       shapes", "Scaling is what makes FP8 usable", "The scaling granularity
 *       ladder", "DeepSeek-V3: fp8 training in the wild");
 *   "FP8 Mixed-Precision Serving in Production ..." ("The Mathematics of FP8",
 *       "Quantization Granularity and Scaling Topologies", "Engineering
 *       Trade-Offs and Best Practices");
 *   "Low precision: FP8, FP4, and microscaling" (qdq_e4m3 listing,
 *       microscaling paragraphs, DeepSeek-V3 promotion paragraph).
 *
 * Conventions shared by every entry point
 *   - All pointers named *_dev are DEVICE pointers owned by the caller. The
 *     library never allocates, frees or synchronises; it enqueues kernels on
 *     `stream` (NULL = the legacy default stream) and returns.
 *   - Matrices are row-major. bf16 and fp8 elements are stored as raw bit
 *     patterns (uint16 / uint8). A GEMM operand pair is X [M x K] and
 *     W [N x K], both K-contiguous ("TN"); the output is Out = X W^T [M x N]
 *     bf16, row-major with leading dimension N.
 *   - Argument checks run on the host before any launch; a failed check
 *     returns a non-zero fp8_status_t and enqueues nothing. A CUDA error at
 *     launch returns FP8_ERR_CUDA. Every wait inside a kernel is bounded: on
 *     expiry the kernel stores FP8_ERR_TIMEOUT into *dev_status (when
 *     non-NULL), drains its own copies in flight, frees its tensor memory and
 *     returns; the caller zeroes *dev_status beforehand and reads it after the
 *     stream completes. The library writes *dev_status only on error.
 *   - An empty problem (a zero dimension) is valid and enqueues nothing.
 *   - Stream order holds as for ordinary launches. The block-scaled GEMM
 *     kernels are launched as programmatic dependent launches: they may be
 *     scheduled while the kernel ahead of them in the stream is finishing and
 *     do their setup then, but they read no input (operands or scales) and
 *     write no output before that kernel has completed.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *fp8_stream_t;

/* FP8 element formats ("07 -- The FP8 Family", format table and bit layout).
 * E4M3: bias 7, max 448, no infinities, NaN = S1111111.
 * E5M2: bias 15, max 57344, IEEE infinities and NaNs. */
typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_format_t;

/* Scaling granularity ("07 -- The FP8 Family", scaling granularity ladder;
 * "FP8 Mixed-Precision Serving", Quantization Granularity and Scaling
 * Topologies). Scale arrays, for an operand of [rows x cols]:
 *   TENSOR         float[1]
 *   TOKEN          float[rows]                      (one per row)
 *   TILE_1x128     float[cols/128][rows]            (rows contiguous)
 *   BLOCK_128x128  float[ceil(rows/128)][cols/128]
 *   MX32           uint8 UE8M0 (2^(b-127)), one per 32 consecutive elements
 *                  of a row, in the layout chosen by fp8_sf_layout_t.
 *   CHANNEL        float[cols] (one per column: per-channel scales of a
 *                  [tokens x channels] tensor such as a K or V cache -- "FP8
 *                  Serving" guide, Things to try; "FP8 Mixed-Precision
 *                  Serving", FP8 KV Cache). Quantize/dequantize only; not a
 *                  GEMM operand granularity (it does not factor out of a K sum). */
typedef enum {
  FP8_GRAN_TENSOR = 0,
  FP8_GRAN_TOKEN = 1,
  FP8_GRAN_TILE_1x128 = 2,
  FP8_GRAN_BLOCK_128x128 = 3,
  FP8_GRAN_MX32 = 4,
  FP8_GRAN_CHANNEL = 5
} fp8_gran_t;

/* MX scale-factor layouts.
 *   LINEAR   uint8[rows][cols/32].
 *   TCGEN05  the tiled layout the tensor-core block-scaled MMA consumes
 *            ("Low precision", microscaling: "a scale-factor tensor in its
 *            required tiled layout"): rows cut into blocks of 128, the
 *            32-element groups into blocks of 4; each 128x4 block is 512
 *            bytes, blocks row-block-major; inside a block the byte of
 *            (row r, group j) is at (r%32)*16 + ((r%128)/32)*4 + (j%4).
 *            Size: ceil(rows/128) * ceil(cols/128) * 512 bytes; padding bytes
 *            are written as 0.
 *   TCGEN05_X4  (MX-32 only) the TCGEN05 layout with each 512-byte block
 *            stored four times in a row (2048 bytes per block; block b's
 *            copies at 2048*b + 512*i, i = 0..3). A layout of this library,
 *            not of the pages: the GEMM moves such blocks into tensor memory
 *            with fewer, wider copies (fp8_gemm_mx_x4). Size: 4 times
 *            TCGEN05's. */
typedef enum { FP8_SF_LINEAR = 0, FP8_SF_TCGEN05 = 1, FP8_SF_TCGEN05_X4 = 2 } fp8_sf_layout_t;

typedef enum {
  FP8_OK = 0,
  FP8_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, bad combination      */
  FP8_ERR_ALIGNMENT = 2,         /* pointer or leading dimension misaligned      */
  FP8_ERR_UNSUPPORTED_SHAPE = 3, /* dimension rule violated (no fallback path)   */
  FP8_ERR_WORKSPACE = 4,         /* workspace missing or too small               */
  FP8_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed            */
  FP8_ERR_TIMEOUT = 6            /* written to *dev_status by an expired wait    */
} fp8_status_t;

/* Human-readable name of a status code (static storage, never NULL). */
const char *fp8_status_string(fp8_status_t status);

/* Bytes of the scale array fp8_quantize writes for this shape, or 0 for an
 * invalid combination. */
size_t fp8_scales_bytes(int64_t rows, int64_t cols, fp8_gran_t gran, fp8_sf_layout_t sf_layout);

/* Workspace bytes fp8_quantize needs: 256 for dynamic per-tensor scaling (the
 * grid-wide amax of the first pass lives there), cols*4 rounded up to 256 for
 * per-channel scaling (the column maxima of the first pass), 0 otherwise. */
size_t fp8_quantize_workspace_bytes(int64_t rows, int64_t cols, fp8_gran_t gran);

/* Dynamic (or static per-tensor) quantization of a bf16 matrix.
 *   "07 -- The FP8 Family", Scaling is what makes FP8 usable: x_fp8 =
 *   clip(round(x/s)); "FP8 Mixed-Precision Serving", per-tensor static, current
 *   scaling and block-wise scaling: s = max|X_group| / V_max; "Low precision",
 *   qdq_e4m3 listing: multiply by 1/s, round to nearest even, saturate.
 * Per group: amax = max |x|; s = fp32(amax / V_max) with V_max = 448 (E4M3) or
 * 57344 (E5M2); s_inv = fp32(1 / s), replaced by 0 when s == 0 or 1/s is not
 * finite; q = RNE_satfinite(fp32(x * s_inv)). MX32: e = ceil(log2(fp32(amax /
 * V_max))) clamped to [-127, 127] (-127 for amax 0), byte = e + 127, q =
 * RNE_satfinite(x * 2^-e). TENSOR with static_scale_dev != NULL uses s =
 * *static_scale_dev (calibrated scaling) and copies it to scales_out.
 *   x_dev        bf16 [rows x cols], leading dimension ld_x (elements)
 *   q_dev        fp8 out [rows x cols], leading dimension ld_q (bytes)
 *   scales_dev   out, fp8_scales_bytes(rows, cols, gran, sf_layout) bytes
 *   workspace    device scratch of fp8_quantize_workspace_bytes() bytes
 *                (may be NULL when that is 0); its contents are clobbered;
 *                concurrent calls must not share it.
 * Shape rules: cols % 16 == 0 (TENSOR, TOKEN, CHANNEL), cols % 128 == 0 (TILE_1x128,
 * BLOCK_128x128), cols % 32 == 0 (MX32); rows <= 65535 * 128 for BLOCK_128x128
 * (one CTA per block, row blocks in the grid's y dimension); other dimensions
 * below 2^31. x_dev and q_dev 16-byte aligned,
 * ld_x % 8 == 0, ld_q % 16 == 0, scales_dev 4-byte aligned. */
fp8_status_t fp8_quantize(const void *x_dev, int64_t rows, int64_t cols, int64_t ld_x, fp8_format_t fmt,
                          fp8_gran_t gran, fp8_sf_layout_t sf_layout, const float *static_scale_dev, void *q_dev,
                          int64_t ld_q, void *scales_dev, void *workspace_dev, size_t workspace_bytes,
                          fp8_stream_t stream);

/* Dynamic per-tensor quantization that allocates nothing and takes no
 * workspace. The pages have no counterpart to this entry point; it exists for
 * callers that cannot call cudaMalloc -- code inside a host framework that owns
 * all device memory (a fixed arena with no allocator exposed to plugins), or a
 * latency-critical path where cudaMalloc's implicit device synchronisation is
 * not acceptable.
 * Computes exactly what fp8_quantize computes for FP8_GRAN_TENSOR without a
 * static scale (same kernels, same results): q_dev [rows x cols] (ld_q bytes)
 * and the single fp32 scale in *scale_dev.
 * Scratch: the grid-wide amax lives in a 256-byte static device array inside
 * the library (every GPU that loads the library holds it until the process
 * exits). A call whose scratch need (fp8_quantize_workspace_bytes for
 * FP8_GRAN_TENSOR) exceeds those 256 bytes is refused with FP8_ERR_WORKSPACE.
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture. Every call clears the amax word before it starts, but all calls
 * share the array: calls whose kernels overlap on the GPU (unordered streams)
 * race and must be serialised by the caller.
 * No cudaMalloc, cudaFree or other allocating routine is called.
 * Shape and alignment rules as fp8_quantize with FP8_GRAN_TENSOR. */
fp8_status_t fp8_quantize_tensor_noalloc(const void *x_dev, int64_t rows, int64_t cols, int64_t ld_x,
                                         fp8_format_t fmt, void *q_dev, int64_t ld_q, float *scale_dev,
                                         fp8_stream_t stream);

/* Per-tensor quantization with delayed scaling ("FP8 Mixed-Precision Serving",
 * Delayed Scaling: rho = FP8MaxValue / (2^m * max(H)) over a rolling amax
 * history H; "Low precision", NVIDIA's taxonomy: per-tensor, delayed). One
 * pass over x instead of current scaling's two.
 *   amax_history_dev  float[history_len] in device memory, owned by the caller,
 *                     initialised to 0 (entries must be >= 0).
 * The scale is s = fp32(fp32(2^margin * max(H)) / V_max) and x is encoded as
 * RNE_satfinite(x * fp32(1/s)) (values beyond the history's range saturate);
 * a history whose maximum is 0 or that holds inf/NaN gives s = 1. s goes to
 * *scale_dev; afterwards history[slot] = amax(x) (the caller advances slot by
 * one per step, modulo history_len). Rules: 0 <= slot < history_len,
 * -126 <= margin <= 127, shape and alignment as fp8_quantize with
 * FP8_GRAN_TENSOR. Two kernels, no workspace. */
fp8_status_t fp8_quantize_delayed(const void *x_dev, int64_t rows, int64_t cols, int64_t ld_x, fp8_format_t fmt,
                                  float *amax_history_dev, int32_t history_len, int32_t slot, int32_t margin,
                                  void *q_dev, int64_t ld_q, float *scale_dev, fp8_stream_t stream);

/* Dequantization ("07 -- The FP8 Family": x_hat = x_fp8 * s; "Low precision",
 * qdq_e4m3 listing: exact decode, then one fp32 multiply by s):
 * out = bf16_RN(fp32(decode(q) * s)). Same layouts and rules as fp8_quantize;
 * out_dev bf16 [rows x cols] with leading dimension ld_out (elements, % 8). */
fp8_status_t fp8_dequantize(const void *q_dev, int64_t rows, int64_t cols, int64_t ld_q, fp8_format_t fmt,
                            fp8_gran_t gran, fp8_sf_layout_t sf_layout, const void *scales_dev, void *out_dev,
                            int64_t ld_out, fp8_stream_t stream);

/* Scaled FP8 GEMM with fp32 accumulation and bf16 output
 * ("07 -- The FP8 Family", Scaling is what makes FP8 usable:
 *  Out = (X_fp8 s_X)(W_fp8 s_W)^T = s_X s_W (X_fp8 W_fp8^T) in fp32).
 * Valid (a_gran, b_gran) pairs:
 *   (TILE_1x128, BLOCK_128x128)  DeepSeek-V3 fine-grained scaling ("07 -- The
 *       FP8 Family", DeepSeek-V3 callout; "Low precision", promotion paragraph):
 *       every 128-wide K chunk's tensor-core partial is multiplied by
 *       s_X[m, kb] * s_W[n/128, kb] and added to an fp32 accumulator. K % 128 == 0.
 *   (TENSOR | TOKEN, TENSOR | TOKEN)  per-tensor, per-token activation and
 *       per-channel weight scales (TOKEN on W = one scale per output column):
 *       the whole K sum accumulates in the tensor core and the scale product is
 *       applied once in the epilogue. K % 16 == 0.
 * a_dev: X fp8 [M x K]; b_dev: W fp8 [N x K]; out_dev: bf16 [M x N].
 * Rules: M >= 1, N % 16 == 0 ("FP8 Mixed-Precision Serving", hardware-aligned
 * sizing: multiples of 16, no slower fallback), M, N, K < 2^31; a_dev, b_dev,
 * out_dev 16-byte aligned; scales 4-byte aligned. a_fmt / b_fmt may differ.
 * dev_status: NULL or a device int (see conventions). */
fp8_status_t fp8_gemm_blockscaled(const void *a_dev, const float *a_scales_dev, fp8_gran_t a_gran,
                                  const void *b_dev, const float *b_scales_dev, fp8_gran_t b_gran,
                                  fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev, int64_t M, int64_t N,
                                  int64_t K, int *dev_status, fp8_stream_t stream);

/* The block-scaled GEMM (1x128 activation tiles x 128x128 weight blocks) with
 * quantization fused into its epilogue ("Low precision", practice 4: fuse
 * quantization into the producing kernel's epilogue -- the per-block amax and
 * scaling run on data already in registers instead of costing a separate pass
 * over HBM). Each 128-column group of an output row is rounded to bf16 (the
 * value fp8_gemm_blockscaled would store), then quantized exactly as
 * fp8_quantize does with FP8_GRAN_TILE_1x128: q_out_dev uint8 [M x N] codes in
 * out_fmt and q_scales_dev float [N/128][M] -- the next layer's activation
 * operand. No bf16 output is written. Rules: K % 128 == 0, N % 128 == 0, other
 * rules as fp8_gemm_blockscaled. */
fp8_status_t fp8_gemm_blockscaled_quantized_out(const void *a_dev, const float *a_scales_dev, const void *b_dev,
                                                const float *b_scales_dev, fp8_format_t a_fmt, fp8_format_t b_fmt,
                                                fp8_format_t out_fmt, void *q_out_dev, float *q_scales_dev,
                                                int64_t M, int64_t N, int64_t K, int *dev_status,
                                                fp8_stream_t stream);

/* MXFP8 GEMM on the tensor core's block-scaled MMA ("Low precision",
 * microscaling: 32 consecutive elements share one UE8M0 scale, applied inside
 * the tensor core). Out[m][n] = sum_k decode(a[m][k]) 2^(sfa(m,k/32)-127)
 * decode(b[n][k]) 2^(sfb(n,k/32)-127), fp32 accumulation over all of K, bf16
 * out. a_sf_dev / b_sf_dev are in the FP8_SF_TCGEN05 layout for [M x K] and
 * [N x K]. Rules: K % 32 == 0, N % 16 == 0, M >= 1, alignment as above. */
fp8_status_t fp8_gemm_mx(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev, const uint8_t *b_sf_dev,
                         fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev, int64_t M, int64_t N, int64_t K,
                         int *dev_status, fp8_stream_t stream);

/* fp8_gemm_mx with a_sf_dev / b_sf_dev in the FP8_SF_TCGEN05_X4 layout (as
 * fp8_quantize writes it for FP8_GRAN_MX32): the same product, bit for bit;
 * each stage's scale blocks reach tensor memory in two copies instead of
 * three. Same rules as fp8_gemm_mx. */
fp8_status_t fp8_gemm_mx_x4(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev, const uint8_t *b_sf_dev,
                            fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev, int64_t M, int64_t N, int64_t K,
                            int *dev_status, fp8_stream_t stream);

/* ------------------------------------------------------------------ NVFP4
 * "Low precision: FP8, FP4, and microscaling" (NVFP4 paragraph): blocks of 16
 * elements, an E4M3 microscale per block and one fp32 scale per tensor that
 * keeps the microscales inside E4M3's range. The page prints neither the FP4
 * element format nor the scale arithmetic; this library takes:
 *   element: FP4 E2M1 (the OCP Microscaling element format the page cites):
 *     sign, 2 exponent bits (bias 1), 1 mantissa bit; +-{0,0.5,1,1.5,2,3,4,6};
 *     round to nearest even, saturating at +-6; codes packed two per byte,
 *     element 2i in the low nibble of byte i of its row;
 *   s_t = fp32(amax_tensor / 2688)  (2688 = 6 * 448; 1 when that is 0 or not
 *     finite);
 *   per block of 16 consecutive elements of a row:
 *     s_b = E4M3(fp32(fp32(amax_block / 6) / s_t))   (stored as its E4M3 code),
 *     S = fp32(s_b * s_t), S_inv = fp32(1 / S) (0 if S = 0 or 1/S not finite),
 *     q = E2M1(fp32(x * S_inv));
 *   value: decode(q) * s_b * s_t.
 * Block scales (uint8 E4M3 codes, one per 16 elements): FP8_SF_LINEAR =
 * uint8[rows][cols/16]; FP8_SF_TCGEN05 = the 128x4-atom layout described above
 * for MX, with cols/16 groups per row (each atom covers 64 elements of K);
 * padding bytes are 0. */

/* Bytes of the NVFP4 block-scale array for [rows x cols], or 0 if invalid. */
size_t fp8_nvfp4_scales_bytes(int64_t rows, int64_t cols, fp8_sf_layout_t sf_layout);

/* Quantize bf16 [rows x cols] (leading dimension ld_x elements) to NVFP4.
 * q_out_dev: uint8 [rows x cols/2], leading dimension ld_q bytes (>= cols/2,
 * multiple of 8). sf_out_dev: fp8_nvfp4_scales_bytes bytes. tensor_scale_out_dev:
 * one device float, s_t. static_tensor_scale_dev: NULL (s_t from this tensor's
 * amax: two passes, workspace of fp8_quantize_workspace_bytes(rows, cols,
 * FP8_GRAN_TENSOR) bytes) or a device float used as s_t (one pass, no
 * workspace). Rules: cols % 16 == 0; x_dev 16-byte aligned, ld_x % 8 == 0;
 * q_out_dev 8-byte aligned. */
fp8_status_t fp8_quantize_nvfp4(const void *x_dev, int64_t rows, int64_t cols, int64_t ld_x,
                                fp8_sf_layout_t sf_layout, const float *static_tensor_scale_dev, void *q_out_dev,
                                int64_t ld_q, void *sf_out_dev, float *tensor_scale_out_dev, void *workspace_dev,
                                size_t workspace_bytes, fp8_stream_t stream);

/* out = bf16(fp32(decode(q) * fp32(s_b * s_t))), bf16 [rows x cols], leading
 * dimension ld_out elements (multiple of 8, out 16-byte aligned). Same q and
 * scale layouts as fp8_quantize_nvfp4; tensor_scale_dev: device float s_t. */
fp8_status_t fp8_dequantize_nvfp4(const void *q_dev, int64_t rows, int64_t cols, int64_t ld_q,
                                  fp8_sf_layout_t sf_layout, const void *sf_dev, const float *tensor_scale_dev,
                                  void *out_dev, int64_t ld_out, fp8_stream_t stream);

/* NVFP4 GEMM on the tensor core's block-scaled MMA
 * (tcgen05.mma kind::mxf4nvf4.block_scale.scale_vec::4X): Out[m][n] =
 * a_ts * b_ts * sum_k E2M1(a[m][k]) s_b(a; m, k/16) E2M1(b[n][k]) s_b(b; n, k/16),
 * fp32 accumulation over all of K, bf16 out [M x N]. a_dev [M x K/2] and
 * b_dev [N x K/2] packed codes (leading dimension K/2 bytes); a_sf_dev /
 * b_sf_dev block scales in the FP8_SF_TCGEN05 layout; a_ts_dev / b_ts_dev the
 * device fp32 tensor scales. Rules: K % 256 == 0, N % 16 == 0; a_dev, b_dev,
 * out_dev, a_sf_dev, b_sf_dev 16-byte aligned. dev_status as above. */
fp8_status_t fp8_gemm_nvfp4(const void *a_dev, const void *a_sf_dev, const float *a_ts_dev, const void *b_dev,
                            const void *b_sf_dev, const float *b_ts_dev, void *out_dev, int64_t M, int64_t N,
                            int64_t K, int *dev_status, fp8_stream_t stream);

/* Codec check (no counterpart on the pages beyond the element step itself):
 * out[i] = RNE_satfinite(x[i]) in `fmt`, computed by the same device routine
 * the quantizers use for their last step ("Low precision", qdq_e4m3 listing:
 * cvt.rn.satfinite), so that every fp32 input can be compared with a
 * reference encoder. x_dev fp32 [n] (16-byte aligned), out_dev uint8 [n]
 * (8-byte aligned), n % 8 == 0. */
fp8_status_t fp8_debug_encode_f32(const float *x_dev, int64_t n, fp8_format_t fmt, void *out_dev,
                                  fp8_stream_t stream);

/* fp8_gemm_mx on a chosen kernel, whatever the shape rule would pick:
 * _pairs the CTA-pair kernel (tcgen05 cta_group::2, 256 x 256 tiles over a
 * cluster of two CTAs, each CTA staging its own halves of the operands),
 * _single the single-CTA kernel (128 x 256 tiles). Same arguments, layouts and
 * rules as fp8_gemm_mx ("Low precision: FP8, FP4, and microscaling",
 * microscaling paragraph); bit-identical results are not promised between
 * them (the accumulation order inside the tensor core may differ), each is
 * within the GEMM tolerance. */
fp8_status_t fp8_debug_gemm_mx_pairs(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev,
                                     const uint8_t *b_sf_dev, fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev,
                                     int64_t M, int64_t N, int64_t K, int *dev_status, fp8_stream_t stream);
fp8_status_t fp8_debug_gemm_mx_single(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev,
                                      const uint8_t *b_sf_dev, fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev,
                                      int64_t M, int64_t N, int64_t K, int *dev_status, fp8_stream_t stream);

/* fp8_gemm_blockscaled with 1x128 / 128x128 scales on the CTA-pair kernel
 * (tcgen05 cta_group::2, 256 x 256 tiles over a cluster of two CTAs) whatever
 * the shape: the kernel the library keeps for shapes it may suit but does not
 * select by default (it measured 2 % slower than the single-CTA kernel on the
 * prefill shapes). Same arguments and rules as fp8_gemm_blockscaled with
 * a_gran = TILE_1x128, b_gran = BLOCK_128x128. */
fp8_status_t fp8_debug_gemm_blockscaled_pairs(const void *a_dev, const float *a_scales_dev, const void *b_dev,
                                              const float *b_scales_dev, fp8_format_t a_fmt, fp8_format_t b_fmt,
                                              void *out_dev, int64_t M, int64_t N, int64_t K, int *dev_status,
                                              fp8_stream_t stream);

/* Codec check for NVFP4's element step (same role as fp8_debug_encode_f32):
 * out[i] = the E2M1 code (low 4 bits of byte i) of x[i], rounded to nearest
 * even and saturated at +-6 by the device routine fp8_quantize_nvfp4 uses.
 * x_dev fp32 [n] (16-byte aligned), out_dev uint8 [n] (8-byte aligned),
 * n % 8 == 0. */
fp8_status_t fp8_debug_encode_e2m1_f32(const float *x_dev, int64_t n, void *out_dev, fp8_stream_t stream);

/* Check of the bounded-wait machinery the GEMM kernels use (no counterpart on
 * the pages): launches one CTA that waits on a barrier nothing ever arrives
 * on, with a limit of timeout_ns nanoseconds; on expiry the kernel stores
 * FP8_ERR_TIMEOUT into *dev_status and returns, leaving the context usable.
 * timeout_ns must be in (0, 10^10]. */
fp8_status_t fp8_debug_wait_probe(int *dev_status, uint64_t timeout_ns, fp8_stream_t stream);

/* Checks of the GEMM kernels' timeout exit (no counterpart on the pages):
 * fp8_gemm_blockscaled and fp8_gemm_mx, same arguments and rules, run on the
 * single-CTA kernels only (no CTA-pair or split-K cluster kernel) with every
 * bounded wait inside the kernel limited to wait_ns nanoseconds instead of 2 s.
 * With a short limit a wait expires: the kernel writes FP8_ERR_TIMEOUT to
 * *dev_status, waits (with its own fixed limit) for its copies and MMAs in
 * flight, frees its tensor memory and returns; the output is then unspecified
 * and the context stays usable. dev_status must be non-NULL; wait_ns in
 * (0, 10^10]. */
fp8_status_t fp8_debug_gemm_blockscaled_wait_limit(const void *a_dev, const float *a_scales_dev, fp8_gran_t a_gran,
                                                   const void *b_dev, const float *b_scales_dev, fp8_gran_t b_gran,
                                                   fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev, int64_t M,
                                                   int64_t N, int64_t K, int *dev_status, uint64_t wait_ns,
                                                   fp8_stream_t stream);
fp8_status_t fp8_debug_gemm_mx_wait_limit(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev,
                                          const uint8_t *b_sf_dev, fp8_format_t a_fmt, fp8_format_t b_fmt,
                                          void *out_dev, int64_t M, int64_t N, int64_t K, int *dev_status,
                                          uint64_t wait_ns, fp8_stream_t stream);

/* Store checks (no counterpart on the pages; a stand-in for a memory checker):
 * a library built with -DFP8BS_CHECK (libfp8bs_check.so) checks, before every
 * plain global store of its kernels, that the store stays inside the extent the
 * call's shape gives the buffer; a store outside it is skipped and the first one
 * is recorded as (source line << 40) | (element offset & (2^40 - 1)). (TMA
 * stores are clipped to their tensor maps by the hardware.) fp8_debug_oob_read
 * synchronises the current device, returns the record (0: no violation) and
 * clears it; in the normal build its kernels carry no checks and it returns 0.
 * fp8_debug_checked_build returns 1 for the checked build, else 0. */
uint64_t fp8_debug_oob_read(void);
int fp8_debug_checked_build(void);

/* Number of kernel launches the library has enqueued since it was loaded
 * (all entry points, all devices); a diagnostic counter. */
uint64_t fp8_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */

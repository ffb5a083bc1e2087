// internal.h -- declarations shared by the translation units of libfp8bs.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8bs.h"

namespace fp8bs {

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Counts kernels enqueued by the library (diagnostic, see fp8_launch_count).
void note_launches(int n);

// Bounded-wait limit used by kernels (nanoseconds).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s: no legitimate wait comes close
constexpr uint64_t kDrainTimeoutNs = 200000000ull;  // 0.2 s for draining copies after an abort

// ----------------------------------------------------------------- quantize
fp8_status_t launch_quantize(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt, int gran,
                             int sf_layout, const float *static_scale, uint8_t *q, int64_t ld_q, void *scales,
                             void *workspace, cudaStream_t stream);

// Per-tensor quantization with its amax scratch in a static device array
// (no workspace argument, no allocation). Refuses scratch_needed beyond the
// array's capacity with FP8_ERR_WORKSPACE.
fp8_status_t launch_quantize_tensor_noalloc(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                                            uint8_t *q, int64_t ld_q, float *scale_out, size_t scratch_needed,
                                            cudaStream_t stream);
size_t noalloc_scratch_capacity();

fp8_status_t launch_quantize_delayed(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                                     float *history, int hlen, int slot, int margin, uint8_t *q, int64_t ld_q,
                                     float *scale_out, cudaStream_t stream);

fp8_status_t launch_encode_f32(const float *x, int64_t n, int fmt, uint8_t *out, cudaStream_t stream);

fp8_status_t launch_dequantize(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q, int fmt, int gran,
                               int sf_layout, const void *scales, uint16_t *out, int64_t ld_out,
                               cudaStream_t stream);

// ----------------------------------------------------------------- GEMMs
enum class EpiScale : int { kTensorTensor = 0, kTensorToken = 1, kTokenTensor = 2, kTokenToken = 3 };

// wait_ns: the kernels' bounded-wait limit (kWaitTimeoutNs in production; the
// timeout-exit check passes a short one). allow_clusters = false keeps to the
// single-CTA kernels (no CTA-pair or split-K cluster kernel).
fp8_status_t launch_gemm_fold(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb, int a_fmt,
                              int b_fmt, uint16_t *out, int64_t M, int64_t N, int64_t K, int *dev_status,
                              cudaStream_t stream, uint64_t wait_ns = kWaitTimeoutNs, bool allow_clusters = true);

fp8_status_t launch_gemm_fold_pairs(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb, int a_fmt,
                                    int b_fmt, uint16_t *out, int64_t M, int64_t N, int64_t K, int *dev_status,
                                    cudaStream_t stream);
fp8_status_t launch_gemm_fold_quantized(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb,
                                        int a_fmt, int b_fmt, int out_fmt, uint8_t *q_out, float *q_scales,
                                        int64_t M, int64_t N, int64_t K, int *dev_status, cudaStream_t stream);

fp8_status_t launch_gemm_epilogue_scaled(const uint8_t *a, const float *sa, bool a_token, const uint8_t *b,
                                         const float *sb, bool b_token, int a_fmt, int b_fmt, uint16_t *out,
                                         int64_t M, int64_t N, int64_t K, int *dev_status, cudaStream_t stream,
                                         uint64_t wait_ns = kWaitTimeoutNs);

// mode: 0 the shape rule, 1 the single-CTA kernel, 2 the CTA-pair kernel
fp8_status_t launch_gemm_mx(const uint8_t *a, const uint8_t *sfa, const uint8_t *b, const uint8_t *sfb, int a_fmt,
                            int b_fmt, uint16_t *out, int64_t M, int64_t N, int64_t K, int *dev_status,
                            cudaStream_t stream, uint64_t wait_ns = kWaitTimeoutNs, int mode = 0);

fp8_status_t launch_wait_probe(int *dev_status, uint64_t timeout_ns, cudaStream_t stream);

// amax pass of the per-tensor quantizers (cols % 8 == 0, 16-byte aligned rows)
fp8_status_t launch_amax(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, uint32_t *amax_bits,
                         cudaStream_t stream);

// NVFP4 (nvfp4.cu): codes [rows x cols/2] bytes, E4M3 block scales (tiled or
// linear [rows][cols/16]), fp32 tensor scale in device memory.
fp8_status_t launch_quantize_nvfp4(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, bool tiled,
                                   const float *static_ts, uint8_t *q, int64_t ld_q, uint8_t *sf, float *ts_out,
                                   uint32_t *amax_ws, cudaStream_t stream);
fp8_status_t launch_dequantize_nvfp4(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q, bool tiled,
                                     const uint8_t *sf, const float *ts, uint16_t *out, int64_t ld_out,
                                     cudaStream_t stream);
fp8_status_t launch_encode_e2m1(const float *x, int64_t n, uint8_t *out, cudaStream_t stream);
fp8_status_t launch_gemm_nvfp4(const uint8_t *a, const uint8_t *sfa, const float *ta, const uint8_t *b,
                               const uint8_t *sfb, const float *tb, uint16_t *out, int64_t M, int64_t N, int64_t K,
                               int *dev_status, cudaStream_t stream);

// Store-check records of the FP8BS_CHECK build, one per translation unit
// (0 in the normal build): read and cleared.
uint64_t oob_record_quantize();
uint64_t oob_record_nvfp4();
uint64_t oob_record_gemm();

// 2-D tensor map over a row-major uint8 matrix [rows x cols] (cols contiguous,
// row stride ld bytes), box = box_cols x box_rows, 128-byte swizzle.
bool make_tmap_u8(void *tmap_out, const void *base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows,
                  uint32_t box_cols);
// The same over a row-major 16-bit matrix (bf16 output): ld in elements; the
// box's inner extent box_cols x 2 bytes must be at most 128 bytes.
bool make_tmap_u16(void *tmap_out, const void *base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows,
                   uint32_t box_cols);
// The same over a row-major fp32 matrix, unswizzled (scale vectors): ld in
// elements, a multiple of 4; the box's inner extent box_cols x 4 bytes a
// multiple of 16; elements outside the matrix read as zero.
bool make_tmap_f32(void *tmap_out, const void *base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows,
                   uint32_t box_cols);

}  // namespace fp8bs

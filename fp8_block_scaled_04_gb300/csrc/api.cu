// api.cu -- the C ABI of libfp8bs: argument checks on the host, then a launch
// on the caller's stream. Nothing here allocates, frees or synchronises.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "fp8bs.h"
#include "internal.h"

namespace fp8bs {

namespace {
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool valid_fmt(int f) { return f == FP8_E4M3 || f == FP8_E5M2; }
bool valid_gran(int g) { return g >= FP8_GRAN_TENSOR && g <= FP8_GRAN_CHANNEL; }
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
constexpr int64_t kMaxBlockRows = int64_t{65535} * 128;  // FP8_GRAN_BLOCK_128x128
}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < kMaxDevices) {
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int sms = 1;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms < 1) sms = 1;
  if (dev < kMaxDevices) g_sm_count[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

static bool make_tmap_2d(void *tmap_out, CUtensorMapDataType dtype, uint32_t elem_bytes, const void *base,
                        uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows, uint32_t box_cols,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(static_cast<CUtensorMap *>(tmap_out), dtype, 2, const_cast<void *>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_u8(void *tmap_out, const void *base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows,
                  uint32_t box_cols) {
  return make_tmap_2d(tmap_out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, ld, box_rows, box_cols);
}

bool make_tmap_u16(void *tmap_out, const void *base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows,
                   uint32_t box_cols) {
  return make_tmap_2d(tmap_out, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, rows, cols, ld, box_rows, box_cols);
}

bool make_tmap_f32(void *tmap_out, const void *base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows,
                   uint32_t box_cols) {
  return make_tmap_2d(tmap_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, rows, cols, ld, box_rows, box_cols,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" {

const char *fp8_status_string(fp8_status_t s) {
  switch (s) {
    case FP8_OK: return "FP8_OK";
    case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG";
    case FP8_ERR_ALIGNMENT: return "FP8_ERR_ALIGNMENT";
    case FP8_ERR_UNSUPPORTED_SHAPE: return "FP8_ERR_UNSUPPORTED_SHAPE";
    case FP8_ERR_WORKSPACE: return "FP8_ERR_WORKSPACE";
    case FP8_ERR_CUDA: return "FP8_ERR_CUDA";
    case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT";
    default: return "FP8_ERR_UNKNOWN";
  }
}

uint64_t fp8_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t fp8_debug_oob_read(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return ~0ull;
  const uint64_t r[3] = {oob_record_quantize(), oob_record_nvfp4(), oob_record_gemm()};
  for (uint64_t v : r)
    if (v != 0) return v;
  return 0;
}

int fp8_debug_checked_build(void) {
#ifdef FP8BS_CHECK
  return 1;
#else
  return 0;
#endif
}

size_t fp8_scales_bytes(int64_t rows, int64_t cols, fp8_gran_t gran, fp8_sf_layout_t sf_layout) {
  if (rows < 0 || cols < 0) return 0;
  switch (gran) {
    case FP8_GRAN_TENSOR: return sizeof(float);
    case FP8_GRAN_TOKEN: return static_cast<size_t>(rows) * sizeof(float);
    case FP8_GRAN_CHANNEL: return static_cast<size_t>(cols) * sizeof(float);
    case FP8_GRAN_TILE_1x128:
      return cols % 128 ? 0 : static_cast<size_t>(cols / 128) * static_cast<size_t>(rows) * sizeof(float);
    case FP8_GRAN_BLOCK_128x128:
      return cols % 128 ? 0 : static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>(cols / 128) * sizeof(float);
    case FP8_GRAN_MX32:
      if (cols % 32) return 0;
      if (sf_layout == FP8_SF_TCGEN05 || sf_layout == FP8_SF_TCGEN05_X4)
        return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((cols + 127) / 128) *
               (sf_layout == FP8_SF_TCGEN05 ? 512 : 2048);
      if (sf_layout == FP8_SF_LINEAR) return static_cast<size_t>(rows) * static_cast<size_t>(cols / 32);
      return 0;
    default: return 0;
  }
}

size_t fp8_quantize_workspace_bytes(int64_t rows, int64_t cols, fp8_gran_t gran) {
  (void)rows;
  if (gran == FP8_GRAN_TENSOR) return 256;
  if (gran == FP8_GRAN_CHANNEL && cols > 0) return (static_cast<size_t>(cols) * sizeof(float) + 255) / 256 * 256;
  return 0;
}

static fp8_status_t check_quant_shape(int64_t rows, int64_t cols, int gran) {
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return FP8_ERR_UNSUPPORTED_SHAPE;
  switch (gran) {
    case FP8_GRAN_TENSOR:
    case FP8_GRAN_TOKEN:
    case FP8_GRAN_CHANNEL: return cols % 16 ? FP8_ERR_UNSUPPORTED_SHAPE : FP8_OK;
    case FP8_GRAN_TILE_1x128: return cols % 128 ? FP8_ERR_UNSUPPORTED_SHAPE : FP8_OK;
    // one CTA per 128 x 128 block, row blocks in gridDim.y (at most 65535)
    case FP8_GRAN_BLOCK_128x128: return cols % 128 || rows > kMaxBlockRows ? FP8_ERR_UNSUPPORTED_SHAPE : FP8_OK;
    case FP8_GRAN_MX32: return cols % 32 ? FP8_ERR_UNSUPPORTED_SHAPE : FP8_OK;
    default: return FP8_ERR_INVALID_ARG;
  }
}

fp8_status_t fp8_quantize(const void *x_dev, int64_t rows, int64_t cols, int64_t ld_x, fp8_format_t fmt,
                          fp8_gran_t gran, fp8_sf_layout_t sf_layout, const float *static_scale_dev, void *q_dev,
                          int64_t ld_q, void *scales_dev, void *workspace_dev, size_t workspace_bytes,
                          fp8_stream_t stream) {
  if (!valid_fmt(fmt) || !valid_gran(gran)) return FP8_ERR_INVALID_ARG;
  if (sf_layout != FP8_SF_LINEAR &&
      !(gran == FP8_GRAN_MX32 && (sf_layout == FP8_SF_TCGEN05 || sf_layout == FP8_SF_TCGEN05_X4)))
    return FP8_ERR_INVALID_ARG;
  if (static_scale_dev != nullptr && gran != FP8_GRAN_TENSOR) return FP8_ERR_INVALID_ARG;
  fp8_status_t st = check_quant_shape(rows, cols, gran);
  if (st != FP8_OK) return st;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (x_dev == nullptr || q_dev == nullptr || scales_dev == nullptr) return FP8_ERR_INVALID_ARG;
  if (ld_x < cols || ld_q < cols) return FP8_ERR_INVALID_ARG;
  if (!aligned(x_dev, 16) || !aligned(q_dev, 16) || ld_x % 8 || ld_q % 16) return FP8_ERR_ALIGNMENT;
  if (!aligned(scales_dev, 4) || (static_scale_dev && !aligned(static_scale_dev, 4))) return FP8_ERR_ALIGNMENT;
  if ((gran == FP8_GRAN_TENSOR && static_scale_dev == nullptr) || gran == FP8_GRAN_CHANNEL) {
    if (workspace_dev == nullptr || workspace_bytes < fp8_quantize_workspace_bytes(rows, cols, gran))
      return FP8_ERR_WORKSPACE;
    if (!aligned(workspace_dev, 4)) return FP8_ERR_ALIGNMENT;
  }
  return launch_quantize(static_cast<const uint16_t *>(x_dev), rows, cols, ld_x, fmt, gran, sf_layout,
                         static_scale_dev, static_cast<uint8_t *>(q_dev), ld_q, scales_dev, workspace_dev,
                         reinterpret_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_quantize_tensor_noalloc(const void *x_dev, int64_t rows, int64_t cols, int64_t ld_x,
                                         fp8_format_t fmt, void *q_dev, int64_t ld_q, float *scale_dev,
                                         fp8_stream_t stream) {
  if (!valid_fmt(fmt)) return FP8_ERR_INVALID_ARG;
  fp8_status_t st = check_quant_shape(rows, cols, FP8_GRAN_TENSOR);
  if (st != FP8_OK) return st;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (x_dev == nullptr || q_dev == nullptr || scale_dev == nullptr) return FP8_ERR_INVALID_ARG;
  if (ld_x < cols || ld_q < cols) return FP8_ERR_INVALID_ARG;
  if (!aligned(x_dev, 16) || !aligned(q_dev, 16) || ld_x % 8 || ld_q % 16) return FP8_ERR_ALIGNMENT;
  if (!aligned(scale_dev, 4)) return FP8_ERR_ALIGNMENT;
  const size_t need = fp8_quantize_workspace_bytes(rows, cols, FP8_GRAN_TENSOR);
  if (need > noalloc_scratch_capacity()) return FP8_ERR_WORKSPACE;
  return launch_quantize_tensor_noalloc(static_cast<const uint16_t *>(x_dev), rows, cols, ld_x, fmt,
                                        static_cast<uint8_t *>(q_dev), ld_q, scale_dev, need,
                                        reinterpret_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_quantize_delayed(const void *x_dev, int64_t rows, int64_t cols, int64_t ld_x, fp8_format_t fmt,
                                  float *amax_history_dev, int32_t history_len, int32_t slot, int32_t margin,
                                  void *q_dev, int64_t ld_q, float *scale_dev, fp8_stream_t stream) {
  if (!valid_fmt(fmt)) return FP8_ERR_INVALID_ARG;
  if (history_len <= 0 || slot < 0 || slot >= history_len || margin < -126 || margin > 127) return FP8_ERR_INVALID_ARG;
  fp8_status_t st = check_quant_shape(rows, cols, FP8_GRAN_TENSOR);
  if (st != FP8_OK) return st;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (x_dev == nullptr || q_dev == nullptr || scale_dev == nullptr || amax_history_dev == nullptr)
    return FP8_ERR_INVALID_ARG;
  if (ld_x < cols || ld_q < cols) return FP8_ERR_INVALID_ARG;
  if (!aligned(x_dev, 16) || !aligned(q_dev, 16) || ld_x % 8 || ld_q % 16) return FP8_ERR_ALIGNMENT;
  if (!aligned(scale_dev, 4) || !aligned(amax_history_dev, 4)) return FP8_ERR_ALIGNMENT;
  return launch_quantize_delayed(static_cast<const uint16_t *>(x_dev), rows, cols, ld_x, fmt, amax_history_dev,
                                 history_len, slot, margin, static_cast<uint8_t *>(q_dev), ld_q, scale_dev,
                                 reinterpret_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_dequantize(const void *q_dev, int64_t rows, int64_t cols, int64_t ld_q, fp8_format_t fmt,
                            fp8_gran_t gran, fp8_sf_layout_t sf_layout, const void *scales_dev, void *out_dev,
                            int64_t ld_out, fp8_stream_t stream) {
  if (!valid_fmt(fmt) || !valid_gran(gran)) return FP8_ERR_INVALID_ARG;
  if (sf_layout != FP8_SF_LINEAR &&
      !(gran == FP8_GRAN_MX32 && (sf_layout == FP8_SF_TCGEN05 || sf_layout == FP8_SF_TCGEN05_X4)))
    return FP8_ERR_INVALID_ARG;
  fp8_status_t st = check_quant_shape(rows, cols, gran);
  if (st != FP8_OK) return st;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (q_dev == nullptr || out_dev == nullptr || scales_dev == nullptr) return FP8_ERR_INVALID_ARG;
  if (ld_q < cols || ld_out < cols) return FP8_ERR_INVALID_ARG;
  if (!aligned(q_dev, 16) || !aligned(out_dev, 16) || ld_q % 16 || ld_out % 8) return FP8_ERR_ALIGNMENT;
  if (!aligned(scales_dev, gran == FP8_GRAN_MX32 ? 1 : 4)) return FP8_ERR_ALIGNMENT;
  return launch_dequantize(static_cast<const uint8_t *>(q_dev), rows, cols, ld_q, fmt, gran, sf_layout, scales_dev,
                           static_cast<uint16_t *>(out_dev), ld_out, reinterpret_cast<cudaStream_t>(stream));
}

static fp8_status_t check_gemm_common(const void *a, const void *b, void *out, int64_t M, int64_t N, int64_t K,
                                      int a_fmt, int b_fmt) {
  if (!valid_fmt(a_fmt) || !valid_fmt(b_fmt)) return FP8_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (N % 16) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return FP8_OK;
  if (K == 0) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (a == nullptr || b == nullptr || out == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(out, 16)) return FP8_ERR_ALIGNMENT;
  return FP8_OK;
}

static fp8_status_t gemm_blockscaled_impl(const void *a_dev, const float *a_scales_dev, fp8_gran_t a_gran,
                                          const void *b_dev, const float *b_scales_dev, fp8_gran_t b_gran,
                                          fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev, int64_t M,
                                          int64_t N, int64_t K, int *dev_status, fp8_stream_t stream,
                                          uint64_t wait_ns, bool allow_clusters) {
  const bool fold = a_gran == FP8_GRAN_TILE_1x128 && b_gran == FP8_GRAN_BLOCK_128x128;
  const bool epi = (a_gran == FP8_GRAN_TENSOR || a_gran == FP8_GRAN_TOKEN) &&
                   (b_gran == FP8_GRAN_TENSOR || b_gran == FP8_GRAN_TOKEN);
  if (!fold && !epi) return FP8_ERR_INVALID_ARG;
  fp8_status_t st = check_gemm_common(a_dev, b_dev, out_dev, M, N, K, a_fmt, b_fmt);
  if (st != FP8_OK || M == 0 || N == 0) return st;
  if (fold ? (K % 128 != 0) : (K % 16 != 0)) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (a_scales_dev == nullptr || b_scales_dev == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(a_scales_dev, 4) || !aligned(b_scales_dev, b_gran == FP8_GRAN_TOKEN ? 16 : 4))
    return FP8_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return FP8_ERR_ALIGNMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fold)
    return launch_gemm_fold(static_cast<const uint8_t *>(a_dev), a_scales_dev, static_cast<const uint8_t *>(b_dev),
                            b_scales_dev, a_fmt, b_fmt, static_cast<uint16_t *>(out_dev), M, N, K, dev_status, s,
                            wait_ns, allow_clusters);
  return launch_gemm_epilogue_scaled(static_cast<const uint8_t *>(a_dev), a_scales_dev, a_gran == FP8_GRAN_TOKEN,
                                     static_cast<const uint8_t *>(b_dev), b_scales_dev, b_gran == FP8_GRAN_TOKEN,
                                     a_fmt, b_fmt, static_cast<uint16_t *>(out_dev), M, N, K, dev_status, s,
                                     wait_ns);
}

fp8_status_t fp8_gemm_blockscaled(const void *a_dev, const float *a_scales_dev, fp8_gran_t a_gran,
                                  const void *b_dev, const float *b_scales_dev, fp8_gran_t b_gran,
                                  fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev, int64_t M, int64_t N,
                                  int64_t K, int *dev_status, fp8_stream_t stream) {
  return gemm_blockscaled_impl(a_dev, a_scales_dev, a_gran, b_dev, b_scales_dev, b_gran, a_fmt, b_fmt, out_dev, M, N,
                               K, dev_status, stream, kWaitTimeoutNs, true);
}

fp8_status_t fp8_gemm_blockscaled_quantized_out(const void *a_dev, const float *a_scales_dev, const void *b_dev,
                                                const float *b_scales_dev, fp8_format_t a_fmt, fp8_format_t b_fmt,
                                                fp8_format_t out_fmt, void *q_out_dev, float *q_scales_dev,
                                                int64_t M, int64_t N, int64_t K, int *dev_status,
                                                fp8_stream_t stream) {
  if (!valid_fmt(out_fmt)) return FP8_ERR_INVALID_ARG;
  fp8_status_t st = check_gemm_common(a_dev, b_dev, q_out_dev, M, N, K, a_fmt, b_fmt);
  if (st != FP8_OK || M == 0 || N == 0) return st;
  if (K % 128 != 0 || N % 128 != 0) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (a_scales_dev == nullptr || b_scales_dev == nullptr || q_scales_dev == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(a_scales_dev, 4) || !aligned(b_scales_dev, 4) || !aligned(q_scales_dev, 4)) return FP8_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return FP8_ERR_ALIGNMENT;
  return launch_gemm_fold_quantized(static_cast<const uint8_t *>(a_dev), a_scales_dev,
                                    static_cast<const uint8_t *>(b_dev), b_scales_dev, a_fmt, b_fmt, out_fmt,
                                    static_cast<uint8_t *>(q_out_dev), q_scales_dev, M, N, K, dev_status,
                                    reinterpret_cast<cudaStream_t>(stream));
}

static fp8_status_t gemm_mx_impl(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev,
                                 const uint8_t *b_sf_dev, fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev,
                                 int64_t M, int64_t N, int64_t K, int *dev_status, fp8_stream_t stream,
                                 uint64_t wait_ns, int mode = 0) {
  fp8_status_t st = check_gemm_common(a_dev, b_dev, out_dev, M, N, K, a_fmt, b_fmt);
  if (st != FP8_OK || M == 0 || N == 0) return st;
  if (K % 32) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (a_sf_dev == nullptr || b_sf_dev == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(a_sf_dev, 16) || !aligned(b_sf_dev, 16)) return FP8_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return FP8_ERR_ALIGNMENT;
  return launch_gemm_mx(static_cast<const uint8_t *>(a_dev), a_sf_dev, static_cast<const uint8_t *>(b_dev), b_sf_dev,
                        a_fmt, b_fmt, static_cast<uint16_t *>(out_dev), M, N, K, dev_status,
                        reinterpret_cast<cudaStream_t>(stream), wait_ns, mode);
}

fp8_status_t fp8_gemm_mx(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev, const uint8_t *b_sf_dev,
                         fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev, int64_t M, int64_t N, int64_t K,
                         int *dev_status, fp8_stream_t stream) {
  return gemm_mx_impl(a_dev, a_sf_dev, b_dev, b_sf_dev, a_fmt, b_fmt, out_dev, M, N, K, dev_status, stream,
                      kWaitTimeoutNs);
}

fp8_status_t fp8_gemm_mx_x4(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev, const uint8_t *b_sf_dev,
                            fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev, int64_t M, int64_t N, int64_t K,
                            int *dev_status, fp8_stream_t stream) {
  return gemm_mx_impl(a_dev, a_sf_dev, b_dev, b_sf_dev, a_fmt, b_fmt, out_dev, M, N, K, dev_status, stream,
                      kWaitTimeoutNs, 3);
}

fp8_status_t fp8_debug_gemm_mx_pairs(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev,
                                     const uint8_t *b_sf_dev, fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev,
                                     int64_t M, int64_t N, int64_t K, int *dev_status, fp8_stream_t stream) {
  return gemm_mx_impl(a_dev, a_sf_dev, b_dev, b_sf_dev, a_fmt, b_fmt, out_dev, M, N, K, dev_status, stream,
                      kWaitTimeoutNs, 2);
}

fp8_status_t fp8_debug_gemm_mx_single(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev,
                                      const uint8_t *b_sf_dev, fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev,
                                      int64_t M, int64_t N, int64_t K, int *dev_status, fp8_stream_t stream) {
  return gemm_mx_impl(a_dev, a_sf_dev, b_dev, b_sf_dev, a_fmt, b_fmt, out_dev, M, N, K, dev_status, stream,
                      kWaitTimeoutNs, 1);
}

fp8_status_t fp8_debug_gemm_blockscaled_wait_limit(const void *a_dev, const float *a_scales_dev, fp8_gran_t a_gran,
                                                   const void *b_dev, const float *b_scales_dev, fp8_gran_t b_gran,
                                                   fp8_format_t a_fmt, fp8_format_t b_fmt, void *out_dev, int64_t M,
                                                   int64_t N, int64_t K, int *dev_status, uint64_t wait_ns,
                                                   fp8_stream_t stream) {
  if (dev_status == nullptr || wait_ns == 0 || wait_ns > 10000000000ull) return FP8_ERR_INVALID_ARG;
  return gemm_blockscaled_impl(a_dev, a_scales_dev, a_gran, b_dev, b_scales_dev, b_gran, a_fmt, b_fmt, out_dev, M, N,
                               K, dev_status, stream, wait_ns, false);
}

fp8_status_t fp8_debug_gemm_mx_wait_limit(const void *a_dev, const uint8_t *a_sf_dev, const void *b_dev,
                                          const uint8_t *b_sf_dev, fp8_format_t a_fmt, fp8_format_t b_fmt,
                                          void *out_dev, int64_t M, int64_t N, int64_t K, int *dev_status,
                                          uint64_t wait_ns, fp8_stream_t stream) {
  if (dev_status == nullptr || wait_ns == 0 || wait_ns > 10000000000ull) return FP8_ERR_INVALID_ARG;
  return gemm_mx_impl(a_dev, a_sf_dev, b_dev, b_sf_dev, a_fmt, b_fmt, out_dev, M, N, K, dev_status, stream,
                      wait_ns);
}

size_t fp8_nvfp4_scales_bytes(int64_t rows, int64_t cols, fp8_sf_layout_t sf_layout) {
  if (rows < 0 || cols < 0 || cols % 16 || rows > kMaxDim || cols > kMaxDim) return 0;
  const int64_t ng = cols / 16;
  if (sf_layout == FP8_SF_LINEAR) return static_cast<size_t>(rows * ng);
  if (sf_layout == FP8_SF_TCGEN05) return static_cast<size_t>(((rows + 127) / 128) * ((ng + 3) / 4) * 512);
  return 0;
}

fp8_status_t fp8_quantize_nvfp4(const void *x_dev, int64_t rows, int64_t cols, int64_t ld_x,
                                fp8_sf_layout_t sf_layout, const float *static_tensor_scale_dev, void *q_out_dev,
                                int64_t ld_q, void *sf_out_dev, float *tensor_scale_out_dev, void *workspace_dev,
                                size_t workspace_bytes, fp8_stream_t stream) {
  if (sf_layout != FP8_SF_LINEAR && sf_layout != FP8_SF_TCGEN05) return FP8_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim || cols % 16) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (x_dev == nullptr || q_out_dev == nullptr || sf_out_dev == nullptr || tensor_scale_out_dev == nullptr)
    return FP8_ERR_INVALID_ARG;
  if (ld_x < cols || ld_q < cols / 2) return FP8_ERR_INVALID_ARG;
  if (!aligned(x_dev, 16) || ld_x % 8 || !aligned(q_out_dev, 8) || ld_q % 8 || !aligned(tensor_scale_out_dev, 4))
    return FP8_ERR_ALIGNMENT;
  if (static_tensor_scale_dev != nullptr) {
    if (!aligned(static_tensor_scale_dev, 4)) return FP8_ERR_ALIGNMENT;
  } else {
    if (workspace_dev == nullptr || workspace_bytes < fp8_quantize_workspace_bytes(rows, cols, FP8_GRAN_TENSOR))
      return FP8_ERR_WORKSPACE;
    if (!aligned(workspace_dev, 4)) return FP8_ERR_ALIGNMENT;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool tiled = sf_layout == FP8_SF_TCGEN05;
  if (tiled && (rows % 128 || (cols / 16) % 4)) {
    // padding bytes of partial atoms are 0 (scale 0)
    if (cudaMemsetAsync(sf_out_dev, 0, fp8_nvfp4_scales_bytes(rows, cols, sf_layout), s) != cudaSuccess)
      return FP8_ERR_CUDA;
  }
  return launch_quantize_nvfp4(static_cast<const uint16_t *>(x_dev), rows, cols, ld_x, tiled,
                               static_tensor_scale_dev, static_cast<uint8_t *>(q_out_dev), ld_q,
                               static_cast<uint8_t *>(sf_out_dev), tensor_scale_out_dev,
                               static_cast<uint32_t *>(workspace_dev), s);
}

fp8_status_t fp8_dequantize_nvfp4(const void *q_dev, int64_t rows, int64_t cols, int64_t ld_q,
                                  fp8_sf_layout_t sf_layout, const void *sf_dev, const float *tensor_scale_dev,
                                  void *out_dev, int64_t ld_out, fp8_stream_t stream) {
  if (sf_layout != FP8_SF_LINEAR && sf_layout != FP8_SF_TCGEN05) return FP8_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim || cols % 16) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (q_dev == nullptr || sf_dev == nullptr || tensor_scale_dev == nullptr || out_dev == nullptr)
    return FP8_ERR_INVALID_ARG;
  if (ld_q < cols / 2 || ld_out < cols) return FP8_ERR_INVALID_ARG;
  if (!aligned(q_dev, 8) || ld_q % 8 || !aligned(out_dev, 16) || ld_out % 8 || !aligned(tensor_scale_dev, 4))
    return FP8_ERR_ALIGNMENT;
  return launch_dequantize_nvfp4(static_cast<const uint8_t *>(q_dev), rows, cols, ld_q,
                                 sf_layout == FP8_SF_TCGEN05, static_cast<const uint8_t *>(sf_dev), tensor_scale_dev,
                                 static_cast<uint16_t *>(out_dev), ld_out, reinterpret_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_gemm_nvfp4(const void *a_dev, const void *a_sf_dev, const float *a_ts_dev, const void *b_dev,
                            const void *b_sf_dev, const float *b_ts_dev, void *out_dev, int64_t M, int64_t N,
                            int64_t K, int *dev_status, fp8_stream_t stream) {
  fp8_status_t st = check_gemm_common(a_dev, b_dev, out_dev, M, N, K, FP8_E4M3, FP8_E4M3);
  if (st != FP8_OK || M == 0 || N == 0) return st;
  if (K % 256) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (a_sf_dev == nullptr || b_sf_dev == nullptr || a_ts_dev == nullptr || b_ts_dev == nullptr)
    return FP8_ERR_INVALID_ARG;
  if (!aligned(a_sf_dev, 16) || !aligned(b_sf_dev, 16) || !aligned(a_ts_dev, 4) || !aligned(b_ts_dev, 4))
    return FP8_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return FP8_ERR_ALIGNMENT;
  return launch_gemm_nvfp4(static_cast<const uint8_t *>(a_dev), static_cast<const uint8_t *>(a_sf_dev), a_ts_dev,
                           static_cast<const uint8_t *>(b_dev), static_cast<const uint8_t *>(b_sf_dev), b_ts_dev,
                           static_cast<uint16_t *>(out_dev), M, N, K, dev_status,
                           reinterpret_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_debug_encode_f32(const float *x_dev, int64_t n, fp8_format_t fmt, void *out_dev,
                                  fp8_stream_t stream) {
  if (!valid_fmt(fmt) || n < 0 || n % 8) return FP8_ERR_INVALID_ARG;
  if (n == 0) return FP8_OK;
  if (x_dev == nullptr || out_dev == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(x_dev, 16) || !aligned(out_dev, 8)) return FP8_ERR_ALIGNMENT;
  return launch_encode_f32(x_dev, n, fmt, static_cast<uint8_t *>(out_dev), reinterpret_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_debug_gemm_blockscaled_pairs(const void *a_dev, const float *a_scales_dev, const void *b_dev,
                                              const float *b_scales_dev, fp8_format_t a_fmt, fp8_format_t b_fmt,
                                              void *out_dev, int64_t M, int64_t N, int64_t K, int *dev_status,
                                              fp8_stream_t stream) {
  fp8_status_t st = check_gemm_common(a_dev, b_dev, out_dev, M, N, K, a_fmt, b_fmt);
  if (st != FP8_OK || M == 0 || N == 0) return st;
  if (K % 128 != 0) return FP8_ERR_UNSUPPORTED_SHAPE;
  if (a_scales_dev == nullptr || b_scales_dev == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(a_scales_dev, 4) || !aligned(b_scales_dev, 4)) return FP8_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return FP8_ERR_ALIGNMENT;
  return launch_gemm_fold_pairs(static_cast<const uint8_t *>(a_dev), a_scales_dev,
                                static_cast<const uint8_t *>(b_dev), b_scales_dev, a_fmt, b_fmt,
                                static_cast<uint16_t *>(out_dev), M, N, K, dev_status,
                                reinterpret_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_debug_encode_e2m1_f32(const float *x_dev, int64_t n, void *out_dev, fp8_stream_t stream) {
  if (n < 0 || n % 8) return FP8_ERR_INVALID_ARG;
  if (n == 0) return FP8_OK;
  if (x_dev == nullptr || out_dev == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(x_dev, 16) || !aligned(out_dev, 8)) return FP8_ERR_ALIGNMENT;
  return launch_encode_e2m1(x_dev, n, static_cast<uint8_t *>(out_dev), reinterpret_cast<cudaStream_t>(stream));
}

fp8_status_t fp8_debug_wait_probe(int *dev_status, uint64_t timeout_ns, fp8_stream_t stream) {
  if (dev_status == nullptr || timeout_ns == 0 || timeout_ns > 10000000000ull) return FP8_ERR_INVALID_ARG;
  if (!aligned(dev_status, 4)) return FP8_ERR_ALIGNMENT;
  return launch_wait_probe(dev_status, timeout_ns, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

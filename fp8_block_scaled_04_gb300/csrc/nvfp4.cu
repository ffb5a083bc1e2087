// nvfp4.cu -- NVFP4 quantizer and dequantizer ("Low precision: FP8, FP4, and
// microscaling": blocks of 16 elements, an E4M3 microscale per block and one
// fp32 scale per tensor that keeps the microscales inside E4M3's range).
//
// Element format: FP4 E2M1 (the OCP Microscaling element format the page
// cites): +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}, converted with
// cvt.rn.satfinite.e2m1x2.f32 (round to nearest even, saturating at +-6).
// Scale arithmetic (the page prints none; every step is one IEEE fp32
// operation rounded to nearest):
//   s_t = amax_tensor / (6 * 448)              (1 if that is 0 or not finite)
//   u   = (amax_block / 6) / s_t,  s_b = E4M3(u)   (stored as its E4M3 code)
//   S   = s_b * s_t,  S_inv = 1 / S            (0 if S is 0 or 1/S not finite)
//   q   = E2M1(x * S_inv)
// Packed codes: element 2i in the low nibble of byte i of the row.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"
#include "check.cuh"

namespace fp8bs {
namespace {

constexpr int kThreads = 256;

#ifndef NVF4_QUANT_BLOCKS_PER_LANE
#define NVF4_QUANT_BLOCKS_PER_LANE 4  // 16-element blocks one lane of the quantizer encodes per task (2: -7 %)
#endif

__device__ __forceinline__ float tensor_scale_of(float amax) {
  float s = __fdiv_rn(amax, 2688.0f);  // 6 * 448
  if (s == 0.0f || !isfinite(s)) s = 1.0f;
  return s;
}

// E4M3 code (round to nearest even, saturating) of a non-negative fp32.
__device__ __forceinline__ uint32_t e4m3_code(float u) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(u));
  return r & 0xffu;
}

// Exact value of an E4M3 code.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
}

// Eight fp32 values -> eight E2M1 codes in 32 bits (value i in nibble i).
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Value of the E2M1 code in the low 4 bits of c.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float mag = e == 0 ? 0.5f * static_cast<float>(m) : __int_as_float(static_cast<int>((e + 126u) << 23 | m << 22));
  return (c & 8u) ? -mag : mag;
}

__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t g, int64_t ng, bool tiled) {
  if (!tiled) return r * ng + g;
  const int64_t ncb = (ng + 3) / 4;
  return ((r / 128) * ncb + g / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (g % 4);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// Streaming 16-byte load that does not allocate in L1 (each byte is read once).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Per-tensor constants of the block-scale step. The block scale is
// u = fp32(fp32(amax_b / 6) / s_t), and only its E4M3 rounding is kept. The
// fast path forms u' = fp32(amax_b * c) with c = fp32(fp32(1/6) / s_t): each
// of the five roundings involved is within 2^-24 relative as long as every
// intermediate is an fp32 normal -- c (checked per tensor), amax_b / 6 (so
// amax_b >= 6 * 2^-126, checked per block: below it fp32(amax_b / 6) is
// subnormal and its rounding error is far larger) and u' (>= 2^-6) -- so
// |u' - u| is at most 5 units in the last place of u, and when the 20 fp32
// mantissa bits that E4M3 discards are at least 6 units away from the rounding
// midpoint (and u' is in E4M3's normal range below saturation) u and u' round
// to the same code. Other blocks (about 1 in 10^5 in the midpoint band, plus
// zero, tiny and non-finite ones) take the two IEEE divisions. s_inv of a code depends on
// the code alone, so a table of the 256 codes replaces the per-block
// reciprocal.
struct BlockScaleStep {
  float s_t, c;
  bool fast;
  const float *s_inv;  // [256], shared memory
};

__device__ __forceinline__ BlockScaleStep block_scale_step(float s_t, float *table) {
  static_assert(kThreads >= 256, "one table entry per thread");
  if (threadIdx.x < 256) {
    const float S = __fmul_rn(e4m3_value(threadIdx.x), s_t);
    float s_inv = __frcp_rn(S);
    if (S == 0.0f || !isfinite(s_inv)) s_inv = 0.0f;
    table[threadIdx.x] = s_inv;
  }
  __syncthreads();
  BlockScaleStep st;
  st.s_t = s_t;
  st.c = __fdiv_rn(__fdiv_rn(1.0f, 6.0f), s_t);
  st.fast = isfinite(st.c) && fabsf(st.c) >= 1.17549435e-38f;  // normal
  st.s_inv = table;
  return st;
}

// One 16-element block: its E4M3 scale code and the eight packed code bytes.
__device__ __forceinline__ void encode_block(const uint4 v0, const uint4 v1, const BlockScaleStep &bs, uint32_t &code,
                                             uint2 &packed) {
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = max(m, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
  const float amax_b = bf16_bits_to_f32(m);
  float u = __fmul_rn(amax_b, bs.c);
  const int d = static_cast<int>(__float_as_uint(u) & 0xfffffu) - 0x80000;
  if (!(bs.fast && amax_b >= 0x1.8p-124f && u >= 0.015625f && u <= 440.0f && (d >= 6 || d <= -6)))
    u = __fdiv_rn(__fdiv_rn(amax_b, 6.0f), bs.s_t);
  code = e4m3_code(u);
  const float s_inv = bs.s_inv[code];
  float lo[8], hi[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lo[2 * i] = __fmul_rn(bf16_bits_to_f32(w[i] & 0xffffu), s_inv);
    lo[2 * i + 1] = __fmul_rn(bf16_bits_to_f32(w[i] >> 16), s_inv);
    hi[2 * i] = __fmul_rn(bf16_bits_to_f32(w[4 + i] & 0xffffu), s_inv);
    hi[2 * i + 1] = __fmul_rn(bf16_bits_to_f32(w[4 + i] >> 16), s_inv);
  }
  packed = make_uint2(e2m1x8(lo), e2m1x8(hi));
}

// A warp covers 32 * NB consecutive blocks of a row per task: lane l takes
// blocks l, l + 32, ... (all 2 * NB of its 16-byte loads in flight before any
// arithmetic).
// amax_bits: the tensor's amax (fp32 bits) from the amax pass, or nullptr when
// static_ts gives the tensor scale.
template <int NB>
__global__ void __launch_bounds__(kThreads)
    nvfp4_quant_kernel(const uint16_t *__restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                       const uint32_t *__restrict__ amax_bits, const float *__restrict__ static_ts,
                       uint8_t *__restrict__ q, int64_t ldq, uint8_t *__restrict__ sf, bool tiled,
                       float *__restrict__ ts_out) {
  const float s_t = static_ts != nullptr ? *static_ts : tensor_scale_of(__uint_as_float(*amax_bits));
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts_out = s_t;
  __shared__ float s_inv_table[256];
  const BlockScaleStep bs = block_scale_step(s_t, s_inv_table);
  const int lane = threadIdx.x & 31;
  const int64_t ng = cols / 16;
  const int64_t chunks = (ng + 32 * NB - 1) / (32 * NB);
  const int64_t tasks = rows * chunks;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  for (int64_t t = warp0; t < tasks; t += nwarps) {
    const int64_t r = t / chunks;
    const int64_t gbase = (t - r * chunks) * (32 * NB) + lane;
    const uint16_t *row = x + r * ldx;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    uint4 v[NB][2];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int64_t g = gbase + 32 * j;
      v[j][0] = g < ng ? ld_stream16(row + g * 16) : zero;
      v[j][1] = g < ng ? ld_stream16(row + g * 16 + 8) : zero;
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int64_t g = gbase + 32 * j;
      uint32_t c;
      uint2 p;
      encode_block(v[j][0], v[j][1], bs, c, p);
      if (g < ng) {
        if (FP8BS_GUARD(r * ldq + g * 8, 8, (rows - 1) * ldq + cols / 2))
          *reinterpret_cast<uint2 *>(q + r * ldq + g * 8) = p;
        const int64_t so = sf_offset(r, g, ng, tiled);
        if (FP8BS_GUARD(so, 1, tiled ? ((rows + 127) / 128) * ((ng + 3) / 4) * 512 : rows * ng))
          sf[so] = static_cast<uint8_t>(c);
      }
    }
  }
}

// out = bf16(decode(q) * fp32(s_b * s_t)); one lane per 16-element block.
__global__ void __launch_bounds__(kThreads)
    nvfp4_dequant_kernel(const uint8_t *__restrict__ q, int64_t rows, int64_t cols, int64_t ldq,
                         const uint8_t *__restrict__ sf, bool tiled, const float *__restrict__ ts,
                         uint16_t *__restrict__ out, int64_t ldo) {
  const float s_t = *ts;
  const int64_t ng = cols / 16;
  const int64_t total = rows * ng;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t r = t / ng, g = t - r * ng;
    const float S = __fmul_rn(e4m3_value(sf[sf_offset(r, g, ng, tiled)]), s_t);
    const uint2 c = *reinterpret_cast<const uint2 *>(q + r * ldq + g * 8);
    const uint32_t cw[2] = {c.x, c.y};
    uint32_t o[8];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = __fmul_rn(e2m1_value(cw[h] >> (8 * i)), S);
        const float b = __fmul_rn(e2m1_value(cw[h] >> (8 * i + 4)), S);
        uint32_t p;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(p) : "f"(b), "f"(a));
        o[4 * h + i] = p;
      }
    if (FP8BS_GUARD(r * ldo + g * 16, 16, (rows - 1) * ldo + cols)) {
      uint4 *dst = reinterpret_cast<uint4 *>(out + r * ldo + g * 16);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

// out[i] = E2M1 code of x[i] (one code per byte), the quantizer's element step.
__global__ void __launch_bounds__(kThreads)
    e2m1_encode_kernel(const float *__restrict__ x, int64_t n8, uint8_t *__restrict__ out) {
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; t < n8;
       t += static_cast<int64_t>(gridDim.x) * kThreads) {
    const float4 a = reinterpret_cast<const float4 *>(x)[2 * t];
    const float4 b = reinterpret_cast<const float4 *>(x)[2 * t + 1];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const uint32_t c = e2m1x8(v);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo |= ((c >> (4 * i)) & 15u) << (8 * i);
      hi |= ((c >> (16 + 4 * i)) & 15u) << (8 * i);
    }
    if (FP8BS_GUARD(t, 1, n8)) reinterpret_cast<uint2 *>(out)[t] = make_uint2(lo, hi);
  }
}

int grid_for(int64_t work_items) {
  const int64_t per_cta = kThreads;
  int64_t g = (work_items + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

FP8BS_OOB_READER(oob_record_nvfp4)

fp8_status_t launch_quantize_nvfp4(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, bool tiled,
                                   const float *static_ts, uint8_t *q, int64_t ld_q, uint8_t *sf, float *ts_out,
                                   uint32_t *amax_ws, cudaStream_t stream) {
  constexpr int NB = NVF4_QUANT_BLOCKS_PER_LANE;
  const int64_t tasks = rows * ((cols / 16 + 32 * NB - 1) / (32 * NB));
  if (static_ts == nullptr) {
    if (cudaMemsetAsync(amax_ws, 0, sizeof(uint32_t), stream) != cudaSuccess) return FP8_ERR_CUDA;
    if (launch_amax(x, rows, cols, ld_x, amax_ws, stream) != FP8_OK) return FP8_ERR_CUDA;
  }
  nvfp4_quant_kernel<NB><<<grid_for(tasks * 32), kThreads, 0, stream>>>(
      x, rows, cols, ld_x, static_ts ? nullptr : amax_ws, static_ts, q, ld_q, sf, tiled, ts_out);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t launch_dequantize_nvfp4(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q, bool tiled,
                                     const uint8_t *sf, const float *ts, uint16_t *out, int64_t ld_out,
                                     cudaStream_t stream) {
  nvfp4_dequant_kernel<<<grid_for(rows * (cols / 16)), kThreads, 0, stream>>>(q, rows, cols, ld_q, sf, tiled, ts, out,
                                                                                 ld_out);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t launch_encode_e2m1(const float *x, int64_t n, uint8_t *out, cudaStream_t stream) {
  e2m1_encode_kernel<<<grid_for(n / 8), kThreads, 0, stream>>>(x, n / 8, out);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8bs

// fp8_math.cuh -- the element arithmetic of FP8 quantization shared by the
// quantize kernels and the GEMM epilogue that quantizes its own output:
// group amax on bf16 bit patterns, scale and reciprocal in IEEE fp32, the MX
// shared exponent, and the packed round-to-nearest-even saturating encode.
// Internal to libfp8bs.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8bs.h"
#include "ptx.cuh"

namespace fp8bs {

__device__ __forceinline__ float vmax_of(int fmt) { return fmt == FP8_E4M3 ? 448.0f : 57344.0f; }

// max |x| of eight bf16 (as the 15-bit magnitude pattern, which orders like the value)
__device__ __forceinline__ uint32_t absmax_bits8(uint4 v) {
  const uint32_t m = 0x7fff7fffu;
  uint32_t a = __vmaxu2(__vmaxu2(v.x & m, v.y & m), __vmaxu2(v.z & m, v.w & m));
  return max(a & 0xffffu, a >> 16);
}

__device__ __forceinline__ void bf16x8_to_f32(uint4 v, float (&f)[8]) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xffff0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xffff0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xffff0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xffff0000u);
}

__device__ __forceinline__ void scale_pair(float amax, float vmax, float &s, float &s_inv) {
  s = __fdiv_rn(amax, vmax);
  s_inv = __frcp_rn(s);
  if (s == 0.0f || !isfinite(s_inv)) s_inv = 0.0f;
}

// ceil(log2(fp32(amax / vmax))) from the bits, clamped to UE8M0's range.
__device__ __forceinline__ int mx_shared_exponent(float amax, float vmax) {
  const uint32_t u = __float_as_uint(__fdiv_rn(amax, vmax)) & 0x7fffffffu;
  if (u == 0) return -127;
  if (u >= 0x7f800000u) return 127;
  const uint32_t ex = u >> 23, fr = u & 0x7fffffu;
  int e;
  if (ex != 0)
    e = static_cast<int>(ex) - 127 + (fr != 0 ? 1 : 0);
  else
    e = (31 - __clz(fr)) - 149 + ((fr & (fr - 1u)) != 0 ? 1 : 0);
  return min(127, max(-127, e));
}

// 2^p exactly, p in [-127, 127]
__device__ __forceinline__ float exp2_exact(int p) {
  return p >= -126 ? __uint_as_float(static_cast<uint32_t>(p + 127) << 23) : __uint_as_float(0x00400000u);
}

template <int FMT>
__device__ __forceinline__ uint2 encode8(const float (&f)[8], float s_inv) {
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(f[i], s_inv);
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = FMT == FP8_E4M3 ? cvt_e4m3x2(y[2 * i], y[2 * i + 1]) : cvt_e5m2x2(y[2 * i], y[2 * i + 1]);
  return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}


}  // namespace fp8bs

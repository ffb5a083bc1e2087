// quantize.cu -- bf16 -> FP8 quantizers (per-tensor two-pass, per-token,
// 1x128 tile, 128x128 block, MX-32) and the FP8 -> bf16 dequantizer.
//
// Arithmetic follows "FP8 Mixed-Precision Serving in Production" (Quantization
// Granularity and Scaling Topologies: s = max|X_group| / V_max) and the
// qdq_e4m3 listing of "Low precision: FP8, FP4, and microscaling" (multiply
// by 1/s, cvt.rn.satfinite, exact decode through f16, one fp32 multiply by s):
//   s     = fp32_RN(amax / V_max)       (__fdiv_rn)
//   s_inv = fp32_RN(1 / s), 0 if s == 0 or 1/s is not finite
//   q     = RNE_satfinite(fp32_RN(x * s_inv))
// MX-32 (microscaling paragraph of the same page): e = ceil(log2(fp32_RN(amax
// / V_max))) clamped to [-127, 127], UE8M0 byte e + 127, q = RNE_satfinite(x * 2^-e).
//
// All kernels are bandwidth-bound streams: each warp reads whole 512-byte
// lines with 16-byte loads (4 independent loads in flight per lane), reduces
// the group amax with warp shuffles and writes the codes with 8-byte stores.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "fp8_math.cuh"
#include "ptx.cuh"
#include "check.cuh"

namespace fp8bs {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerLane = 4;                   // 16-byte vectors in flight per lane
constexpr int kSegVec = 32 * kVecPerLane;        // vectors a warp covers per task (1024 elements)
// the 1x128 quantizer keeps eight 16-byte loads in flight per lane (measured
// +3 % over four: it is latency-bound); the MX-32 quantizer keeps four (eight
// measured 3 % slower: with 8-element groups its per-group scales then need
// two rounds of pairs and a gather of every slot's maximum)
#ifndef FP8BS_TILE_VPL
#define FP8BS_TILE_VPL 8
#endif
constexpr int kTileVecPerLane = FP8BS_TILE_VPL;
#ifndef FP8BS_MX_VPL
#define FP8BS_MX_VPL 4
#endif
constexpr int kMxVecPerLane = FP8BS_MX_VPL;

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ int64_t mx_tiled_index(int64_t r, int64_t j, int64_t ngroups) {
  const int64_t col_blocks = (ngroups + 3) >> 2;
  return (((r >> 7) * col_blocks + (j >> 2)) << 9) + ((r & 31) << 4) + (((r & 127) >> 5) << 2) + (j & 3);
}
// The same byte in the staged-four-times layout (each 512-byte block stored
// four times in a row): its first copy; the others follow 512 bytes apart.
__device__ __forceinline__ int64_t mx_tiled_x4_index(int64_t r, int64_t j, int64_t ngroups) {
  const int64_t t = mx_tiled_index(r, j, ngroups);
  return ((t >> 9) << 11) + (t & 511);
}

// ------------------------------------------------------------ group kernels
// GROUP elements share a scale (128: 1x128 tile, 32: MX). A warp task is one
// row segment of 32 * VPL vectors (VPL slots of 32 lanes x 8 elements); groups
// never straddle rows or lanes. The per-group scale arithmetic (an IEEE
// division and reciprocal, or the MX exponent) is done once per group: lanes
// take one (slot, group) pair each, then hand the results back by shuffles.
// m[i] for a lane-dependent i, by selects (no local-memory array)
template <int N>
__device__ __forceinline__ uint32_t pick(const uint32_t (&m)[N], int i) {
  if constexpr (N == 4) {
    return i == 0 ? m[0] : (i == 1 ? m[1] : (i == 2 ? m[2] : m[3]));
  } else {
    uint32_t r = m[0];
#pragma unroll
    for (int k = 1; k < N; ++k) r = i == k ? m[k] : r;
    return r;
  }
}

// TILED (MX): 0 linear scales, 1 the tensor-core tiled layout, 4 that layout
// with each 512-byte block stored four times in a row
template <int FMT, int GROUP, bool MX, int TILED, int VPL = kVecPerLane>
__global__ void __launch_bounds__(kThreads) quant_group_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                               int64_t cols, int64_t ldx, uint8_t *__restrict__ q,
                                                               int64_t ldq, void *__restrict__ scales) {
  constexpr int TPG = GROUP / 8;            // lanes per group
  constexpr int GPS = 32 / TPG;             // groups per slot (2 for 1x128, 8 for MX)
  constexpr int PAIRS = VPL * GPS;           // (slot, group) pairs per task
  constexpr int ROUNDS = (PAIRS + 31) / 32;  // pairs per lane
  // one shuffle fetches a pair's amax when a lane of the pair's group has
  // the pair's slot index as its own (TPG a multiple of VPL); otherwise the
  // lane gathers every slot's maximum of the group and picks its slot
  constexpr bool DIRECT = TPG % VPL == 0;
  static_assert(ROUNDS <= 2 && (DIRECT || ROUNDS == 2 || PAIRS == 32), "pair layout");
  static_assert(VPL > 0 && (VPL & (VPL - 1)) == 0, "slots per lane: a power of two");
  grid_dependents_launch();  // a GEMM launched after this may set itself up meanwhile
  const int lane = threadIdx.x & 31;
  const int64_t vec_per_row = cols >> 3;
  const int64_t segs = (vec_per_row + (32 * VPL) - 1) / (32 * VPL);
  const int64_t tasks = rows * segs;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  const float vmax = vmax_of(FMT);
  for (int64_t t = warp0; t < tasks; t += nwarps) {
    const int64_t r = t / segs;
    const int64_t cv0 = (t - r * segs) * (32 * VPL);
    uint4 v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int64_t cv = cv0 + i * 32 + lane;
      v[i] = cv < vec_per_row ? ld_stream_v4(x + r * ldx + cv * 8) : make_uint4(0, 0, 0, 0);
    }
    uint32_t m[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      m[i] = absmax_bits8(v[i]);
#pragma unroll
      for (int o = TPG / 2; o > 0; o >>= 1) m[i] = max(m[i], __shfl_xor_sync(0xffffffffu, m[i], o));
    }
    // lane l computes the scales of pairs l + 32 k (slot = pair % VPL, group =
    // pair / VPL): every lane of a group holds that group's amax for every slot
    float my_inv[ROUNDS];
#pragma unroll
    for (int k = 0; k < ROUNDS; ++k) {
      const int pr = lane + 32 * k;
      const int p_slot = pr % VPL;
      const int p_grp = (pr / VPL) % GPS;
      uint32_t pm;
      if constexpr (DIRECT) {
        // lane p_grp * TPG + p_slot is in the group and offers slot p_slot's value
        pm = __shfl_sync(0xffffffffu, pick(m, p_slot), p_grp * TPG + p_slot);
      } else {
        pm = 0;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const uint32_t g = __shfl_sync(0xffffffffu, m[i], p_grp * TPG);
          pm = i == p_slot ? g : pm;
        }
      }
      const float amax = __uint_as_float(pm << 16);
      const int64_t pcv = cv0 + p_slot * 32 + p_grp * TPG;  // first vector of the pair's group
      if (MX) {
        const int e = mx_shared_exponent(amax, vmax);
        my_inv[k] = exp2_exact(-e);
        if (pr < PAIRS && pcv < vec_per_row) {
          const int64_t j = pcv / TPG;
          const int64_t ng = cols / 32;
          uint8_t *sf = static_cast<uint8_t *>(scales);
          if constexpr (TILED == 4) {
            const int64_t si = mx_tiled_x4_index(r, j, ng);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (FP8BS_GUARD(si + 512 * k, 1, ((rows + 127) / 128) * ((ng + 3) / 4) * 2048))
                sf[si + 512 * k] = static_cast<uint8_t>(e + 127);
          } else {
            const int64_t si = TILED ? mx_tiled_index(r, j, ng) : r * ng + j;
            if (FP8BS_GUARD(si, 1, TILED ? ((rows + 127) / 128) * ((ng + 3) / 4) * 512 : rows * ng))
              sf[si] = static_cast<uint8_t>(e + 127);
          }
        }
      } else {
        float s;
        scale_pair(amax, vmax, s, my_inv[k]);
        if (pr < PAIRS && pcv < vec_per_row && FP8BS_GUARD((pcv / TPG) * rows + r, 1, (cols / GROUP) * rows))
          static_cast<float *>(scales)[(pcv / TPG) * rows + r] = s;
      }
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      // pair (slot i, this lane's group) = group * VPL + i, computed in round
      // pair / 32 by lane pair % 32
      const int pr = (lane / TPG) * VPL + i;
      float s_inv = __shfl_sync(0xffffffffu, my_inv[0], pr % 32);
      if constexpr (ROUNDS > 1) {
        const float s1 = __shfl_sync(0xffffffffu, my_inv[ROUNDS - 1], pr % 32);
        s_inv = pr >= 32 ? s1 : s_inv;
      }
      const int64_t cv = cv0 + i * 32 + lane;
      if (cv >= vec_per_row) continue;
      float f[8];
      bf16x8_to_f32(v[i], f);
      if (FP8BS_GUARD(r * ldq + cv * 8, 8, (rows - 1) * ldq + cols))
        *reinterpret_cast<uint2 *>(q + r * ldq + cv * 8) = encode8<FMT>(f, s_inv);
    }
  }
}

// ------------------------------------------------------------ per-tensor
// Pass 1: grid-wide amax. Non-negative floats order like their bit patterns,
// so the reduction is an unsigned atomicMax on the fp32 bits.
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                        int64_t ldx, uint32_t *__restrict__ amax_bits) {
  const int lane = threadIdx.x & 31;
  const int64_t vec_per_row = cols >> 3;
  const int64_t segs = (vec_per_row + kSegVec - 1) / kSegVec;
  const int64_t tasks = rows * segs;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  uint32_t m = 0;
  for (int64_t t = warp0; t < tasks; t += nwarps) {
    const int64_t r = t / segs;
    const int64_t cv0 = (t - r * segs) * kSegVec;
    uint4 v[kVecPerLane];
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
      const int64_t cv = cv0 + i * 32 + lane;
      v[i] = cv < vec_per_row ? ld_stream_v4(x + r * ldx + cv * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) m = max(m, absmax_bits8(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[kThreads / 32];
  if (lane == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) b = max(b, red[w]);
    atomicMax(amax_bits, b << 16);
  }
}

// Pass 2: encode with one scale; the scale comes from the amax of pass 1 or
// from the caller (static scaling).
// record_amax (nullable): also reduce this tensor's amax into *record_amax
// (fp32 bits, atomicMax) -- the history update of delayed scaling.
template <int FMT>
__global__ void __launch_bounds__(kThreads) quant_tensor_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                                int64_t cols, int64_t ldx, uint8_t *__restrict__ q,
                                                                int64_t ldq, float *__restrict__ scale_out,
                                                                const uint32_t *__restrict__ amax_bits,
                                                                const float *__restrict__ static_scale,
                                                                uint32_t *__restrict__ record_amax = nullptr) {
  float s, s_inv;
  if (static_scale != nullptr) {
    s = *static_scale;
    s_inv = __frcp_rn(s);
    if (s == 0.0f || !isfinite(s_inv)) s_inv = 0.0f;
  } else {
    scale_pair(__uint_as_float(*amax_bits), vmax_of(FMT), s, s_inv);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && scale_out != nullptr) *scale_out = s;
  const int lane = threadIdx.x & 31;
  uint32_t rec = 0;
  const int64_t vec_per_row = cols >> 3;
  const int64_t segs = (vec_per_row + kSegVec - 1) / kSegVec;
  const int64_t tasks = rows * segs;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  for (int64_t tt = warp0; tt < tasks; tt += nwarps) {
    const int64_t t = tasks - 1 - tt;  // reverse of pass 1: its last rows are still in L2
    const int64_t r = t / segs;
    const int64_t cv0 = (t - r * segs) * kSegVec;
    uint4 v[kVecPerLane];
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
      const int64_t cv = cv0 + i * 32 + lane;
      v[i] = cv < vec_per_row ? ld_stream_v4(x + r * ldx + cv * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
      const int64_t cv = cv0 + i * 32 + lane;
      if (cv >= vec_per_row) continue;
      if (record_amax != nullptr) rec = max(rec, absmax_bits8(v[i]));
      float f[8];
      bf16x8_to_f32(v[i], f);
      if (FP8BS_GUARD(r * ldq + cv * 8, 8, (rows - 1) * ldq + cols))
        *reinterpret_cast<uint2 *>(q + r * ldq + cv * 8) = encode8<FMT>(f, s_inv);
    }
  }
  if (record_amax != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rec = max(rec, __shfl_xor_sync(0xffffffffu, rec, o));
    __shared__ uint32_t red[kThreads / 32];
    if (lane == 0) red[threadIdx.x >> 5] = rec;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t b = 0;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) b = max(b, red[w]);
      atomicMax(record_amax, b << 16);
    }
  }
}

// ------------------------------------------------------------ delayed scaling
// One CTA: s from the amax history (max over non-negative finite entries;
// a non-finite entry or an all-zero history gives s = 1), then the slot the
// current tensor's amax goes into is cleared for the encode kernel's atomicMax.
__global__ void __launch_bounds__(kThreads) delayed_scale_kernel(float *__restrict__ history, int hlen, int slot,
                                                                 int margin, int fmt, float *__restrict__ scale_out) {
  uint32_t best = 0;
  int bad = 0;
  for (int i = threadIdx.x; i < hlen; i += kThreads) {
    const uint32_t u = __float_as_uint(history[i]);
    if ((u & 0x7fffffffu) >= 0x7f800000u)
      bad = 1;
    else if ((u >> 31) == 0)
      best = max(best, u);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  }
  __shared__ uint32_t rb[kThreads / 32];
  __shared__ int rbad[kThreads / 32];
  if ((threadIdx.x & 31) == 0) {
    rb[threadIdx.x >> 5] = best;
    rbad[threadIdx.x >> 5] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    int any_bad = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      b = max(b, rb[w]);
      any_bad |= rbad[w];
    }
    float s = 1.0f;
    if (!any_bad && b != 0) {
      const float scaled = __fmul_rn(__uint_as_float(b), exp2_exact(margin));  // 2^m * max(H), one rounding
      s = __fdiv_rn(scaled, vmax_of(fmt));
    }
    *scale_out = s;
    if (FP8BS_GUARD(slot, 1, hlen)) history[slot] = 0.0f;
  }
}

// ------------------------------------------------------------ per-token
// One CTA per row; the row stays in registers between the amax reduction and
// the encode (U vectors per thread, rows up to 256 * U * 8 elements).
template <int FMT, int U>
__global__ void __launch_bounds__(kThreads) quant_token_kernel(const uint16_t *__restrict__ x, int64_t cols,
                                                               int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                                                               float *__restrict__ scales) {
  const int64_t r = blockIdx.x;
  const int64_t vec_per_row = cols >> 3;
  const uint16_t *xr = x + r * ldx;
  uint4 v[U];
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < U; ++i) {
    const int64_t cv = threadIdx.x + static_cast<int64_t>(i) * kThreads;
    v[i] = cv < vec_per_row ? ld_stream_v4(xr + cv * 8) : make_uint4(0, 0, 0, 0);
    m = max(m, absmax_bits8(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  uint32_t b = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) b = max(b, red[w]);
  float s, s_inv;
  scale_pair(__uint_as_float(b << 16), vmax_of(FMT), s, s_inv);
  if (threadIdx.x == 0 && FP8BS_GUARD(r, 1, gridDim.x)) scales[r] = s;
#pragma unroll
  for (int i = 0; i < U; ++i) {
    const int64_t cv = threadIdx.x + static_cast<int64_t>(i) * kThreads;
    if (cv < vec_per_row) {
      float f[8];
      bf16x8_to_f32(v[i], f);
      if (FP8BS_GUARD(r * ldq + cv * 8, 8, (static_cast<int64_t>(gridDim.x) - 1) * ldq + cols))
        *reinterpret_cast<uint2 *>(q + r * ldq + cv * 8) = encode8<FMT>(f, s_inv);
    }
  }
}

// Rows longer than the register-resident kernel handles: amax loop, then an
// encode loop that re-reads the row (mostly from L2).
template <int FMT>
__global__ void __launch_bounds__(kThreads) quant_token_long_kernel(const uint16_t *__restrict__ x, int64_t cols,
                                                                    int64_t ldx, uint8_t *__restrict__ q,
                                                                    int64_t ldq, float *__restrict__ scales) {
  const int64_t r = blockIdx.x;
  const int64_t vec_per_row = cols >> 3;
  const uint16_t *xr = x + r * ldx;
  uint32_t m = 0;
  for (int64_t cv = threadIdx.x; cv < vec_per_row; cv += kThreads) m = max(m, absmax_bits8(ld_stream_v4(xr + cv * 8)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  uint32_t b = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) b = max(b, red[w]);
  float s, s_inv;
  scale_pair(__uint_as_float(b << 16), vmax_of(FMT), s, s_inv);
  if (threadIdx.x == 0 && FP8BS_GUARD(r, 1, gridDim.x)) scales[r] = s;
  for (int64_t cv = threadIdx.x; cv < vec_per_row; cv += kThreads) {
    float f[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xr + cv * 8), f);
    if (FP8BS_GUARD(r * ldq + cv * 8, 8, (static_cast<int64_t>(gridDim.x) - 1) * ldq + cols))
      *reinterpret_cast<uint2 *>(q + r * ldq + cv * 8) = encode8<FMT>(f, s_inv);
  }
}

// ------------------------------------------------------------ 128x128 blocks
// One CTA per block: thread t holds column vector t%16 of rows t/16 + 16*i.
template <int FMT>
__global__ void __launch_bounds__(kThreads) quant_block_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                               int64_t cols, int64_t ldx, uint8_t *__restrict__ q,
                                                               int64_t ldq, float *__restrict__ scales) {
  const int64_t kb = blockIdx.x, rb = blockIdx.y;
  const int cvl = threadIdx.x & 15;
  const int r0 = threadIdx.x >> 4;
  uint4 v[8];
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = rb * 128 + r0 + 16 * i;
    v[i] = r < rows ? ld_stream_v4(x + r * ldx + kb * 128 + cvl * 8) : make_uint4(0, 0, 0, 0);
    m = max(m, absmax_bits8(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  uint32_t b = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) b = max(b, red[w]);
  float s, s_inv;
  scale_pair(__uint_as_float(b << 16), vmax_of(FMT), s, s_inv);
  if (threadIdx.x == 0 && FP8BS_GUARD(rb * (cols / 128) + kb, 1, ((rows + 127) / 128) * (cols / 128)))
    scales[rb * (cols / 128) + kb] = s;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = rb * 128 + r0 + 16 * i;
    if (r < rows) {
      float f[8];
      bf16x8_to_f32(v[i], f);
      if (FP8BS_GUARD(r * ldq + kb * 128 + cvl * 8, 8, (rows - 1) * ldq + cols))
        *reinterpret_cast<uint2 *>(q + r * ldq + kb * 128 + cvl * 8) = encode8<FMT>(f, s_inv);
    }
  }
}

// ------------------------------------------------------------ per-channel
// One scale per column (two passes, like per-tensor). A CTA owns a strip of at
// most 256 16-byte column vectors (2048 columns) and a chunk of rows. When the
// strip is narrower than 256 vectors the CTA's threads form several row slabs
// (slab = thread / strip width), so every thread loads: a thread keeps one
// vector (8 columns) and walks the rows r0 + slab, r0 + slab + slabs, ....
// Pass 1 keeps the column maxima in registers, combines the slabs in shared
// memory and issues one atomicMax per column per CTA. Pass 2 walks each
// thread's rows in reverse, so the rows pass 1 read last (still in L2) come first.

struct ChanGeom {
  int64_t strip_vec;  // vectors per strip (<= 256)
  int slabs;          // row slabs per CTA
};

// Strips of at most 256 vectors; a CTA of `threads` threads forms
// threads / strip_vec row slabs.
__host__ __device__ inline ChanGeom chan_geom(int64_t cols, int threads) {
  const int64_t vec = cols / 8;
  ChanGeom g;
  g.strip_vec = vec < kThreads ? vec : kThreads;
  g.slabs = static_cast<int>(threads / g.strip_vec);
  return g;
}

// The amax pass reads every byte from HBM and needs enough bytes in flight
// without the drain a register batch has at each step (issue eight loads,
// wait for all eight): each thread streams its rows through its own slots of a
// shared-memory ring with 16-byte cp.async copies, kChanStages groups of
// kChanStageRows rows in flight (192 KB per SM), and waits only for the oldest
// group (cp.async.wait_group, a hardware wait). A thread reads back only what
// it copied itself, so no barrier is needed inside the loop. One 1024-thread
// CTA per SM (one wave); the CTAs of a strip take interleaved blocks of
// `slabs` rows (CTA y: blocks y, y + gridDim.y, ...), so the whole grid sweeps
// the tensor front to back (6 x 2 and interleaving measured 3-4 % faster than
// 4 x 3 and contiguous chunks per CTA).
constexpr int kChanAmaxThreads = 1024;
constexpr int kChanStages = 6;
constexpr int kChanStageRows = 2;
constexpr int kChanAmaxSmem = kChanStages * kChanStageRows * kChanAmaxThreads * 16;

__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gsrc, bool pred) {
  // src-size 0 fills the 16 bytes with zeros and reads nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc),
               "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kChanAmaxThreads, 1) channel_amax_kernel(const uint16_t *__restrict__ x,
                                                                           int64_t rows, int64_t cols, int64_t ldx,
                                                                           uint32_t *__restrict__ col_amax) {
  extern __shared__ uint4 ring[];  // [stage][row][thread]
  const ChanGeom g = chan_geom(cols, kChanAmaxThreads);
  const int slab = static_cast<int>(threadIdx.x / g.strip_vec);
  const int64_t v = static_cast<int64_t>(blockIdx.x) * g.strip_vec + threadIdx.x % g.strip_vec;
  const bool active = slab < g.slabs && v < cols / 8;
  // this thread's rows first + stride * k, k = 0 .. n - 1
  const int64_t first = static_cast<int64_t>(blockIdx.y) * g.slabs + slab;
  const int64_t stride = static_cast<int64_t>(gridDim.y) * g.slabs;
  const int64_t n = active && first < rows ? (rows - 1 - first) / stride + 1 : 0;
  const uint16_t *px = x + first * ldx + v * 8;
  const int64_t step = stride * ldx;
  auto slot = [&](int st, int i) -> uint4 * {
    return ring + (st * kChanStageRows + i) * kChanAmaxThreads + threadIdx.x;
  };
  auto issue = [&](int64_t k0, int st) {
#pragma unroll
    for (int i = 0; i < kChanStageRows; ++i) {
      const int64_t k = k0 + i;
      cp_async_16(slot(st, i), k < n ? px + k * step : x, k < n);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int st = 0; st < kChanStages; ++st) issue(static_cast<int64_t>(st) * kChanStageRows, st);
  uint32_t m2[4] = {0u, 0u, 0u, 0u};  // packed 16-bit magnitude maxima of column pairs
  int st = 0;
  for (int64_t k0 = 0; k0 < n; k0 += kChanStageRows) {
    cp_async_wait<kChanStages - 1>();  // the oldest group (rows k0 ..) has landed
#pragma unroll
    for (int i = 0; i < kChanStageRows; ++i) {
      const uint4 vv = *slot(st, i);  // zero past the thread's rows
      m2[0] = __vmaxu2(m2[0], vv.x & 0x7fff7fffu);
      m2[1] = __vmaxu2(m2[1], vv.y & 0x7fff7fffu);
      m2[2] = __vmaxu2(m2[2], vv.z & 0x7fff7fffu);
      m2[3] = __vmaxu2(m2[3], vv.w & 0x7fff7fffu);
    }
    issue(k0 + static_cast<int64_t>(kChanStages) * kChanStageRows, st);  // refill the slots just read
    st = st + 1 == kChanStages ? 0 : st + 1;
  }
  cp_async_wait<0>();
  // combine the slabs in the (now idle) ring: slab 0 of each vector takes the
  // maximum over the others
  __syncthreads();
  uint4 *part = ring;
  part[threadIdx.x] = make_uint4(m2[0], m2[1], m2[2], m2[3]);
  __syncthreads();
  if (active && slab == 0) {
    for (int s = 1; s < g.slabs; ++s) {
      const uint4 o = part[threadIdx.x + s * g.strip_vec];
      m2[0] = __vmaxu2(m2[0], o.x);
      m2[1] = __vmaxu2(m2[1], o.y);
      m2[2] = __vmaxu2(m2[2], o.z);
      m2[3] = __vmaxu2(m2[3], o.w);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      atomicMax(col_amax + v * 8 + 2 * j, (m2[j] & 0xffffu) << 16);
      atomicMax(col_amax + v * 8 + 2 * j + 1, m2[j] & 0xffff0000u);
    }
  }
}

// The encode pass streams the same way (one 1024-thread CTA per SM and strip
// chunk, the same ring), walking each thread's rows from the last: those are
// the rows the amax pass read last, the ones most likely still in L2.
template <int FMT>
__global__ void __launch_bounds__(kChanAmaxThreads, 1) channel_quant_kernel(const uint16_t *__restrict__ x,
                                                                            int64_t rows, int64_t cols, int64_t ldx,
                                                                            const uint32_t *__restrict__ col_amax,
                                                                            uint8_t *__restrict__ q, int64_t ldq,
                                                                            float *__restrict__ scales) {
  extern __shared__ uint4 ring[];  // [stage][row][thread]
  const ChanGeom g = chan_geom(cols, kChanAmaxThreads);
  const int slab = static_cast<int>(threadIdx.x / g.strip_vec);
  const int64_t v = static_cast<int64_t>(blockIdx.x) * g.strip_vec + threadIdx.x % g.strip_vec;
  const bool active = slab < g.slabs && v < cols / 8;
  float s_inv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float s = 0.0f;
    s_inv[j] = 0.0f;
    if (active) {
      scale_pair(__uint_as_float(col_amax[v * 8 + j]), vmax_of(FMT), s, s_inv[j]);
      if (blockIdx.y == 0 && slab == 0 && FP8BS_GUARD(v * 8 + j, 1, cols)) scales[v * 8 + j] = s;
    }
  }
  // this thread's rows first + stride * k (the amax pass's), k = n - 1 down
  // to 0: the j-th row it visits is k = n - 1 - j
  const int64_t first = static_cast<int64_t>(blockIdx.y) * g.slabs + slab;
  const int64_t stride = static_cast<int64_t>(gridDim.y) * g.slabs;
  const int64_t n = active && first < rows ? (rows - 1 - first) / stride + 1 : 0;
  auto row_of = [&](int64_t j) -> int64_t { return first + (n - 1 - j) * stride; };
  auto slot = [&](int st, int i) -> uint4 * {
    return ring + (st * kChanStageRows + i) * kChanAmaxThreads + threadIdx.x;
  };
  auto issue = [&](int64_t j0, int st) {
#pragma unroll
    for (int i = 0; i < kChanStageRows; ++i) {
      const int64_t j = j0 + i;
      cp_async_16(slot(st, i), j < n ? x + row_of(j) * ldx + v * 8 : x, j < n);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int st = 0; st < kChanStages; ++st) issue(static_cast<int64_t>(st) * kChanStageRows, st);
  int st = 0;
  for (int64_t j0 = 0; j0 < n; j0 += kChanStageRows) {
    cp_async_wait<kChanStages - 1>();  // the oldest group (rows j0 ..) has landed
    uint4 vv[kChanStageRows];
#pragma unroll
    for (int i = 0; i < kChanStageRows; ++i) vv[i] = *slot(st, i);
    issue(j0 + static_cast<int64_t>(kChanStages) * kChanStageRows, st);  // refill the slots just read
    st = st + 1 == kChanStages ? 0 : st + 1;
#pragma unroll
    for (int i = 0; i < kChanStageRows; ++i) {
      const int64_t j = j0 + i;
      if (j >= n) break;
      float f[8];
      bf16x8_to_f32(vv[i], f);
#pragma unroll
      for (int c = 0; c < 8; ++c) f[c] = __fmul_rn(f[c], s_inv[c]);
      const int64_t off = row_of(j) * ldq + v * 8;
      if (FP8BS_GUARD(off, 8, (rows - 1) * ldq + cols)) *reinterpret_cast<uint2 *>(q + off) = encode8<FMT>(f, 1.0f);
    }
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------ dequantize
template <int FMT>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const uint8_t *__restrict__ q, int64_t rows, int64_t cols,
                                                           int64_t ldq, int gran, int sf_layout,
                                                           const void *__restrict__ scales,
                                                           uint16_t *__restrict__ out, int64_t ldo) {
  const int lane = threadIdx.x & 31;
  const int64_t vec_per_row = cols >> 4;  // 16 codes per vector
  const int64_t segs = (vec_per_row + kSegVec - 1) / kSegVec;
  const int64_t tasks = rows * segs;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  const float *sf = static_cast<const float *>(scales);
  const uint8_t *sb = static_cast<const uint8_t *>(scales);
  for (int64_t t = warp0; t < tasks; t += nwarps) {
    const int64_t r = t / segs;
    const int64_t cv0 = (t - r * segs) * kSegVec;
    uint4 v[kVecPerLane];
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
      const int64_t cv = cv0 + i * 32 + lane;
      v[i] = cv < vec_per_row ? ld_stream_v4(q + r * ldq + cv * 16) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
      const int64_t cv = cv0 + i * 32 + lane;
      if (cv >= vec_per_row) continue;
      const int64_t c = cv * 16;
      float s;
      switch (gran) {
        case FP8_GRAN_TENSOR: s = sf[0]; break;
        case FP8_GRAN_TOKEN: s = sf[r]; break;
        case FP8_GRAN_TILE_1x128: s = sf[(c >> 7) * rows + r]; break;
        case FP8_GRAN_BLOCK_128x128: s = sf[(r >> 7) * (cols >> 7) + (c >> 7)]; break;
        case FP8_GRAN_CHANNEL: s = 1.0f; break;
        default: {
          const int64_t ng = cols >> 5;
          const uint8_t e = sb[sf_layout == FP8_SF_TCGEN05      ? mx_tiled_index(r, c >> 5, ng)
                               : sf_layout == FP8_SF_TCGEN05_X4 ? mx_tiled_x4_index(r, c >> 5, ng)
                                                                : r * ng + (c >> 5)];
          s = e == 0xff ? __uint_as_float(0x7fc00000u) : exp2_exact(static_cast<int>(e) - 127);
        }
      }
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      float sc[16];  // per-element scales (differ only for per-channel scaling)
#pragma unroll
      for (int e = 0; e < 16; ++e) sc[e] = gran == FP8_GRAN_CHANNEL ? sf[c + e] : s;
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint16_t pair = static_cast<uint16_t>(w[j] >> (16 * h));
          const uint32_t hx2 = FMT == FP8_E4M3 ? cvt_e4m3x2_to_f16x2(pair) : cvt_e5m2x2_to_f16x2(pair);
          const __half2 hh = *reinterpret_cast<const __half2 *>(&hx2);
          const float lo = __fmul_rn(__low2float(hh), sc[4 * j + 2 * h]);
          const float hi = __fmul_rn(__high2float(hh), sc[4 * j + 2 * h + 1]);
          const uint32_t blo = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
          const uint32_t bhi = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
          o[2 * j + h] = blo | (bhi << 16);
        }
      }
      if (FP8BS_GUARD(r * ldo + c, 16, (rows - 1) * ldo + cols)) {
        uint4 *dst = reinterpret_cast<uint4 *>(out + r * ldo + c);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  }
}

// ------------------------------------------------------------ codec check
// Encodes fp32 inputs with the quantizers' element step (scale 1), so every
// fp32 bit pattern can be checked against the reference codec.
template <int FMT>
__global__ void __launch_bounds__(kThreads) encode_f32_kernel(const float *__restrict__ x, int64_t n8,
                                                              uint8_t *__restrict__ out) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const float4 a = reinterpret_cast<const float4 *>(x)[2 * i];
    const float4 b = reinterpret_cast<const float4 *>(x)[2 * i + 1];
    const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if (FP8BS_GUARD(i, 1, n8)) reinterpret_cast<uint2 *>(out)[i] = encode8<FMT>(f, 1.0f);
  }
}

// CTAs of `kernel` (256 threads, no dynamic shared memory) resident per SM,
// looked up once per kernel.
int resident_per_sm(const void *kernel) {
  struct Entry {
    std::atomic<const void *> fn{nullptr};
    std::atomic<int> occ{0};
  };
  static Entry table[48];
  for (Entry &e : table) {
    const void *f = e.fn.load(std::memory_order_acquire);
    if (f == kernel) {
      const int o = e.occ.load(std::memory_order_acquire);
      if (o > 0) return o;
      break;
    }
    if (f == nullptr) break;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0) != cudaSuccess || occ < 1) occ = 1;
  for (Entry &e : table) {
    const void *expected = nullptr;
    if (e.fn.compare_exchange_strong(expected, kernel) || expected == kernel) {
      e.occ.store(occ, std::memory_order_release);
      break;
    }
  }
  return occ;
}

// One wave of the CTAs that can be resident at once (the grid-stride loops
// assume every warp is running: a second, partial wave of CTAs only lengthens
// the tail); never more CTAs than warp tasks need.
template <typename KernelT>
int stream_grid(KernelT kernel, int64_t tasks) {
  const int64_t full =
      static_cast<int64_t>(device_sm_count()) * resident_per_sm(reinterpret_cast<const void *>(kernel));
  const int64_t need = (tasks + (kThreads / 32) - 1) / (kThreads / 32);
  return static_cast<int>(need < full ? (need > 0 ? need : 1) : full);
}

}  // namespace

FP8BS_OOB_READER(oob_record_quantize)

fp8_status_t launch_quantize(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt, int gran,
                             int sf_layout, const float *static_scale, uint8_t *q, int64_t ld_q, void *scales,
                             void *workspace, cudaStream_t stream) {
  const int64_t tasks = rows * ((cols / 8 + kSegVec - 1) / kSegVec);
  auto grid_of = [&](auto kernel) { return stream_grid(kernel, tasks); };
  const bool e4 = fmt == FP8_E4M3;
  int launches = 0;
  switch (gran) {
    case FP8_GRAN_TENSOR: {
      uint32_t *amax = static_cast<uint32_t *>(workspace);
      if (static_scale == nullptr) {
        if (cudaMemsetAsync(amax, 0, sizeof(uint32_t), stream) != cudaSuccess) return FP8_ERR_CUDA;
        amax_kernel<<<grid_of(amax_kernel), kThreads, 0, stream>>>(x, rows, cols, ld_x, amax);
        ++launches;
      }
      if (e4)
        quant_tensor_kernel<FP8_E4M3><<<grid_of(quant_tensor_kernel<FP8_E4M3>), kThreads, 0, stream>>>(
            x, rows, cols, ld_x, q, ld_q, static_cast<float *>(scales), amax, static_scale);
      else
        quant_tensor_kernel<FP8_E5M2><<<grid_of(quant_tensor_kernel<FP8_E5M2>), kThreads, 0, stream>>>(
            x, rows, cols, ld_x, q, ld_q, static_cast<float *>(scales), amax, static_scale);
      ++launches;
      break;
    }
    case FP8_GRAN_TOKEN: {
      const int64_t vec = cols / 8;
      float *s = static_cast<float *>(scales);
      const unsigned nb = static_cast<unsigned>(rows);
#define FP8BS_TOKEN(U)                                                                         \
  (e4 ? (quant_token_kernel<FP8_E4M3, U><<<nb, kThreads, 0, stream>>>(x, cols, ld_x, q, ld_q, s)) \
      : (quant_token_kernel<FP8_E5M2, U><<<nb, kThreads, 0, stream>>>(x, cols, ld_x, q, ld_q, s)))
      if (vec <= kThreads)
        FP8BS_TOKEN(1);
      else if (vec <= 2 * kThreads)
        FP8BS_TOKEN(2);
      else if (vec <= 4 * kThreads)
        FP8BS_TOKEN(4);
      else if (vec <= 8 * kThreads)
        FP8BS_TOKEN(8);
      else if (e4)
        quant_token_long_kernel<FP8_E4M3><<<nb, kThreads, 0, stream>>>(x, cols, ld_x, q, ld_q, s);
      else
        quant_token_long_kernel<FP8_E5M2><<<nb, kThreads, 0, stream>>>(x, cols, ld_x, q, ld_q, s);
#undef FP8BS_TOKEN
      ++launches;
      break;
    }
    case FP8_GRAN_TILE_1x128: {
      const int64_t tile_tasks = rows * ((cols / 8 + 32 * kTileVecPerLane - 1) / (32 * kTileVecPerLane));
#define FP8BS_TILE(F)                                                                                   \
  quant_group_kernel<F, 128, false, 0, kTileVecPerLane>                                                 \
      <<<stream_grid(quant_group_kernel<F, 128, false, 0, kTileVecPerLane>, tile_tasks), kThreads, 0, \
         stream>>>(x, rows, cols, ld_x, q, ld_q, scales)
      if (e4)
        FP8BS_TILE(FP8_E4M3);
      else
        FP8BS_TILE(FP8_E5M2);
#undef FP8BS_TILE
      ++launches;
      break;
    }
    case FP8_GRAN_BLOCK_128x128: {
      dim3 g(static_cast<unsigned>(cols / 128), static_cast<unsigned>((rows + 127) / 128));
      if (e4)
        quant_block_kernel<FP8_E4M3><<<g, kThreads, 0, stream>>>(x, rows, cols, ld_x, q, ld_q,
                                                                 static_cast<float *>(scales));
      else
        quant_block_kernel<FP8_E5M2><<<g, kThreads, 0, stream>>>(x, rows, cols, ld_x, q, ld_q,
                                                                 static_cast<float *>(scales));
      ++launches;
      break;
    }
    case FP8_GRAN_MX32: {
      // 0 linear, 1 tiled, 4 tiled and staged four times
      const int tiled = sf_layout == FP8_SF_TCGEN05 ? 1 : (sf_layout == FP8_SF_TCGEN05_X4 ? 4 : 0);
      const int64_t mx_tasks = rows * ((cols / 8 + 32 * kMxVecPerLane - 1) / (32 * kMxVecPerLane));
      if (tiled && (rows % 128 != 0 || cols % 128 != 0)) {
        const size_t bytes =
            static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((cols + 127) / 128) * 512 * tiled;
        if (cudaMemsetAsync(scales, 0, bytes, stream) != cudaSuccess) return FP8_ERR_CUDA;
      }
#define FP8BS_MX(F, T)                                                                              \
  quant_group_kernel<F, 32, true, T, kMxVecPerLane>                                                    \
      <<<stream_grid(quant_group_kernel<F, 32, true, T, kMxVecPerLane>, mx_tasks), kThreads, 0, stream>>>( \
          x, rows, cols, ld_x, q, ld_q, scales)
      if (e4 && tiled == 4)
        FP8BS_MX(FP8_E4M3, 4);
      else if (e4 && tiled)
        FP8BS_MX(FP8_E4M3, 1);
      else if (e4)
        FP8BS_MX(FP8_E4M3, 0);
      else if (tiled == 4)
        FP8BS_MX(FP8_E5M2, 4);
      else if (tiled)
        FP8BS_MX(FP8_E5M2, 1);
      else
        FP8BS_MX(FP8_E5M2, 0);
#undef FP8BS_MX
      ++launches;
      break;
    }
    case FP8_GRAN_CHANNEL: {
      uint32_t *col_amax = static_cast<uint32_t *>(workspace);
      if (cudaMemsetAsync(col_amax, 0, static_cast<size_t>(cols) * sizeof(uint32_t), stream) != cudaSuccess)
        return FP8_ERR_CUDA;
      // strips of <= 256 vectors x CTAs taking interleaved row blocks: one
      // wave of one CTA per SM (the ring takes most of shared memory), both
      // passes on the same grid
      const ChanGeom ag = chan_geom(cols, kChanAmaxThreads);
      const int64_t strips = (cols / 8 + ag.strip_vec - 1) / ag.strip_vec;
      int64_t ca = (static_cast<int64_t>(device_sm_count()) + strips - 1) / strips;
      const int64_t max_ca = (rows + ag.slabs - 1) / ag.slabs;
      if (ca > max_ca) ca = max_ca;
      if (ca < 1) ca = 1;
      const dim3 ga(static_cast<unsigned>(strips), static_cast<unsigned>(ca));
      if (cudaFuncSetAttribute(channel_amax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kChanAmaxSmem) !=
          cudaSuccess)
        return FP8_ERR_CUDA;
      channel_amax_kernel<<<ga, kChanAmaxThreads, kChanAmaxSmem, stream>>>(x, rows, cols, ld_x, col_amax);
      if (e4) {
        if (cudaFuncSetAttribute(channel_quant_kernel<FP8_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kChanAmaxSmem) != cudaSuccess)
          return FP8_ERR_CUDA;
        channel_quant_kernel<FP8_E4M3><<<ga, kChanAmaxThreads, kChanAmaxSmem, stream>>>(x, rows, cols, ld_x,
                                                                                       col_amax, q, ld_q,
                                                                                       static_cast<float *>(scales));
      } else {
        if (cudaFuncSetAttribute(channel_quant_kernel<FP8_E5M2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kChanAmaxSmem) != cudaSuccess)
          return FP8_ERR_CUDA;
        channel_quant_kernel<FP8_E5M2><<<ga, kChanAmaxThreads, kChanAmaxSmem, stream>>>(x, rows, cols, ld_x,
                                                                                       col_amax, q, ld_q,
                                                                                       static_cast<float *>(scales));
      }
      launches += 2;
      break;
    }
    default:
      return FP8_ERR_INVALID_ARG;
  }
  note_launches(launches);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t launch_quantize_delayed(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                                     float *history, int hlen, int slot, int margin, uint8_t *q, int64_t ld_q,
                                     float *scale_out, cudaStream_t stream) {
  delayed_scale_kernel<<<1, kThreads, 0, stream>>>(history, hlen, slot, margin, fmt, scale_out);
  const int64_t tasks = rows * ((cols / 8 + kSegVec - 1) / kSegVec);
  auto grid_of = [&](auto kernel) { return stream_grid(kernel, tasks); };
  uint32_t *rec = reinterpret_cast<uint32_t *>(history + slot);
  if (fmt == FP8_E4M3)
    quant_tensor_kernel<FP8_E4M3><<<grid_of(quant_tensor_kernel<FP8_E4M3>), kThreads, 0, stream>>>(
        x, rows, cols, ld_x, q, ld_q, nullptr, nullptr, scale_out, rec);
  else
    quant_tensor_kernel<FP8_E5M2><<<grid_of(quant_tensor_kernel<FP8_E5M2>), kThreads, 0, stream>>>(
        x, rows, cols, ld_x, q, ld_q, nullptr, nullptr, scale_out, rec);
  note_launches(2);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t launch_encode_f32(const float *x, int64_t n, int fmt, uint8_t *out, cudaStream_t stream) {
  const int64_t n8 = n / 8;
  auto grid_of = [&](auto kernel) { return stream_grid(kernel, (n8 + 31) / 32); };
  if (fmt == FP8_E4M3)
    encode_f32_kernel<FP8_E4M3><<<grid_of(encode_f32_kernel<FP8_E4M3>), kThreads, 0, stream>>>(x, n8, out);
  else
    encode_f32_kernel<FP8_E5M2><<<grid_of(encode_f32_kernel<FP8_E5M2>), kThreads, 0, stream>>>(x, n8, out);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t launch_dequantize(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q, int fmt, int gran,
                               int sf_layout, const void *scales, uint16_t *out, int64_t ld_out,
                               cudaStream_t stream) {
  const int64_t tasks = rows * ((cols / 16 + kSegVec - 1) / kSegVec);
  auto grid_of = [&](auto kernel) { return stream_grid(kernel, tasks); };
  if (fmt == FP8_E4M3)
    dequant_kernel<FP8_E4M3><<<grid_of(dequant_kernel<FP8_E4M3>), kThreads, 0, stream>>>(
        q, rows, cols, ld_q, gran, sf_layout, scales, out, ld_out);
  else
    dequant_kernel<FP8_E5M2><<<grid_of(dequant_kernel<FP8_E5M2>), kThreads, 0, stream>>>(
        q, rows, cols, ld_q, gran, sf_layout, scales, out, ld_out);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8bs

// ---------------------------------------------------------------------------
// Allocation-free per-tensor quantization.
//
// Some callers cannot call cudaMalloc: code running inside a host framework
// that owns every byte of device memory (a fixed arena handed to plugins with
// no allocator behind it), or a latency-critical path on which cudaMalloc's
// implicit device-wide synchronisation is not acceptable. For them the grid-wide
// amax of the two-pass per-tensor quantizer lives in this file-scope device
// array instead of a caller-provided workspace. Every GPU that loads the
// library holds these bytes until the process exits.
//
// In host code the name g_noalloc_scratch is only a host-side stand-in for the
// symbol, not a device address; the device address comes from
// cudaGetSymbolAddress, taken once per device (with that device current) on the
// first call made on that device. All calls share the array: each call clears
// the amax word before using it, and calls whose kernels overlap on the GPU
// (different streams, no ordering between them) race on it.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace fp8bs {
namespace {
constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxScratchDevices] = {};
}  // namespace

size_t noalloc_scratch_capacity() { return kNoAllocScratchBytes; }

// Device address of g_noalloc_scratch on the current device (set up once per device).
static fp8_status_t noalloc_scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return FP8_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return FP8_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FP8_OK;
}

// The amax pass alone (fp32 bits of max |x| reduced into *amax_bits, which the
// caller zeroes), for quantizers in other files.
fp8_status_t launch_amax(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, uint32_t *amax_bits,
                         cudaStream_t stream) {
  const int64_t tasks = rows * ((cols / 8 + kSegVec - 1) / kSegVec);
  amax_kernel<<<stream_grid(amax_kernel, tasks), kThreads, 0, stream>>>(x, rows, cols, ld_x, amax_bits);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t launch_quantize_tensor_noalloc(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                                            uint8_t *q, int64_t ld_q, float *scale_out, size_t scratch_needed,
                                            cudaStream_t stream) {
  if (scratch_needed > kNoAllocScratchBytes) return FP8_ERR_WORKSPACE;
  void *scratch = nullptr;
  const fp8_status_t st = noalloc_scratch_address(&scratch);
  if (st != FP8_OK) return st;
  uint32_t *amax = static_cast<uint32_t *>(scratch);
  if (cudaMemsetAsync(amax, 0, sizeof(uint32_t), stream) != cudaSuccess) return FP8_ERR_CUDA;
  const int64_t tasks = rows * ((cols / 8 + kSegVec - 1) / kSegVec);
  auto grid_of = [&](auto kernel) { return stream_grid(kernel, tasks); };
  amax_kernel<<<grid_of(amax_kernel), kThreads, 0, stream>>>(x, rows, cols, ld_x, amax);
  if (fmt == FP8_E4M3)
    quant_tensor_kernel<FP8_E4M3><<<grid_of(quant_tensor_kernel<FP8_E4M3>), kThreads, 0, stream>>>(
        x, rows, cols, ld_x, q, ld_q, scale_out, amax, nullptr);
  else
    quant_tensor_kernel<FP8_E5M2><<<grid_of(quant_tensor_kernel<FP8_E5M2>), kThreads, 0, stream>>>(
        x, rows, cols, ld_x, q, ld_q, scale_out, amax, nullptr);
  note_launches(2);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8bs

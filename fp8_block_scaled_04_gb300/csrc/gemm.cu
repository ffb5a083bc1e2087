// gemm.cu -- scaled FP8 GEMMs on the sm_103a tensor cores (tcgen05 + TMA).
//
// Out[M x N] (bf16) = X[M x K] W[N x K]^T with FP8 operands and fp32
// accumulation ("07 -- The FP8 Family", Scaling is what makes FP8 usable).
// The kernels share one warp-specialised, persistent structure:
//   warp 0      TMA producer: operand tiles (and scale-factor atoms) into a
//               ring of shared-memory stages;
//   warp 1      tensor-memory owner and MMA issuer (one elected thread; the
//               fold kernels add a second issuer in warp 2, alternate k-blocks);
//   other warps scale-factor copiers (block-scaled kinds) and consumers that
//               read tensor memory with tcgen05.ld.
//
// gemm_fold_kernel -- 1x128 activation tiles x 128x128 weight blocks (the
//   DeepSeek-V3 scheme of "07 -- The FP8 Family"; the promotion paragraph of
//   "Low precision: FP8, FP4, and microscaling"). Each 128-wide K chunk is one
//   MMA group into a fresh tensor-memory buffer; the consumer warps fold it
//   into fp32 registers as acc += (s_x[m,kb] * s_w[n/128,kb]) * partial. Two
//   tensor-memory buffers let the MMA of chunk kb+1 run while chunk kb folds.
//   gemm_fold_pair_kernel is the same on CTA pairs (cta_group::2); the
//   gemm_fold_swap kernels take few activation rows (decode), with W on the
//   MMA's 128-row side, optionally splitting K over a CTA cluster.
// gemm_tmem_kernel<KIND_EPI> -- per-tensor / per-token / per-channel scales:
//   the whole K sum stays in tensor memory and the scale product is applied
//   once in the epilogue.
// gemm_tmem_kernel<KIND_MX8> -- MXFP8: kind::mxf8f6f4.block_scale applies one
//   UE8M0 scale per 32 K-elements inside the tensor core ("Low precision",
//   microscaling); scale-factor atoms go smem -> tensor memory with tcgen05.cp.
//   KIND_MX8W is the same product on scales staged four times over, which
//   tensor memory takes in two wide copies per stage instead of three.
// gemm_tmem_kernel<KIND_NVF4> -- NVFP4: kind::mxf4nvf4.block_scale.scale_vec::4X
//   with E2M1 operands and one E4M3 scale per 16 K-elements; the two fp32
//   tensor scales multiply the accumulator in the epilogue.
//
// Every barrier wait is bounded (see mbar_wait): on expiry the CTA records
// FP8_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees tensor memory
// and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "internal.h"
#include "fp8_math.cuh"
#include "ptx.cuh"
#include "check.cuh"

namespace fp8bs {
namespace {

constexpr int BM = 128;  // tile rows (MMA M)
#ifndef MX_BN
#define MX_BN 256      // MXFP8 tile width
#define MX_STAGES 4
#define MX_NACC 1      // one accumulator: tensor memory also holds the scale factors
#endif
constexpr int BK = 128;  // K per stage (bytes of FP8)

struct SharedCtl {
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void flag_abort(SharedCtl *ctl, int *dev_status) {
  *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
  if (dev_status != nullptr) atomicExch(dev_status, static_cast<int>(FP8_ERR_TIMEOUT));
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Two fp32 -> bf16 round-to-nearest-even conversions in one instruction
// (cvt.rn.bf16x2.f32); lo lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Store 32 fp32 values (one row, 32 consecutive columns) as bf16 at element
// offset off of out (extent elements); n_left is the number of valid columns
// (multiple of 8).
__device__ __forceinline__ void store_row32(uint16_t *out, int64_t off, int64_t extent, const float (&v)[32],
                                            int n_left) {
  uint16_t *dst = out + off;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (8 * j < n_left && FP8BS_GUARD(off + 8 * j, 8, extent)) {
      uint4 w = make_uint4(pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                           pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
      *reinterpret_cast<uint4 *>(dst + 8 * j) = w;
    }
  }
}

#ifndef FOLD_PAIR_STAGES
#define FOLD_PAIR_STAGES 6  // 32 KB stages of the CTA-pair fold kernel
#endif
#ifndef FOLD_WIDE_STAGES
#define FOLD_WIDE_STAGES 4  // stages of the 128 x 256 fold kernel (3 leaves room for two epilogue slots per warp)
#endif
#ifndef NVF4_COPIERS
#define NVF4_COPIERS 2  // scale-copier warps of the NVFP4 GEMM (12 atom copies per k-block)
#endif
#ifndef SF_COPIER
#define SF_COPIER 1  // block-scaled GEMMs: separate warps may copy scale atoms to tensor memory
#endif
#ifndef MX8_COPIER
#define MX8_COPIER 0  // MXFP8: 0 = the MMA thread copies a stage's three atoms itself (+2.4 %), 1 = a copier warp
#endif
#ifndef FOLD_USE_PAIRS
#define FOLD_USE_PAIRS 0  // 1: block-scaled GEMMs with M > 128 run on CTA pairs (measured slower)
#endif

#ifndef FOLD_BF16_BN
#define FOLD_BF16_BN 256  // bf16-output fold GEMM: 256 (two partial buffers) or 128 (four)
#endif

#ifndef FOLD_MMA_ISSUERS
#define FOLD_MMA_ISSUERS 2  // threads (in warps 1..) issuing the fold kernels' MMAs, k-blocks dealt round robin
#endif

#ifndef SWAP_MMA_ISSUERS
#define SWAP_MMA_ISSUERS 2  // decode kernel: threads (in warps 1..) issuing its MMAs, k-blocks dealt round robin
#endif

#ifndef SWAP_FOLD_COLS
#define SWAP_FOLD_COLS 16  // decode kernel: activation rows per fold warp (16 or 32)
#endif

#ifndef FOLD_CHUNK
#define FOLD_CHUNK 64  // tensor-memory columns per fold load (16 or 32: pipelined; 64: one round trip per half)
#endif

// acc[base + i] += sc * (r[2i], r[2i+1]) for i < CH/2, as packed fp32x2 FMAs.
template <int CH, int NA>
__device__ __forceinline__ void fold_chunk(float2 (&acc)[NA], int base, float2 sc2, const uint32_t (&r)[CH]) {
#pragma unroll
  for (int i = 0; i < CH / 2; ++i)
    acc[base + i] = __ffma2_rn(sc2, make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), acc[base + i]);
}

// Producer drain after an abort: wait (bounded) for the copies of the last
// in-flight iterations so that no TMA write lands after the CTA exits.
template <int STAGES>
__device__ void drain_stages(uint64_t *full, int issued) {
  const int first = issued > STAGES ? issued - STAGES : 0;
  for (int j = first; j < issued; ++j) mbar_wait(&full[j % STAGES], (j / STAGES) & 1, kDrainTimeoutNs, nullptr);
}

// Tile order: consecutive CTAs walk down M inside one N band so that a band
// of W stays hot in L2 while X tiles are re-read.
// Tiles are taken in groups of `group_m` M-tiles: inside a group consecutive
// tiles walk down M, then move to the next N band; the next group starts after
// all N bands. A wave of CTAs therefore touches group_m X tiles (their rows stay
// in L2 across the whole group) and a few W bands; the host sizes group_m so the
// group's X rows take at most kRasterGroupBytes.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group_m, int &mt, int &nt) {
  const int per_group = group_m * num_n;
  const int g = tile / per_group;
  const int local = tile - g * per_group;
  const int first_m = g * group_m;
  const int gm = min(group_m, num_m - first_m);
  mt = first_m + local % gm;
  nt = local / gm;
}

// =====================================================================
// Fold kernel: 1x128 x 128x128 scales, per-chunk fp32 fold in registers
// =====================================================================
// Warp layout: warpgroup 0 = producer (warp 0), tensor-memory owner and MMA
// issuer (warp 1), second MMA issuer (warp 2), one idle warp; the other
// warpgroups are fold warps. One thread issuing every k-block's four MMAs,
// its commit and its two barrier waits needed ~800 cycles per k-block against
// 512 of tensor work; two issuers taking alternate k-blocks (each owning one
// partial buffer, so a buffer's MMAs stay in issue order) overlap that work. NBUF
// partial buffers of BN columns sit in tensor memory (NBUF x BN <= 512): with
// two, the fold of k-block kc gates the MMA of kc + 2; with four (128-wide
// tiles) the MMA may run four k-blocks ahead of the fold. Each fold thread
// owns WC columns of one row (128 with two buffers; 64 with four, so that
// eight warps share the tensor-memory reads of a 128-wide tile). The fold
// warps get most of the register file (setmaxnreg), the other warpgroup gives
// registers back.
template <int BN, int STAGES, int NBUF = 2>
struct FoldCfg {
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int WC = NBUF == 4 ? 64 : 128;        // columns per fold thread
  static constexpr int CONSUMER_WARPS = 4 * (BN / WC);  // 4 lane quarters x BN / WC column slabs
  static constexpr int FIRST_CONSUMER_WARP = 4;
  static constexpr int THREADS = 32 * (FIRST_CONSUMER_WARP + CONSUMER_WARPS);
  static_assert(NBUF * BN <= 512 && (NBUF == 2 || NBUF == 4), "partial buffers exceed tensor memory");
  // the fold warps wait on the stage barrier by parity: k-block kc + STAGES
  // cannot complete before they have released the buffer of kc + STAGES - NBUF
  static_assert(STAGES >= NBUF, "stage barrier parity needs STAGES >= NBUF");
  static constexpr uint32_t TMEM_COLS = NBUF * BN <= 256 ? 256 : 512;
  // output staging for the TMA-store epilogue: EPI_SLOTS 4 KB slots per fold
  // warp (two make the epilogue wait-free), as many as the shared memory left
  // by the stages holds
  static constexpr int SMEM_LIMIT = 232448 - 1024 - 512;  // opt-in maximum - alignment - static barriers
  static constexpr int EPI_SLOTS = (SMEM_LIMIT - STAGES * STAGE_BYTES) / (CONSUMER_WARPS * 4096) >= 2 ? 2 : 1;
  static constexpr int EPI_BYTES = EPI_SLOTS * CONSUMER_WARPS * 4096;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + 1024;
  static_assert(SMEM + 512 <= 232448, "shared memory budget");
  // setmaxnreg budgets. The increases are served from the registers the CTA
  // was launched with (registers per thread x THREADS), so the split must fit
  // in that pool or the increase never completes; launch_fold_tiles checks it
  // against the compiled register count before launching.
  static constexpr uint32_t REGS_CONTROL = 40;
  static constexpr uint32_t REGS_FOLD = CONSUMER_WARPS == 8 ? 224 : 240;
  static constexpr uint32_t REGS_NEEDED = REGS_CONTROL * 32 * FIRST_CONSUMER_WARP + REGS_FOLD * 32 * CONSUMER_WARPS;
};

// True when the kernel's launch register pool covers the setmaxnreg split.
template <typename KernelT>
bool reg_split_fits(KernelT kernel, int threads, uint32_t needed) {
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kernel) != cudaSuccess) return false;
  return static_cast<uint64_t>(attr.numRegs) * static_cast<uint64_t>(threads) >= needed;
}

// Epilogue through shared memory and TMA stores. The warp's 32 rows x 128
// columns leave as boxes 128 bytes wide and 32 rows high (bf16: two boxes of 64
// columns, the first at column n0 and the second at n1; fp8 codes: one box of
// 128 columns at n0), each written into one of the
// warp's NSLOTS 4 KB staging slots in the 128-byte swizzled layout of the
// output tensor map (16-byte chunk c of row r at chunk c ^ (r % 8)). Lane 0
// issues the stores and returns at once; a slot is rewritten only after the
// stores that read it have finished reading (bulk wait, read side). Rows past
// M and columns past N lie outside the tensor map and are not written.
// mid() runs once the first store is issued, while that store reads shared
// memory (the caller issues the next tile's first scale loads there, so their
// latency hides behind the rest of the epilogue).
template <int QFMT, int NSLOTS, int NA, typename Mid>
__device__ __forceinline__ void fold_epilogue_tma(float2 (&acc)[NA], int m, int row0, int n0, int n1, int M,
                                                  int N, const CUtensorMap *tmo, uint8_t *slots, float *q_scales,
                                                  int lane, Mid &&mid) {
  static_assert(NA == 32 || NA == 64, "32 or 64 column pairs per thread");
  static_assert(QFMT < 0 || NA == 64, "the quantized output needs a whole 1x128 group per thread");
  const bool rows_in = row0 < M;
  uint8_t *my_row = slots + lane * 128;
  const int swz = lane & 7;
  // the previous tile's stores from these slots have been read out
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  if constexpr (QFMT < 0) {
    uint32_t p[NA];
#pragma unroll
    for (int i = 0; i < NA; ++i) p[i] = pack_bf16x2(acc[i].x, acc[i].y);
#pragma unroll
    for (int bx = 0; bx < NA / 32; ++bx) {
      uint8_t *row = my_row + (bx % NSLOTS) * 4096;
      if (bx >= NSLOTS) {
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(row + ((c ^ swz) << 4)) =
            make_uint4(p[32 * bx + 4 * c], p[32 * bx + 4 * c + 1], p[32 * bx + 4 * c + 2], p[32 * bx + 4 * c + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      const int nb = bx == 0 ? n0 : n1;
      if (lane == 0 && rows_in && nb < N) {
        tma_store_2d(tmo, slots + (bx % NSLOTS) * 4096, nb, row0);
        bulk_commit_group();
      }
      if (bx == 0) mid();
    }
  } else {
    // this thread's 128 columns are exactly one 1x128 group of the output row:
    // round to bf16 (the unfused output), amax, scale, encode
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const uint32_t p = pack_bf16x2(acc[i].x, acc[i].y);
      acc[i] = make_float2(__uint_as_float(p << 16), __uint_as_float(p & 0xffff0000u));
      mx = max(mx, max(p & 0x7fffu, (p >> 16) & 0x7fffu));
    }
    float s, s_inv;
    scale_pair(__uint_as_float(mx << 16), vmax_of(QFMT), s, s_inv);
    if (m < M && n0 < N && FP8BS_GUARD(static_cast<int64_t>(n0 >> 7) * M + m, 1, static_cast<int64_t>(N / 128) * M))
      q_scales[static_cast<int64_t>(n0 >> 7) * M + m] = s;
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // 16 codes per chunk
      float f[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        f[2 * i] = acc[8 * j + i].x;
        f[2 * i + 1] = acc[8 * j + i].y;
      }
      const uint2 lo = encode8<QFMT>(reinterpret_cast<const float(&)[8]>(f[0]), s_inv);
      const uint2 hi = encode8<QFMT>(reinterpret_cast<const float(&)[8]>(f[8]), s_inv);
      *reinterpret_cast<uint4 *>(my_row + ((j ^ swz) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && rows_in && n0 < N) {
      tma_store_2d(tmo, slots, n0, row0);
      bulk_commit_group();
    }
    mid();
  }
}

// QFMT < 0: bf16 output. QFMT = FP8_E4M3 / FP8_E5M2: the epilogue quantizes
// its own bf16-rounded output with 1x128 scales (the next layer's activation
// format) and writes codes + scales instead of bf16.
template <int BN, int STAGES, int QFMT, int NBUF>
__global__ void __launch_bounds__(FoldCfg<BN, STAGES, NBUF>::THREADS, 1)
    gemm_fold_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO, const float *__restrict__ sa,
                     const float *__restrict__ sb, float *__restrict__ q_scales, int M, int N, int K, uint32_t idesc,
                     int *dev_status, int group_m, uint64_t wait_ns) {
  using C = FoldCfg<BN, STAGES, NBUF>;
  constexpr int ISSUERS = FOLD_MMA_ISSUERS;
  static_assert(ISSUERS >= 1 && ISSUERS <= 3 && NBUF % ISSUERS == 0, "each partial buffer needs one issuer");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  // One commit per k-block: empty[s] completes when the MMAs of the k-block in
  // stage s are done, which frees the stage for the producer and tells the fold
  // warps that the partial of that k-block is in tensor memory. The fold warps
  // can wait on it by parity because the stage's next k-block (kc + STAGES)
  // cannot complete before they release the buffer of k-block kc + STAGES - NBUF.
  __shared__ uint64_t full[STAGES], empty[STAGES], tempty[NBUF], drain;
  __shared__ SharedCtl ctl;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = K / BK;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int ntiles = num_m * num_n;
  const int nblk128 = (N + 127) / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) mbar_init(&tempty[b], C::CONSUMER_WARPS);
    mbar_init(&drain, ISSUERS);
    ctl.abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // setup above overlaps the previous kernel (dependent launch); its outputs
  // (the operands and scales) are read only after this
  grid_dependency_wait();
  const uint32_t tmem = ctl.tmem_base;

  if (warp < C::FIRST_CONSUMER_WARP) {
    regs_dealloc<C::REGS_CONTROL>();
    if (warp == 0 && lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        int mt, nt;
        tile_coords(tile, num_m, num_n, group_m, mt, nt);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          uint8_t *a_s = smem + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          tma_load_2d(a_s, &tmA, kb * BK, mt * BM, &full[s]);
          tma_load_2d(a_s + C::A_BYTES, &tmB, kb * BK, nt * BN, &full[s]);
        }
      }
      if (!ok) {
        flag_abort(&ctl, dev_status);
        drain_stages<STAGES>(full, it);
      }
    } else if (warp >= 1 && warp <= ISSUERS && lane == 0) {
      // MMA issuers: issuer j takes the k-blocks with kc % ISSUERS == j, so each
      // partial buffer is written by one thread only (its MMAs stay in order)
      // while the issue work of consecutive k-blocks overlaps
      const int me = warp - 1;
      int it = 0, kc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++it, ++kc) {
          if (ISSUERS > 1 && kc % ISSUERS != me) continue;
          const int b = kc % NBUF;
          const int s = it % STAGES;
          const uint32_t a0 = smem_u32(smem + s * C::STAGE_BYTES);
          const uint64_t adesc = sdesc_k_sw128(a0), bdesc = sdesc_k_sw128(a0 + C::A_BYTES);
          const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
          // the stage's operands first (they usually landed long before), then
          // the partial buffer: the fold's release is the critical path, and a
          // wait on an already completed barrier still costs ~100 cycles
          if (!mbar_wait(&full[s], (it / STAGES) & 1, wait_ns, &ctl.abort) ||
              !mbar_wait(&tempty[b], ((kc / NBUF) & 1) ^ 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // K step k: both descriptors advance 32 bytes (2 units of 16 bytes)
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
          tc_commit(&empty[s]);
        }
      }
      if (!ok) flag_abort(&ctl, dev_status);
      tc_commit(&drain);
      mbar_wait(&drain, 0, kDrainTimeoutNs, nullptr);
    }
  } else {
    regs_alloc<C::REGS_FOLD>();
    // ------------------------------------------------ fold consumers
    const int cw = warp - C::FIRST_CONSUMER_WARP;
    constexpr int WC = C::WC;
    const int quarter = warp & 3;  // tensor-memory lanes this warp may access
    const int half = cw >> 2;      // which WC-column slab of the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int kc = 0;
    bool ok = true;
    float2 acc[WC / 2];
    // Scales: each k-block's pair (s_x of this thread's row, s_w of its slab's
    // weight block) is loaded two k-blocks before its fold into one of two
    // register slots, and the slot is reloaded right after it is read. The
    // k-block loop runs in pairs so that each slot is a fixed register: no
    // register copy ever waits on a load in flight (a shifted ring of loaded
    // values stalls every k-block for a whole global-load latency). Indices are
    // clamped instead of predicated, so no select consumes a load either: a
    // clamped load only feeds rows or k-blocks that are never stored.
    // The first two pairs of a tile are loaded during the previous tile's
    // epilogue (see fold_epilogue_tma), else at the top of the tile.
    auto first_scales = [&](int t, float &a0, float &b0, float &a1, float &b1) {
      int tm, tn;
      tile_coords(t, num_m, num_n, group_m, tm, tn);
      const int tr = min(tm * BM + quarter * 32 + lane, M - 1);
      const int tb = min((tn * BN + half * WC) / 128, nblk128 - 1);
      const float *pa = sa + tr;
      const float *pb = sb + static_cast<int64_t>(tb) * KB;
      const int k1 = KB > 1 ? 1 : 0;
      a0 = __ldg(pa);
      b0 = __ldg(pb);
      a1 = __ldg(pa + static_cast<int64_t>(k1) * M);
      b1 = __ldg(pb + k1);
    };
    float nsa0 = 0.0f, nsb0 = 0.0f, nsa1 = 0.0f, nsb1 = 0.0f;
    bool have_next = false;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      int mt, nt;
      tile_coords(tile, num_m, num_n, group_m, mt, nt);
      const int m = mt * BM + quarter * 32 + lane;
      const int nb = (nt * BN + half * WC) / 128;  // weight block of this slab
      const float *sa_row = sa + min(m, M - 1);
      const float *sb_blk = sb + static_cast<int64_t>(min(nb, nblk128 - 1)) * KB;
#pragma unroll
      for (int i = 0; i < WC / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);
      float sa0, sb0, sa1, sb1;  // slot 0: even k-blocks, slot 1: odd k-blocks
      if (have_next) {
        sa0 = nsa0;
        sb0 = nsb0;
        sa1 = nsa1;
        sb1 = nsb1;
      } else {
        first_scales(tile, sa0, sb0, sa1, sb1);
      }
      // fold k-block kb with the scales in (sa_s, sb_s), then reload that slot for kb + 2
      auto fold_one = [&](int kb, float &sa_s, float &sb_s) -> bool {
        const int b = kc % NBUF;
        const float sc = sa_s * sb_s;
        const float2 sc2 = make_float2(sc, sc);
        const int kn = min(kb + 2, KB - 1);
        sa_s = __ldg(sa_row + static_cast<int64_t>(kn) * M);
        sb_s = __ldg(sb_blk + kn);
        const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(b * BN + half * WC);
        // every lane polls (one polling lane and a broadcast measured 7 % slower)
        const bool got = mbar_wait(&empty[kc % STAGES], (kc / STAGES) & 1, wait_ns, &ctl.abort);
        if (!__all_sync(0xffffffffu, got)) return false;
        tc_fence_after();
        constexpr int CH = FOLD_CHUNK < WC ? FOLD_CHUNK : WC, NCH = WC / CH;
        if constexpr (CH >= 64) {
          // few large loads, one round trip each: load, wait, fold
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            uint32_t rb[CH];
            tmem_ld_chunk<CH>(taddr + CH * c, rb);
            tmem_wait_ld_regs(rb);
            if (c + 1 == NCH) {
              // every load of this buffer has landed: hand it back to its MMA issuer
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty[b]);
            }
            fold_chunk<CH>(acc, c * (CH / 2), sc2, rb);
          }
        } else {
          // two chunk buffers: the load of chunk c+1 is in flight while chunk c
          // folds; the fold is packed fp32x2 FMA (two IEEE fmas per instruction)
          uint32_t rbuf[2][CH];
          tmem_ld_chunk<CH>(taddr, rbuf[0]);
          tmem_wait_ld_regs(rbuf[0]);
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            if (c + 1 < NCH) tmem_ld_chunk_keep<CH>(taddr + CH * (c + 1), rbuf[(c + 1) & 1], rbuf[c & 1]);
            fold_chunk<CH>(acc, c * (CH / 2), sc2, rbuf[c & 1]);
            if (c + 1 < NCH) {
              tmem_wait_ld_regs(rbuf[(c + 1) & 1]);
              if (c + 2 == NCH) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[b]);
              }
            }
          }
        }
        ++kc;
        return true;
      };
      for (int kb = 0; kb < KB && ok; kb += 2) {
        ok = fold_one(kb, sa0, sb0);
        if (ok && kb + 1 < KB) ok = fold_one(kb + 1, sa1, sb1);
      }
      if (!ok) break;
      const int next = tile + static_cast<int>(gridDim.x);
      fold_epilogue_tma<QFMT, C::EPI_SLOTS>(acc, m, mt * BM + quarter * 32, nt * BN + half * WC,
                                            nt * BN + half * WC + 64, M, N, &tmO,
                                            smem + STAGES * C::STAGE_BYTES + cw * C::EPI_SLOTS * 4096, q_scales,
                                            lane, [&]() {
                                              have_next = next < ntiles;
                                              if (have_next) first_scales(next, nsa0, nsb0, nsa1, nsb1);
                                            });
    }
    if (!ok && lane == 0) flag_abort(&ctl, dev_status);
    if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// =====================================================================
// Fold kernel on CTA pairs (cta_group::2): 256 x 256 output tiles
// =====================================================================
// A cluster of two CTAs computes one 256 x 256 tile. Each CTA loads its own
// 128 rows of X and its 128 rows of W (the pair MMA takes A rows and B columns
// half from each CTA's shared memory, at the same offsets) and holds its 128
// output rows x 256 columns in its own tensor memory. The even CTA issues the
// pair MMAs; both CTAs' copies complete on its stage barriers, its commits
// arrive on both CTAs' barriers, and both CTAs' fold warps hand partial
// buffers back to it. A stage is 32 KB per CTA instead of 48 KB (6 stages fit,
// more copies in flight) and each W tile is fetched once per pair.
template <int STAGES>
struct FoldPairCfg {
  static constexpr int A_BYTES = BM * BK;   // this CTA's 128 rows of X
  static constexpr int B_BYTES = 128 * BK;  // this CTA's 128 rows of W
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TM = 256, TN = 256;  // pair tile
  static constexpr int CONSUMER_WARPS = 8;  // per CTA: 4 lane quarters x 2 column halves
  static constexpr int FIRST_CONSUMER_WARP = 4;
  static constexpr int THREADS = 32 * (FIRST_CONSUMER_WARP + CONSUMER_WARPS);
  static constexpr uint32_t TMEM_COLS = 512;  // two partial buffers of 256 columns
  // output staging of the TMA-store epilogue (one 4 KB slot per fold warp); it
  // follows the last stage, so even a read of all 256 W rows from one CTA's
  // last stage would stay inside the allocation
  static constexpr int SMEM_LIMIT = 232448 - 1024 - 512;
  static constexpr int EPI_SLOTS = (SMEM_LIMIT - STAGES * STAGE_BYTES) / (CONSUMER_WARPS * 4096) >= 2 ? 2 : 1;
  static constexpr int EPI_BYTES = EPI_SLOTS * CONSUMER_WARPS * 4096;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + 1024;
  static_assert(SMEM + 512 <= 232448, "shared memory budget");
  static constexpr uint32_t REGS_CONTROL = 40;
  static constexpr uint32_t REGS_FOLD = 224;
  static constexpr uint32_t REGS_NEEDED = REGS_CONTROL * 32 * FIRST_CONSUMER_WARP + REGS_FOLD * 32 * CONSUMER_WARPS;
};

template <int STAGES, int QFMT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FoldPairCfg<STAGES>::THREADS, 1)
    gemm_fold_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmO, const float *__restrict__ sa,
                          const float *__restrict__ sb, float *__restrict__ q_scales, int M, int N, int K,
                          uint32_t idesc, int *dev_status, int group_m) {
  using C = FoldPairCfg<STAGES>;
  constexpr int ISSUERS = FOLD_MMA_ISSUERS;
  static_assert(ISSUERS == 1 || ISSUERS == 2, "each partial buffer needs one issuer");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  // one commit per k-block (multicast to both CTAs' empty[s]), as in the
  // single-CTA kernel: the fold warps wait on the stage barrier
  __shared__ uint64_t full[STAGES], empty[STAGES], tempty[2], drain;
  __shared__ SharedCtl ctl;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int KB = K / BK;
  const int num_m = (M + C::TM - 1) / C::TM;
  const int num_n = (N + C::TN - 1) / C::TN;
  const int ntiles = num_m * num_n;
  const int nblk128 = (N + 127) / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&tempty[b], 2 * C::CONSUMER_WARPS);  // both CTAs' fold warps release to the even CTA
    mbar_init(&drain, ISSUERS);
    ctl.abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctl.tmem_base, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t full_lead = cluster_addr(&full[0], 0);      // stage s at + 8 s
  const uint32_t tempty_lead = cluster_addr(&tempty[0], 0);  // buffer b at + 8 b

  if (warp < C::FIRST_CONSUMER_WARP) {
    regs_dealloc<C::REGS_CONTROL>();
    if (warp == 0 && lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = pair; tile < ntiles && ok; tile += npairs) {
        int mt, nt;
        tile_coords(tile, num_m, num_n, group_m, mt, nt);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, kWaitTimeoutNs, &ctl.abort)) {
            ok = false;
            break;
          }
          uint8_t *a_s = smem + s * C::STAGE_BYTES;
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
          const uint32_t bar = full_lead + 8u * static_cast<uint32_t>(s);
          tma_load_2d_pair(a_s, &tmA, kb * BK, mt * C::TM + static_cast<int>(rank) * 128, bar);
          tma_load_2d_pair(a_s + C::A_BYTES, &tmB, kb * BK, nt * C::TN + static_cast<int>(rank) * 128, bar);
        }
      }
      if (!ok) {
        flag_abort(&ctl, dev_status);
        if (leader) {
          drain_stages<STAGES>(full, it);
        } else {
          // this CTA's copies complete on the even CTA's barriers; give them time to land
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) {
          }
        }
      }
    } else if (warp >= 1 && warp <= ISSUERS && lane == 0 && leader) {
      // pair MMA issuers, k-blocks dealt round robin as in the single-CTA kernel
      const int me = warp - 1;
      int it = 0, kc = 0;
      bool ok = true;
      for (int tile = pair; tile < ntiles && ok; tile += npairs) {
        for (int kb = 0; kb < KB; ++kb, ++it, ++kc) {
          if (ISSUERS > 1 && kc % ISSUERS != me) continue;
          const int b = kc & 1;
          const int s = it % STAGES;
          if (!mbar_wait(&tempty[b], ((kc >> 1) & 1) ^ 1, kWaitTimeoutNs, &ctl.abort) ||
              !mbar_wait(&full[s], (it / STAGES) & 1, kWaitTimeoutNs, &ctl.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t b0 = a0 + C::A_BYTES;
          const uint32_t d = tmem + static_cast<uint32_t>(b * C::TN);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_f8f6f4_pair(d, sdesc_k_sw128(a0 + 32 * k), sdesc_k_sw128(b0 + 32 * k), idesc, k > 0 ? 1u : 0u);
          tc_commit_pair_mc(&empty[s], 0x3);
        }
      }
      if (!ok) flag_abort(&ctl, dev_status);
      tc_commit_pair(&drain);
      mbar_wait(&drain, 0, kDrainTimeoutNs, nullptr);
    }
  } else {
    regs_alloc<C::REGS_FOLD>();
    const int cw = warp - C::FIRST_CONSUMER_WARP;
    const int quarter = warp & 3;
    const int half = cw >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int kc = 0;
    bool ok = true;
    float2 acc[64];
    // first two scale pairs of a tile, in two fixed register slots reloaded in
    // place with clamped indices, as in the single-CTA kernel
    auto first_scales = [&](int t, float &a0, float &b0, float &a1, float &b1) {
      int tm, tn;
      tile_coords(t, num_m, num_n, group_m, tm, tn);
      const int tr = min(tm * C::TM + static_cast<int>(rank) * 128 + quarter * 32 + lane, M - 1);
      const int tb = min(tn * 2 + half, nblk128 - 1);
      const float *pa = sa + tr;
      const float *pb = sb + static_cast<int64_t>(tb) * KB;
      const int k1 = KB > 1 ? 1 : 0;
      a0 = __ldg(pa);
      b0 = __ldg(pb);
      a1 = __ldg(pa + static_cast<int64_t>(k1) * M);
      b1 = __ldg(pb + k1);
    };
    float nsa0 = 0.0f, nsb0 = 0.0f, nsa1 = 0.0f, nsb1 = 0.0f;
    bool have_next = false;
    for (int tile = pair; tile < ntiles && ok; tile += npairs) {
      int mt, nt;
      tile_coords(tile, num_m, num_n, group_m, mt, nt);
      const int m = mt * C::TM + static_cast<int>(rank) * 128 + quarter * 32 + lane;
      const int nb = nt * 2 + half;
      const float *sa_row = sa + min(m, M - 1);
      const float *sb_blk = sb + static_cast<int64_t>(min(nb, nblk128 - 1)) * KB;
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);
      float sa0, sb0, sa1, sb1;
      if (have_next) {
        sa0 = nsa0;
        sb0 = nsb0;
        sa1 = nsa1;
        sb1 = nsb1;
      } else {
        first_scales(tile, sa0, sb0, sa1, sb1);
      }
      auto fold_one = [&](int kb, float &sa_s, float &sb_s) -> bool {
        const int b = kc & 1;
        const float sc = sa_s * sb_s;
        const float2 sc2 = make_float2(sc, sc);
        const int kn = min(kb + 2, KB - 1);
        sa_s = __ldg(sa_row + static_cast<int64_t>(kn) * M);
        sb_s = __ldg(sb_blk + kn);
        const bool got = mbar_wait(&empty[kc % STAGES], (kc / STAGES) & 1, kWaitTimeoutNs, &ctl.abort);
        if (!__all_sync(0xffffffffu, got)) return false;
        tc_fence_after();
        const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(b * C::TN + half * 128);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t rb[64];
          tmem_ld_32x32b_x64(taddr + 64 * c, rb);
          tmem_wait_ld_regs(rb);
          if (c == 1) {
            // both loads of this buffer have landed: release it to the even CTA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_lead + 8u * static_cast<uint32_t>(b));
          }
          fold_chunk<64>(acc, c * 32, sc2, rb);
        }
        ++kc;
        return true;
      };
      for (int kb = 0; kb < KB && ok; kb += 2) {
        ok = fold_one(kb, sa0, sb0);
        if (ok && kb + 1 < KB) ok = fold_one(kb + 1, sa1, sb1);
      }
      if (!ok) break;
      const int next = tile + npairs;
      fold_epilogue_tma<QFMT, C::EPI_SLOTS>(acc, m, mt * C::TM + static_cast<int>(rank) * 128 + quarter * 32,
                                            nb * 128, nb * 128 + 64, M, N, &tmO,
                                            smem + STAGES * C::STAGE_BYTES + cw * C::EPI_SLOTS * 4096, q_scales,
                                            lane, [&]() {
                                              have_next = next < ntiles;
                                              if (have_next) first_scales(next, nsa0, nsb0, nsa1, nsb1);
                                            });
    }
    if (!ok && lane == 0) flag_abort(&ctl, dev_status);
    if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the even CTA's MMAs and both CTAs' tensor-memory reads are done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

// =====================================================================
// Fold kernel, operands swapped for few activation rows (decode shapes)
// =====================================================================
// D[n, m] = sum_k W[n, k] X[m, k]: the MMA's M side is 128 rows of W (one
// 128x128 weight block per K chunk, so one weight scale per chunk), its N side
// is BX rows of X. Each fold thread owns one W row and BXW = BX / G of the BX
// activation rows (G groups of four fold warps, BXW = SWAP_FOLD_COLS: with
// all 64 rows per warp the fold warps, not HBM, set the k-block rate); the
// activation scales s_x[kb, m] vary along its row and reach every lane as
// shared-memory broadcasts. Two threads issue the MMAs, alternate k-blocks;
// a warp of its own copies the scale chunks, so that the W stream never waits
// for a chunk slot.
template <int BX, int STAGES>
struct SwapCfg {
  static constexpr int W_BYTES = BM * BK;
  static constexpr int X_BYTES = BX * BK;
  static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
  static constexpr int NBUF = 4;                       // tensor-memory partial buffers
  static constexpr int G = BX > SWAP_FOLD_COLS ? BX / SWAP_FOLD_COLS : 1;  // fold warp groups
  static constexpr int BXW = BX / G;                   // activation rows per fold warp
  static constexpr int FOLD_WARPS = 4 * G;
  static constexpr int ISSUERS = SWAP_MMA_ISSUERS;      // MMA-issuing warps 1 .. ISSUERS
  static constexpr int SCALE_WARP = 1 + ISSUERS;       // copies the scale chunks (tensor-copy path)
  static constexpr int FIRST_FOLD_WARP = 2 + ISSUERS;
  static constexpr int THREADS = 32 * (FIRST_FOLD_WARP + FOLD_WARPS);
  static_assert(ISSUERS >= 1 && ISSUERS <= 2 && NBUF % ISSUERS == 0, "each partial buffer needs one issuer");
  static constexpr uint32_t TMEM_COLS = NBUF * BX <= 32 ? 32 : (NBUF * BX <= 64 ? 64 : (NBUF * BX <= 128 ? 128 : 256));
  static constexpr int CBUF_BYTES = FOLD_WARPS * 2 * BXW * 4;   // per fold warp: two slots of BXW fp32 products
  static constexpr int OTILE_BYTES = FOLD_WARPS * BXW * 32 * 2;  // per fold warp: 32 columns x BXW rows, bf16
  // scale chunks (when the scales' layout allows tensor copies): two slots,
  // each KBC k-blocks of s_x[kb, tile's BX rows] followed by s_w[tile, kb]
  static constexpr int KBC = BX >= 64 ? 28 : 64;
  static constexpr int SC_HEAD = 4;  // k-blocks of a chunk whose products come first
  static constexpr int SC_X_BYTES = KBC * BX * 4;
  static constexpr int SC_W_OFF = SC_X_BYTES / 4;                  // in floats
  static constexpr int SC_SLOT_BYTES = SC_X_BYTES + ((KBC * 4 + 127) / 128) * 128;
  static constexpr int SC_TX_BYTES = SC_X_BYTES + KBC * 4;          // the two boxes' bytes
  static constexpr int SC_OFFSET = STAGES * STAGE_BYTES + CBUF_BYTES + OTILE_BYTES;
  static constexpr int SMEM = SC_OFFSET + 2 * SC_SLOT_BYTES + 1024;
  static_assert(KBC % 4 == 0 && KBC <= 256 && SC_X_BYTES % 128 == 0 && SC_OFFSET % 128 == 0, "scale chunk layout");
  static_assert(SC_HEAD > 0 && SC_HEAD < KBC && (SC_HEAD * BX) % 32 == 0, "head of a chunk");
  static_assert(BX % 16 == 0 && BX <= 64, "MMA N side");
  static_assert(SMEM + 256 <= 232448, "shared memory budget");
};

template <int BX, int STAGES>
__global__ void __launch_bounds__(SwapCfg<BX, STAGES>::THREADS, 1)
    gemm_fold_swap_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                          const __grid_constant__ CUtensorMap tmSX, const __grid_constant__ CUtensorMap tmSW,
                          int sc_tma, const float *__restrict__ sa, const float *__restrict__ sb,
                          uint16_t *__restrict__ out, int M, int N, int K, uint32_t idesc, int *dev_status,
                          uint64_t wait_ns) {
  using C = SwapCfg<BX, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  // one commit per k-block; the fold warps wait on the stage barrier (the
  // stage's next k-block needs the release of k-block kc + NBUF first, and
  // STAGES > NBUF)
  static_assert(STAGES > C::NBUF, "stage barrier parity");
  // sfull / phead / pready / sempty: the two scale-chunk slots (landed /
  // products of the first SC_HEAD k-blocks formed by the scale warp / all its
  // products formed / read by every fold warp)
  __shared__ uint64_t full[STAGES], empty[STAGES], tempty[C::NBUF], drain, sfull[2], phead[2], pready[2], sempty[2];
  __shared__ SharedCtl ctl;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = K / BK;
  const int num_x = (M + BX - 1) / BX;
  const int num_w = (N + BM - 1) / BM;
  const int ntiles = num_x * num_w;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::NBUF; ++b) mbar_init(&tempty[b], C::FOLD_WARPS);
    mbar_init(&drain, C::ISSUERS);
    for (int j = 0; j < 2; ++j) {
      mbar_init(&sfull[j], 1);
      mbar_init(&phead[j], 1);
      mbar_init(&pready[j], 1);
      mbar_init(&sempty[j], C::FOLD_WARPS);
    }
    ctl.abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
    if (sc_tma) {
      tma_prefetch_desc(&tmSX);
      tma_prefetch_desc(&tmSW);
    }
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  // the first stages' W boxes of this CTA's first tile go to L2 while the
  // previous kernel finishes (a prefetch reads nothing into this kernel)
  if (warp == 0 && lane == 0 && static_cast<int>(blockIdx.x) < ntiles) {
    const int wt = static_cast<int>(blockIdx.x) / num_x;
    for (int kb = 0; kb < STAGES && kb < KB; ++kb) tma_prefetch_l2_2d(&tmW, kb * BK, wt * BM);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // dependent launch: the setup above overlaps the previous kernel's tail;
  // nothing it writes (X, the scales, Out) is read into this kernel before this wait
  grid_dependents_launch();
  grid_dependency_wait();
  const uint32_t tmem = ctl.tmem_base;
  float *scbuf = reinterpret_cast<float *>(smem + C::SC_OFFSET);

  if (warp == C::SCALE_WARP) {
    // scale chunks (tensor-copy path): KBC k-blocks of s_x[kb, tile rows] and
    // s_w[tile, kb] per chunk into the next of two slots, each as soon as the
    // fold warps have read the chunk that held the slot (boxes past K or M read
    // as zeros); once a chunk has landed the warp turns each s_x in place into
    // the product s_w[kb] * s_x[kb, m] the fold applies (formed once here
    // instead of in every fold warp of the four lane quarters). A warp of its
    // own, so that the weight stream never waits behind these copies.
    if (sc_tma) {
      int chunk = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const int wt = tile / num_x, xt = tile - wt * num_x;
        for (int kb0 = 0; kb0 < KB; kb0 += C::KBC) {
          const int slot = chunk & 1;
          const bool free_slot = mbar_wait(&sempty[slot], ((chunk >> 1) & 1) ^ 1, wait_ns, &ctl.abort);
          if (!__all_sync(0xffffffffu, free_slot)) {
            ok = false;
            break;
          }
          float *dst = scbuf + slot * (C::SC_SLOT_BYTES / 4);
          if (lane == 0) {
            mbar_arrive_expect_tx(&sfull[slot], C::SC_TX_BYTES);
            tma_load_2d(dst, &tmSX, xt * BX, kb0, &sfull[slot]);
            tma_load_2d(dst + C::SC_W_OFF, &tmSW, kb0, wt, &sfull[slot]);
          }
          ++chunk;
          const bool landed = mbar_wait(&sfull[slot], ((chunk - 1) >> 1) & 1, wait_ns, &ctl.abort);
          if (!__all_sync(0xffffffffu, landed)) {
            ok = false;
            break;
          }
          // the first SC_HEAD k-blocks first, so that the fold warps can start
          // the chunk while the rest are formed
#pragma unroll
          for (int i = lane; i < C::SC_HEAD * BX; i += 32) dst[i] = dst[C::SC_W_OFF + i / BX] * dst[i];
          __syncwarp();
          if (lane == 0) mbar_arrive(&phead[slot]);
#pragma unroll 4
          for (int i = C::SC_HEAD * BX + lane; i < C::KBC * BX; i += 32) dst[i] = dst[C::SC_W_OFF + i / BX] * dst[i];
          __syncwarp();
          if (lane == 0) mbar_arrive(&pready[slot]);
        }
      }
      if (!ok && lane == 0) {
        flag_abort(&ctl, dev_status);
        // the last two chunks' copies may still be in flight (an earlier one
        // has been waited for before its slot was reused)
        for (int c = chunk > 2 ? chunk - 2 : 0; c < chunk; ++c)
          mbar_wait(&sfull[c & 1], (c >> 1) & 1, kDrainTimeoutNs, nullptr);
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const int wt = tile / num_x, xt = tile - wt * num_x;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          uint8_t *w_s = smem + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          tma_load_2d(w_s, &tmW, kb * BK, wt * BM, &full[s]);
          tma_load_2d(w_s + C::W_BYTES, &tmX, kb * BK, xt * BX, &full[s]);
        }
      }
      if (!ok) {
        flag_abort(&ctl, dev_status);
        drain_stages<STAGES>(full, it);
      }
    }
  } else if (warp <= C::ISSUERS) {
    // MMA issuers: issuer j takes the k-blocks with kc % ISSUERS == j (so each
    // partial buffer is written by one thread and its MMAs stay in order);
    // one thread's waits, MMAs and commit take about a k-block's worth of HBM
    // time, so consecutive k-blocks' issue work overlaps
    if (lane == 0) {
      const int me = warp - 1;
      int it = 0, kc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++it, ++kc) {
          if (C::ISSUERS > 1 && kc % C::ISSUERS != me) continue;
          const int b = kc % C::NBUF;
          const int s = it % STAGES;
          const uint32_t w0 = smem_u32(smem + s * C::STAGE_BYTES);
          const uint64_t wdesc = sdesc_k_sw128(w0), xdesc = sdesc_k_sw128(w0 + C::W_BYTES);
          const uint32_t d = tmem + static_cast<uint32_t>(b * BX);
          // the partial buffer (usually free) before the stage (the copy in
          // flight from HBM is the critical wait); descriptors formed first
          if (!mbar_wait(&tempty[b], ((kc / C::NBUF) & 1) ^ 1, wait_ns, &ctl.abort) ||
              !mbar_wait(&full[s], (it / STAGES) & 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) mma_f8f6f4(d, wdesc + 2 * k, xdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
          tc_commit(&empty[s]);
        }
      }
      if (!ok) flag_abort(&ctl, dev_status);
      tc_commit(&drain);
      mbar_wait(&drain, 0, kDrainTimeoutNs, nullptr);
    }
  } else {
    constexpr int BXW = C::BXW;
    const int fw = warp - C::FIRST_FOLD_WARP;  // fold warp 0 .. FOLD_WARPS - 1
    const int quarter = warp & 3;           // the tensor-memory lanes (W rows) this warp may read
    const int col0 = (fw / 4) * BXW;        // its activation rows within the tile: col0 .. col0 + BXW - 1
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr int XR = (BXW + 31) / 32;  // activation-scale registers per lane
    // this warp's shared memory: two slots (even / odd k-blocks) of BXW scale
    // products, and its 32 output columns x BXW rows of bf16 for the epilogue
    float *cbuf = reinterpret_cast<float *>(smem + STAGES * C::STAGE_BYTES) + fw * 2 * BXW;
    uint16_t *otile =
        reinterpret_cast<uint16_t *>(smem + STAGES * C::STAGE_BYTES + C::CBUF_BYTES) + fw * BXW * 32;
    int kc = 0, chunk = 0;
    bool ok = true;
    float2 acc[BXW / 2];  // acc[i] = activation rows col0 + 2i, + 1 of this thread's output column
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const int wt = tile / num_x, xt = tile - wt * num_x;
      const int m0 = xt * BX + col0;
      const float *sb_blk = sb + static_cast<int64_t>(wt) * KB;  // one 128-row weight block per tile
#pragma unroll
      for (int j = 0; j < BXW / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
      // Scales, tensor-copy path (sc_tma): the scale warp brings s_x and s_w
      // of KBC k-blocks at a time into a chunk slot and forms the products
      // s_w * s_x there; every lane reads them back as shared-memory
      // broadcasts.
      // Register path (a layout the tensor copies cannot describe): lane l
      // holds s_x[kb, m0 + 32 r + l] and s_w[kb] in one of two fixed register
      // slots (even / odd k-blocks), loaded two k-blocks ahead and reloaded in
      // place (indices clamped, not predicated, so that no copy or select waits
      // on a load in flight; values of rows past M are never stored), forms
      // the products for its rows and leaves them in the warp's slot for this
      // k-block's parity. Either way each product is the same fp32 multiply.
      auto load_sx = [&](int kbq, float (&dst)[XR]) {
        const int kq = min(kbq, KB - 1);
#pragma unroll
        for (int r = 0; r < XR; ++r) dst[r] = __ldg(sa + static_cast<int64_t>(kq) * M + min(m0 + 32 * r + lane, M - 1));
      };
      float xs0[XR], xs1[XR], ws0 = 0.0f, ws1 = 0.0f;
      if (!sc_tma) {
        load_sx(0, xs0);
        load_sx(1, xs1);
        ws0 = __ldg(sb_blk);
        ws1 = __ldg(sb_blk + (KB > 1 ? 1 : 0));
      }
      auto fold_one = [&](int kb, float (&xs)[XR], float &ws) -> bool {
        const int b = kc % C::NBUF;
        const int kl = kb % C::KBC;
        const float *sxc = scbuf + (chunk & 1) * (C::SC_SLOT_BYTES / 4);
        if (sc_tma) {
          if (kl == 0 || kl == C::SC_HEAD) {
            const bool ready =
                mbar_wait(kl == 0 ? &phead[chunk & 1] : &pready[chunk & 1], (chunk >> 1) & 1, wait_ns, &ctl.abort);
            if (!__all_sync(0xffffffffu, ready)) return false;
          }
        } else {
          // the slot is rewritten two k-blocks later, after the __syncwarp
          // that follows this k-block's reads in every lane
          float *cs = cbuf + (kc & 1) * BXW;
#pragma unroll
          for (int q = 0; q < XR; ++q)
            if (32 * q + lane < BXW) cs[32 * q + lane] = ws * xs[q];
          load_sx(kb + 2, xs);
          ws = __ldg(sb_blk + min(kb + 2, KB - 1));
          __syncwarp();
        }
        const bool got = mbar_wait(&empty[kc % STAGES], (kc / STAGES) & 1, wait_ns, &ctl.abort);
        if (!__all_sync(0xffffffffu, got)) return false;
        tc_fence_after();
        const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(b * BX + col0);
        // the warp's BXW columns of the partial in one load and one wait
        uint32_t r[BXW];
        tmem_ld_chunk<BXW>(taddr, r);
        tmem_wait_ld_regs(r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[b]);
        if (sc_tma) {
          // the products s_w * s_x of this k-block's rows col0 .. col0 + BXW - 1
          const float4 *c4 = reinterpret_cast<const float4 *>(sxc + kl * BX + col0);
#pragma unroll
          for (int i = 0; i < BXW / 4; ++i) {
            const float4 c = c4[i];
            acc[2 * i] = __ffma2_rn(make_float2(c.x, c.y),
                                    make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])), acc[2 * i]);
            acc[2 * i + 1] = __ffma2_rn(make_float2(c.z, c.w),
                                        make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])),
                                        acc[2 * i + 1]);
          }
          if (kl == C::KBC - 1 || kb == KB - 1) {
            // this chunk's scales are read (the products above consumed them)
            __syncwarp();
            if (lane == 0) mbar_arrive(&sempty[chunk & 1]);
            ++chunk;
          }
        } else {
          const float4 *c4 = reinterpret_cast<const float4 *>(cbuf + (kc & 1) * BXW);
#pragma unroll
          for (int i = 0; i < BXW / 4; ++i) {
            const float4 c = c4[i];
            acc[2 * i] = __ffma2_rn(make_float2(c.x, c.y),
                                    make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])), acc[2 * i]);
            acc[2 * i + 1] = __ffma2_rn(make_float2(c.z, c.w),
                                        make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])),
                                        acc[2 * i + 1]);
          }
        }
        ++kc;
        return true;
      };
      for (int kb = 0; kb < KB && ok; kb += 2) {
        ok = fold_one(kb, xs0, ws0);
        if (ok && kb + 1 < KB) ok = fold_one(kb + 1, xs1, ws1);
      }
      if (!ok) break;
      // the warp's 32 columns x BXW rows go through shared memory so that each
      // output row's 64 bytes leave in four 16-byte stores (eight rows per
      // warp-wide store) instead of 32 two-byte ones
#pragma unroll
      for (int j = 0; j < BXW / 2; ++j) {
        otile[(2 * j) * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j].x));
        otile[(2 * j + 1) * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j].y));
      }
      __syncwarp();
      const int ncol = wt * BM + quarter * 32 + (lane & 3) * 8;  // N % 16 == 0: a chunk is all in or all out
#pragma unroll
      for (int i = 0; i < BXW / 8; ++i) {
        const int j = 8 * i + (lane >> 2);
        const int m = m0 + j;
        if (m < M && ncol < N && FP8BS_GUARD(static_cast<int64_t>(m) * N + ncol, 8, static_cast<int64_t>(M) * N))
          *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(m) * N + ncol) =
              *reinterpret_cast<const uint4 *>(otile + j * 32 + (lane & 3) * 8);
      }
      __syncwarp();  // the next tile rewrites the slot
    }
    if (!ok && lane == 0) flag_abort(&ctl, dev_status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}


// Split-K variant of the decode kernel, for too few 128-row W blocks to occupy
// the GPU: each tile's K range is split over the S CTAs of a cluster (launch
// attribute). Every CTA folds its share of the k-blocks; the non-leading CTAs
// leave their fp32 partials in their own shared memory and signal the leader
// (rank 0), which adds them in rank order (a fixed order: the result does not
// depend on timing) through distributed shared memory, writes the output and
// lets them go. A separate kernel: folding the split into the unsplit kernel
// made its launches ~2 us slower (measured).
template <int BX, int STAGES>
struct SwapSplitCfg {
  static constexpr int W_BYTES = BM * BK;
  static constexpr int X_BYTES = BX * BK;
  static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
  static constexpr int NBUF = 4;                       // tensor-memory partial buffers
  // fold warps, MMA issuers and the per-warp shared memory as in SwapCfg
  static constexpr int G = BX > SWAP_FOLD_COLS ? BX / SWAP_FOLD_COLS : 1;
  static constexpr int BXW = BX / G;
  static constexpr int FOLD_WARPS = 4 * G;
  static constexpr int ISSUERS = SWAP_MMA_ISSUERS;
  static constexpr int FIRST_FOLD_WARP = 1 + ISSUERS;
  static constexpr int THREADS = 32 * (FIRST_FOLD_WARP + FOLD_WARPS);
  static_assert(ISSUERS >= 1 && ISSUERS <= 2 && NBUF % ISSUERS == 0, "each partial buffer needs one issuer");
  static constexpr uint32_t TMEM_COLS = NBUF * BX <= 32 ? 32 : (NBUF * BX <= 64 ? 64 : (NBUF * BX <= 128 ? 128 : 256));
  static constexpr int RED_BYTES = BM * BX * 4;  // this CTA's partial, [BX][128] fp32
  static constexpr int CBUF_BYTES = FOLD_WARPS * 2 * BXW * 4;
  static constexpr int OTILE_BYTES = FOLD_WARPS * BXW * 32 * 2;
  static constexpr int SMEM = STAGES * STAGE_BYTES + RED_BYTES + CBUF_BYTES + OTILE_BYTES + 1024;
  static_assert(BX % 16 == 0 && BX <= 64, "MMA N side");
  static_assert(SMEM + 256 <= 232448, "shared memory budget");
};

template <int BX, int STAGES>
__global__ void __launch_bounds__(SwapSplitCfg<BX, STAGES>::THREADS, 1)
    gemm_fold_swap_split_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                          const float *__restrict__ sa, const float *__restrict__ sb, uint16_t *__restrict__ out,
                          int M, int N, int K, uint32_t idesc, int *dev_status) {
  using C = SwapSplitCfg<BX, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  // one commit per k-block; the fold warps wait on the stage barrier (the
  // stage's next k-block needs the release of k-block kc + NBUF first, and
  // STAGES > NBUF)
  static_assert(STAGES > C::NBUF, "stage barrier parity");
  __shared__ uint64_t full[STAGES], empty[STAGES], tempty[C::NBUF], drain, red_full, red_done;
  __shared__ SharedCtl ctl;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = K / BK;
  const int num_x = (M + BX - 1) / BX;
  const int num_w = (N + BM - 1) / BM;
  const int ntiles = num_x * num_w;
  // cluster geometry and this CTA's k-blocks
  const int S = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int first_tile = static_cast<int>(blockIdx.x) / S;
  const int tile_step = static_cast<int>(gridDim.x) / S;
  const int kb_lo = rank * KB / S;
  const int kb_hi = (rank + 1) * KB / S;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::NBUF; ++b) mbar_init(&tempty[b], C::FOLD_WARPS);
    mbar_init(&drain, C::ISSUERS);
    mbar_init(&red_full, C::FOLD_WARPS * (S - 1));  // every fold warp of every other CTA
    mbar_init(&red_done, C::FOLD_WARPS);            // the leader's fold warps
    ctl.abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0 && first_tile < ntiles) {  // as in the unsplit kernel
    const int wt = first_tile / num_x;
    for (int kb = kb_lo; kb < kb_hi && kb < kb_lo + STAGES; ++kb) tma_prefetch_l2_2d(&tmW, kb * BK, wt * BM);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA's barriers exist before any remote arrive
  tc_fence_after();
  grid_dependents_launch();  // as in the unsplit kernel
  grid_dependency_wait();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = first_tile; tile < ntiles && ok; tile += tile_step) {
        const int wt = tile / num_x, xt = tile - wt * num_x;
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, kWaitTimeoutNs, &ctl.abort)) {
            ok = false;
            break;
          }
          uint8_t *w_s = smem + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          tma_load_2d(w_s, &tmW, kb * BK, wt * BM, &full[s]);
          tma_load_2d(w_s + C::W_BYTES, &tmX, kb * BK, xt * BX, &full[s]);
        }
      }
      if (!ok) {
        flag_abort(&ctl, dev_status);
        drain_stages<STAGES>(full, it);
      }
    }
  } else if (warp < C::FIRST_FOLD_WARP) {
    // MMA issuers, alternate k-blocks (as in the unsplit kernel)
    if (lane == 0) {
      const int me = warp - 1;
      int it = 0, kc = 0;
      bool ok = true;
      for (int tile = first_tile; tile < ntiles && ok; tile += tile_step) {
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it, ++kc) {
          if (C::ISSUERS > 1 && kc % C::ISSUERS != me) continue;
          const int b = kc % C::NBUF;
          const int s = it % STAGES;
          const uint32_t w0 = smem_u32(smem + s * C::STAGE_BYTES);
          const uint64_t wdesc = sdesc_k_sw128(w0), xdesc = sdesc_k_sw128(w0 + C::W_BYTES);
          const uint32_t d = tmem + static_cast<uint32_t>(b * BX);
          // the partial buffer (usually free) before the stage (the copy in
          // flight from HBM is the critical wait); descriptors formed first
          if (!mbar_wait(&tempty[b], ((kc / C::NBUF) & 1) ^ 1, kWaitTimeoutNs, &ctl.abort) ||
              !mbar_wait(&full[s], (it / STAGES) & 1, kWaitTimeoutNs, &ctl.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) mma_f8f6f4(d, wdesc + 2 * k, xdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
          tc_commit(&empty[s]);
        }
      }
      if (!ok) flag_abort(&ctl, dev_status);
      tc_commit(&drain);
      mbar_wait(&drain, 0, kDrainTimeoutNs, nullptr);
    }
  } else {
    constexpr int BXW = C::BXW;
    const int fw = warp - C::FIRST_FOLD_WARP;  // fold warp 0 .. FOLD_WARPS - 1
    const int quarter = warp & 3;              // the tensor-memory lanes (W rows) this warp may read
    const int col0 = (fw / 4) * BXW;           // its activation rows within the tile
    const int row = quarter * 32 + lane;       // this thread's W row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr int XR = (BXW + 31) / 32;  // activation-scale registers per lane
    float *red = reinterpret_cast<float *>(smem + STAGES * C::STAGE_BYTES);  // [BX][128]
    float *cbuf = reinterpret_cast<float *>(smem + STAGES * C::STAGE_BYTES + C::RED_BYTES) + fw * 2 * BXW;
    uint16_t *otile = reinterpret_cast<uint16_t *>(smem + STAGES * C::STAGE_BYTES + C::RED_BYTES + C::CBUF_BYTES) +
                      fw * BXW * 32;
    int kc = 0, tn = 0;
    bool ok = true;
    float acc[BXW];
    for (int tile = first_tile; tile < ntiles && ok; tile += tile_step, ++tn) {
      const int wt = tile / num_x, xt = tile - wt * num_x;
      const int m0 = xt * BX + col0;
      const float *sb_blk = sb + static_cast<int64_t>(wt) * KB;  // one 128-row weight block per tile
#pragma unroll
      for (int j = 0; j < BXW; ++j) acc[j] = 0.0f;
      // scale slots as in the unsplit kernel, over this CTA's k-blocks [kb_lo, kb_hi)
      auto load_sx = [&](int kbq, float (&dst)[XR]) {
        const int kq = min(kbq, kb_hi - 1);
#pragma unroll
        for (int r = 0; r < XR; ++r) dst[r] = __ldg(sa + static_cast<int64_t>(kq) * M + min(m0 + 32 * r + lane, M - 1));
      };
      float xs0[XR], xs1[XR];
      load_sx(kb_lo, xs0);
      load_sx(kb_lo + 1, xs1);
      float ws0 = __ldg(sb_blk + kb_lo), ws1 = __ldg(sb_blk + min(kb_lo + 1, kb_hi - 1));
      auto fold_one = [&](int kb, float (&xs)[XR], float &ws) -> bool {
        const int b = kc % C::NBUF;
        // products in the warp's slot for this k-block's parity, read back as
        // broadcasts (as in the unsplit kernel's register path)
        float *cs = cbuf + (kc & 1) * BXW;
#pragma unroll
        for (int q = 0; q < XR; ++q)
          if (32 * q + lane < BXW) cs[32 * q + lane] = ws * xs[q];
        load_sx(kb + 2, xs);
        ws = __ldg(sb_blk + min(kb + 2, kb_hi - 1));
        __syncwarp();
        const bool got = mbar_wait(&empty[kc % STAGES], (kc / STAGES) & 1, kWaitTimeoutNs, &ctl.abort);
        if (!__all_sync(0xffffffffu, got)) return false;
        tc_fence_after();
        const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(b * BX + col0);
        uint32_t r[BXW];
        tmem_ld_chunk<BXW>(taddr, r);
        tmem_wait_ld_regs(r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[b]);
        const float4 *c4 = reinterpret_cast<const float4 *>(cs);
#pragma unroll
        for (int i = 0; i < BXW / 4; ++i) {
          const float4 c = c4[i];
          acc[4 * i + 0] = fmaf(c.x, __uint_as_float(r[4 * i + 0]), acc[4 * i + 0]);
          acc[4 * i + 1] = fmaf(c.y, __uint_as_float(r[4 * i + 1]), acc[4 * i + 1]);
          acc[4 * i + 2] = fmaf(c.z, __uint_as_float(r[4 * i + 2]), acc[4 * i + 2]);
          acc[4 * i + 3] = fmaf(c.w, __uint_as_float(r[4 * i + 3]), acc[4 * i + 3]);
        }
        ++kc;
        return true;
      };
      for (int kb = kb_lo; kb < kb_hi && ok; kb += 2) {
        ok = fold_one(kb, xs0, ws0);
        if (ok && kb + 1 < kb_hi) ok = fold_one(kb + 1, xs1, ws1);
      }
      if (!ok) break;
      {
        const uint32_t phase = static_cast<uint32_t>(tn & 1);
        if (rank != 0) {
          // leave this CTA's partial for the leader and wait until it has been read
#pragma unroll
          for (int j = 0; j < BXW; ++j) red[(col0 + j) * BM + row] = acc[j];
          __syncwarp();
          if (lane == 0) mbar_arrive_release_cluster(cluster_addr(&red_full, 0));
          const bool done = mbar_wait(&red_done, phase, kWaitTimeoutNs, &ctl.abort);
          if (!__all_sync(0xffffffffu, done)) ok = false;
          continue;
        }
        const bool in = mbar_wait_acquire_cluster(&red_full, phase, kWaitTimeoutNs);
        if (!__all_sync(0xffffffffu, in)) {
          ok = false;
          break;
        }
        for (int p = 1; p < S; ++p) {
          const uint32_t base = cluster_addr(red, static_cast<uint32_t>(p)) + 4u * static_cast<uint32_t>(row);
#pragma unroll
          for (int j = 0; j < BXW; ++j)
            acc[j] += ld_shared_cluster_f32(base + 4u * static_cast<uint32_t>((col0 + j) * BM));
        }
        __syncwarp();
        if (lane == 0)
          for (int p = 1; p < S; ++p) mbar_arrive_release_cluster(cluster_addr(&red_done, static_cast<uint32_t>(p)));
      }
      // output through the warp's shared tile, 16-byte row stores (as in the unsplit kernel)
#pragma unroll
      for (int j = 0; j < BXW; ++j) otile[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j]));
      __syncwarp();
      const int ncol = wt * BM + quarter * 32 + (lane & 3) * 8;
#pragma unroll
      for (int i = 0; i < BXW / 8; ++i) {
        const int j = 8 * i + (lane >> 2);
        const int m = m0 + j;
        if (m < M && ncol < N && FP8BS_GUARD(static_cast<int64_t>(m) * N + ncol, 8, static_cast<int64_t>(M) * N))
          *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(m) * N + ncol) =
              *reinterpret_cast<const uint4 *>(otile + j * 32 + (lane & 3) * 8);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) flag_abort(&ctl, dev_status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// =====================================================================
// Tensor-memory accumulating kernel: epilogue-scaled (KIND_EPI), block-scaled
// MXFP8 (KIND_MX8: UE8M0 scale per 32 K) or NVFP4 (KIND_NVF4: E2M1 operands,
// E4M3 scale per 16 K, fp32 tensor scales applied in the epilogue)
// =====================================================================
// KIND_MX8W: MXFP8 with both operands' scales in the staged-four-times
// layout (each 512-byte atom stored four times in a row, 2048 bytes).
constexpr int KIND_EPI = 0, KIND_MX8 = 1, KIND_NVF4 = 2, KIND_MX8W = 3;

// A stage always holds 128 bytes of K per row: 128 fp8 or 256 fp4 elements.
// Scale atoms (128 rows x 4 scales, 512 bytes) per stage and 128-row block:
// one for MXFP8 (4 x 32 K), four for NVFP4 (4 x 4 x 16 K).
template <int KIND, int BN, int STAGES, int NACC>
struct AccCfg {
  static constexpr bool MX = KIND != KIND_EPI;
  static constexpr int ATOMS = KIND == KIND_NVF4 ? 4 : (MX ? 1 : 0);
  // KIND_MX8W: a stage's atoms reach tensor memory in two copies instead of
  // three. Each tcgen05.cp costs tensor-pipe time whatever its size, and the
  // 128-lane copy shapes put row r of their source in lane r, so an atom
  // staged four times over (row r = atom row r % 32: what .32x128b.warpx4
  // replicates to the four lane quarters) lets one .128x256b copy take both
  // W atoms (2048 bytes apart) and one .128x128b copy X's; tensor memory ends
  // up the same, byte for byte.
  static constexpr bool WIDE = KIND == KIND_MX8W;
  static constexpr int ATOM_BYTES = WIDE ? 2048 : 512;  // one atom as staged
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int SFA_BYTES = ATOM_BYTES * ATOMS;
  static constexpr int SFB_BYTES = ATOM_BYTES * ATOMS * (BN / 128);
  static_assert(!WIDE || BN == 256, "the wide copy takes two 128-row W atoms");
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int STAGE_STRIDE = (STAGE_BYTES + 1023) / 1024 * 1024;
  static constexpr int CONSUMER_WARPS = 4 * (BN / 128);
  // warp 0 producer, warp 1 MMA issuer, (NVFP4) warps 2 and 3 copy the stage's
  // scale atoms into tensor memory, then the epilogue warps. MXFP8 has three
  // atoms per stage: the MMA thread copies them right before its MMAs (a copier
  // warp and its ready barrier put ~400 cycles of hand-off on the stage ring,
  // which is latency-bound; 2.4 % slower, same-process A/B).
  static constexpr bool COPIER = MX && SF_COPIER && (KIND == KIND_NVF4 || MX8_COPIER);
  // copier warps: the stage's atoms are split round-robin between them
  static constexpr int COPIERS = !COPIER ? 0 : (KIND == KIND_NVF4 ? NVF4_COPIERS : 1);
  static constexpr int FIRST_CONSUMER_WARP = 2 + COPIERS;
  // NVFP4 (12 atom copies per stage): the atoms travel on their own barrier
  // (sf_full) so the copiers start before the operands land, and the MMA
  // thread waits for both (measured +4 %). With an MXFP8 copier warp
  // (MX8_COPIER) the copier waits for the whole stage and sf_ready implies
  // full.
  static constexpr bool SF_SPLIT = COPIER && KIND == KIND_NVF4;
  static constexpr int THREADS = 32 * FIRST_CONSUMER_WARP + 32 * CONSUMER_WARPS;
  // tensor-memory columns per stage (WIDE: 12 used, 16 so that each stage's
  // columns start 16-aligned)
  static constexpr int SF_COLS = WIDE ? 16 : 4 * ATOMS * (1 + BN / 128);
  static constexpr int ACC_COLS = NACC * BN;                    // NACC accumulators (2: epilogue overlaps MMA)
  static constexpr uint32_t TMEM_COLS = ACC_COLS + STAGES * SF_COLS <= 256 ? 256 : 512;
  static constexpr int SMEM = STAGES * STAGE_STRIDE + 1024;
  static_assert(ACC_COLS + STAGES * SF_COLS <= 512, "tensor memory budget");
  static_assert(!WIDE || !COPIER, "the MMA thread copies the staged atoms itself");
};

// A stage's scale atoms, shared memory (A's atoms, then B's per 128-row block;
// sf_desc: descriptor of the first atom, an atom 512 bytes further on is 32
// units of 16 bytes further) -> tensor memory (sf_tmem). MXFP8: one atom per
// 128 rows at +4 columns per block. NVFP4: four atoms per 128 rows; A's atom k
// at +4k, B's at +8k (+4 for the second 128-row block).
// With several copiers, copier `part` of `nparts` issues the atoms whose index
// (in the order below) is congruent to part.
template <int KIND, int BN>
__device__ __forceinline__ void copy_scale_atoms(uint32_t sf_tmem, uint64_t sf_desc, int part = 0, int nparts = 1) {
  constexpr uint64_t ATOM = 512 >> 4;
  if constexpr (KIND == KIND_NVF4) {
    constexpr int PER_K = 1 + BN / 128;  // A's atom, then B's per 128-row block
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if ((k * PER_K) % nparts == part) tmem_cp_32x128b_warpx4(sf_tmem + 4 * k, sf_desc + ATOM * k);
#pragma unroll
      for (int j = 0; j < BN / 128; ++j)
        if ((k * PER_K + 1 + j) % nparts == part)
          tmem_cp_32x128b_warpx4(sf_tmem + 16 + 8 * k + 4 * j, sf_desc + ATOM * (4 + 4 * j + k));
    }
  } else {
    if (part == 0) tmem_cp_32x128b_warpx4(sf_tmem, sf_desc);
#pragma unroll
    for (int j = 0; j < BN / 128; ++j)
      if ((1 + j) % nparts == part) tmem_cp_32x128b_warpx4(sf_tmem + 4 + 4 * j, sf_desc + ATOM * (1 + j));
  }
}

template <int KIND, int BN, int STAGES, int NACC>
__global__ void __launch_bounds__(AccCfg<KIND, BN, STAGES, NACC>::THREADS, 1)
    gemm_tmem_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const float *__restrict__ sa, int sa_per_row, const float *__restrict__ sb, int sb_per_col,
                     const uint8_t *__restrict__ sfa, const uint8_t *__restrict__ sfb, uint16_t *__restrict__ out,
                     int M, int N, int K, uint32_t idesc, int *dev_status, int group_m, uint64_t wait_ns) {
  using C = AccCfg<KIND, BN, STAGES, NACC>;
  constexpr bool MX = C::MX;
  constexpr bool F4 = KIND == KIND_NVF4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  // sf_full[s]: stage s's scale atoms have landed in shared memory (their own
  // barrier, so the copier does not wait for the 48 KB of operands);
  // sf_ready[s]: they are in tensor memory (copier warps)
  __shared__ uint64_t full[STAGES], empty[STAGES], sf_full[STAGES], sf_ready[STAGES], afull[NACC], aempty[NACC],
      drain, cdrain;
  __shared__ SharedCtl ctl;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // k-blocks of 128 bytes per row (K % 256 == 0 for NVFP4)
  const int KB = F4 ? K / 256 : (K + BK - 1) / BK;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int ntiles = num_m * num_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 1);
      mbar_init(&sf_ready[s], C::COPIERS > 0 ? C::COPIERS : 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], C::CONSUMER_WARPS);
    }
    mbar_init(&drain, 1);
    mbar_init(&cdrain, C::COPIERS > 0 ? C::COPIERS : 1);  // every copier's copies are done
    ctl.abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      const int nblk128_b = (N + 127) / 128;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        int mt, nt;
        tile_coords(tile, num_m, num_n, group_m, mt, nt);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          uint8_t *st = smem + s * C::STAGE_STRIDE;
          // scale atoms (block-scaled kinds): [row block][atom along K] x 512
          // bytes, a stage's atoms of one 128-row block contiguous. With
          // SF_SPLIT they go first, on their own barrier, so the copiers start
          // early; otherwise they follow the operands on the stage's barrier
          // (operands first measured 2.6 % faster there).
          auto load_atoms = [&](uint64_t *bar) {
            constexpr int AB = C::ATOM_BYTES * C::ATOMS;
            bulk_load(st + C::A_BYTES + C::B_BYTES, sfa + (static_cast<int64_t>(mt) * KB + kb) * AB, AB, bar);
#pragma unroll
            for (int j = 0; j < BN / 128; ++j) {
              int nb = nt * (BN / 128) + j;
              nb = nb < nblk128_b ? nb : nblk128_b - 1;  // rows past N are zero; any finite scale will do
              bulk_load(st + C::A_BYTES + C::B_BYTES + AB + AB * j, sfb + (static_cast<int64_t>(nb) * KB + kb) * AB,
                        AB, bar);
            }
          };
          if constexpr (C::SF_SPLIT) {
            mbar_arrive_expect_tx(&sf_full[s], C::SFA_BYTES + C::SFB_BYTES);
            load_atoms(&sf_full[s]);
          }
          mbar_arrive_expect_tx(&full[s], C::SF_SPLIT ? C::A_BYTES + C::B_BYTES : C::STAGE_BYTES);
          tma_load_2d(st, &tmA, kb * BK, mt * BM, &full[s]);
          tma_load_2d(st + C::A_BYTES, &tmB, kb * BK, nt * BN, &full[s]);
          if constexpr (MX && !C::SF_SPLIT) load_atoms(&full[s]);
        }
      }
      if (!ok) {
        flag_abort(&ctl, dev_status);
        drain_stages<STAGES>(full, it);
        if (C::SF_SPLIT) drain_stages<STAGES>(sf_full, it);
      }
    }
  } else if (C::COPIER && warp >= 2 && warp < C::FIRST_CONSUMER_WARP) {
    // scale-factor copiers: stage s's atoms smem -> tensor memory once its
    // copies have landed; the slot's previous MMA is done (the producer waited
    // on it before loading the stage)
    if (lane == 0) {
      const int part = warp - 2;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint64_t sf_desc = sdesc_plain_32x16(smem_u32(smem + s * C::STAGE_STRIDE) + C::A_BYTES + C::B_BYTES);
          if (!mbar_wait(C::SF_SPLIT ? &sf_full[s] : &full[s], (it / STAGES) & 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          copy_scale_atoms<KIND, BN>(tmem + static_cast<uint32_t>(C::ACC_COLS + s * C::SF_COLS), sf_desc, part,
                                     C::COPIERS);
          tc_commit(&sf_ready[s]);
        }
      }
      if (!ok) flag_abort(&ctl, dev_status);
      tc_commit(&cdrain);
      mbar_wait(&cdrain, 0, kDrainTimeoutNs, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, tc = 0;
      bool ok = true;
      const uint32_t sf_col0 = static_cast<uint32_t>(C::ACC_COLS);
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++tc) {
        const int b = tc % NACC;
        if (!mbar_wait(&aempty[b], ((tc / NACC) & 1) ^ 1, wait_ns, &ctl.abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t a0 = smem_u32(smem + s * C::STAGE_STRIDE);
          const uint32_t b0 = a0 + C::A_BYTES;
          // descriptors formed before the waits (the MMAs follow the last wait
          // directly); K step k advances both by 32 bytes (2 units of 16)
          const uint64_t adesc = sdesc_k_sw128(a0), bdesc = sdesc_k_sw128(b0);
          // the operands, and (block-scaled kinds) the scale atoms in tensor
          // memory; without SF_SPLIT sf_ready[s] implies full[s]
          if ((!C::COPIER || C::SF_SPLIT) && !mbar_wait(&full[s], (it / STAGES) & 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          if (C::COPIER && !mbar_wait(&sf_ready[s], (it / STAGES) & 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if constexpr (C::WIDE) {
            // X's staged atom at +0 -> columns +8..11; W's two at +2048 and
            // +4096 (16-byte column chunks 0 and 1 of one source) -> +0..7
            const uint32_t sft = tmem + sf_col0 + static_cast<uint32_t>(s * C::SF_COLS);
            const uint32_t sf0 = b0 + C::B_BYTES;
            tmem_cp_128x256b(sft, sdesc_plain(sf0 + C::SFA_BYTES, C::ATOM_BYTES, 128));
            tmem_cp_128x128b(sft + 8, sdesc_plain(sf0, 128, 128));
          } else if constexpr (MX && !C::COPIER) {
            copy_scale_atoms<KIND, BN>(tmem + sf_col0 + static_cast<uint32_t>(s * C::SF_COLS),
                                       sdesc_plain_32x16(b0 + C::B_BYTES));
          }
          if (F4) {
            // NVFP4: one scale atom per MMA (K = 64, four 16-element scales per
            // row); A's atom k at column +4k, B's at +8k (second 128-row block
            // of B at +4, as the block-scaled MMA reads a 256-row B)
            const uint32_t sfa_t = tmem + sf_col0 + static_cast<uint32_t>(s * C::SF_COLS);
            const uint32_t sfb_t = sfa_t + 16;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_mxf4nvf4(d, adesc + 2 * k, bdesc + 2 * k, idesc, sfa_t + 4 * k,
                           sfb_t + 8 * k, (kb > 0 || k > 0) ? 1u : 0u);
          } else if (MX) {
            // X's atom, then W's (the second 128-row block of W 4 columns on,
            // as the block-scaled MMA reads a 256-row B)
            const uint32_t sf_t = tmem + sf_col0 + static_cast<uint32_t>(s * C::SF_COLS);
            const uint32_t sfa_t = C::WIDE ? sf_t + 8 : sf_t;
            const uint32_t sfb_t = C::WIDE ? sf_t : sf_t + 4;
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)
              mma_mxf8f6f4(d, adesc + 2 * k, bdesc + 2 * k,
                           idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29), sfa_t, sfb_t,
                           (kb > 0 || k > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)
              mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, idesc,
                         (kb > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        if (!ok) break;
        tc_commit(&afull[b]);
      }
      if (!ok) flag_abort(&ctl, dev_status);
      tc_commit(&drain);
      mbar_wait(&drain, 0, kDrainTimeoutNs, nullptr);
    }
  } else {
    // ------------------------------------------------ epilogue consumers
    const int cw = warp - C::FIRST_CONSUMER_WARP;
    const int quarter = warp & 3;
    const int half = cw >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int tc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tc) {
      int mt, nt;
      tile_coords(tile, num_m, num_n, group_m, mt, nt);
      const int b = tc % NACC;
      const int m = mt * BM + quarter * 32 + lane;
      const bool row_ok = m < M;
      const int n0 = nt * BN + half * 128;
      const bool got = mbar_wait(&afull[b], (tc / NACC) & 1, wait_ns, &ctl.abort);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s_row = 1.0f;
      if (!MX) s_row = row_ok ? __ldg(sa + (sa_per_row ? m : 0)) : 0.0f;
      // drain this thread's 128 accumulator columns into registers first and
      // hand the accumulator back, so the next tile's MMAs overlap the stores
      uint32_t r[4][32];
      const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(b * BN + half * 128);
      tmem_ld_32x32b_x32(taddr, r[0]);
      tmem_ld_32x32b_x32(taddr + 32, r[1]);
      tmem_ld_32x32b_x32(taddr + 64, r[2]);
      tmem_ld_32x32b_x32(taddr + 96, r[3]);
      tmem_wait_ld_regs(r[0]);
      tmem_wait_ld_regs(r[1]);
      tmem_wait_ld_regs(r[2]);
      tmem_wait_ld_regs(r[3]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[b]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int nc = n0 + 32 * c;
        if (row_ok && nc < N) {
          float v[32];
          if (F4) {
            // the two fp32 tensor scales (sa, sb point at them)
            const float g = __ldg(sa) * __ldg(sb);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[c][i]) * g;
          } else if (MX) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[c][i]);
          } else if (sb_per_col) {
            const float4 *sbv = reinterpret_cast<const float4 *>(sb + nc);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 q = (nc + 4 * i < N) ? __ldg(sbv + i) : make_float4(0.f, 0.f, 0.f, 0.f);
              v[4 * i + 0] = __uint_as_float(r[c][4 * i + 0]) * (s_row * q.x);
              v[4 * i + 1] = __uint_as_float(r[c][4 * i + 1]) * (s_row * q.y);
              v[4 * i + 2] = __uint_as_float(r[c][4 * i + 2]) * (s_row * q.z);
              v[4 * i + 3] = __uint_as_float(r[c][4 * i + 3]) * (s_row * q.w);
            }
          } else {
            const float s = s_row * __ldg(sb);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[c][i]) * s;
          }
          store_row32(out, static_cast<int64_t>(m) * N + nc, static_cast<int64_t>(M) * N, v, N - nc);
        }
      }
    }
    if (!ok && lane == 0) flag_abort(&ctl, dev_status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// =====================================================================
// MXFP8 GEMM on CTA pairs (tcgen05 cta_group::2)
// =====================================================================
// A 256 x 256 tile per pair of CTAs (a cluster of two): each CTA loads its own
// 128 rows of X and 128 rows of W (its half of the pair MMA's B operand), its
// rows' scale atom and both of the tile's W scale atoms (every CTA's tensor
// core applies the scales of all 256 W rows). A k-block therefore moves 32 KB
// of operands per CTA through shared memory instead of 48 KB, which leaves
// room for six stages against the copy latency that bounds the single-CTA
// kernel. The even CTA issues the scale copies and the pair MMAs; the
// accumulator (128 rows x 256 columns per CTA) stays in tensor memory for all
// of K and both CTAs' epilogue warps drain their halves, then release it to
// the even CTA. Measured against the single-CTA kernel (same process): 4 %
// faster on 4096 x 14336 x 4096, 3 % slower on 8192^3 and 5 % slower on
// 2048 x 8192 x 8192. Both are bound by the three scale-atom copies per
// k-block, not by the copies from HBM (without them this kernel ran 14 %
// faster; without the operand copies, 1 %), so the shape rule keeps the
// single-CTA kernel and this one is reached through fp8_debug_gemm_mx_pairs.
#ifndef MX_PAIR_STAGES
#define MX_PAIR_STAGES 6
#endif

template <int STAGES>
struct MxPairCfg {
  static constexpr int A_BYTES = BM * BK;   // this CTA's 128 rows of X
  static constexpr int B_BYTES = 128 * BK;  // this CTA's 128 rows of W
  static constexpr int SFA_BYTES = 512;     // the scale atom of this CTA's X rows
  static constexpr int SFB_BYTES = 1024;    // the atoms of the tile's two 128-row W blocks
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int STAGE_STRIDE = (STAGE_BYTES + 1023) / 1024 * 1024;
  static constexpr int TM = 256, TN = 256;
  static constexpr int CONSUMER_WARPS = 8;  // per CTA: 4 lane quarters x 2 column halves
  static constexpr int FIRST_CONSUMER_WARP = 2;
  static constexpr int THREADS = 32 * (FIRST_CONSUMER_WARP + CONSUMER_WARPS);
  static constexpr int SF_COLS = 12;        // tensor-memory columns per stage: X atom 4, W atoms 8
  static constexpr int ACC_COLS = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(ACC_COLS + STAGES * SF_COLS <= 512, "tensor memory");
  static constexpr int SMEM = STAGES * STAGE_STRIDE + 1024;
  static_assert(SMEM + 512 <= 232448, "shared memory budget");
};

template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MxPairCfg<STAGES>::THREADS, 1)
    gemm_mx_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                        uint16_t *__restrict__ out, int M, int N, int K, uint32_t idesc, int *dev_status, int group_m,
                        uint64_t wait_ns) {
  using C = MxPairCfg<STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  // full[s]: both CTAs' copies of stage s have landed (even CTA's barrier);
  // empty[s]: the pair MMAs of stage s are done (multicast commit);
  // afull / aempty: the accumulator holds a finished tile / both CTAs'
  // epilogue warps have read it (even CTA's barrier)
  __shared__ uint64_t full[STAGES], empty[STAGES], afull, aempty, drain;
  __shared__ SharedCtl ctl;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int KB = (K + BK - 1) / BK;
  const int num_m = (M + C::TM - 1) / C::TM;
  const int num_n = (N + C::TN - 1) / C::TN;
  const int ntiles = num_m * num_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&afull, 1);
    mbar_init(&aempty, 2 * C::CONSUMER_WARPS);  // both CTAs' epilogue warps release to the even CTA
    mbar_init(&drain, 1);
    ctl.abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSA);
    tma_prefetch_desc(&tmSB);
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctl.tmem_base, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t full_lead = cluster_addr(&full[0], 0);  // stage s at + 8 s
  const uint32_t aempty_lead = cluster_addr(&aempty, 0);

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = pair; tile < ntiles && ok; tile += npairs) {
        int mt, nt;
        tile_coords(tile, num_m, num_n, group_m, mt, nt);
        // atom rows: [128-row block][k-block]; blocks past M or N read as zeros
        const int a_atom = (mt * 2 + static_cast<int>(rank)) * KB;
        const int b_atom = nt * 2 * KB;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(&empty[s], ((it / STAGES) & 1) ^ 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          uint8_t *st = smem + s * C::STAGE_STRIDE;
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
          const uint32_t bar = full_lead + 8u * static_cast<uint32_t>(s);
          tma_load_2d_pair(st, &tmA, kb * BK, mt * C::TM + static_cast<int>(rank) * 128, bar);
          tma_load_2d_pair(st + C::A_BYTES, &tmB, kb * BK, nt * C::TN + static_cast<int>(rank) * 128, bar);
          uint8_t *sf = st + C::A_BYTES + C::B_BYTES;
          tma_load_2d_pair(sf, &tmSA, 0, a_atom + kb, bar);
          tma_load_2d_pair(sf + 512, &tmSB, 0, b_atom + kb, bar);
          tma_load_2d_pair(sf + 1024, &tmSB, 0, b_atom + KB + kb, bar);
        }
      }
      if (!ok) {
        flag_abort(&ctl, dev_status);
        if (leader) {
          drain_stages<STAGES>(full, it);
        } else {
          // this CTA's copies complete on the even CTA's barriers; give them time to land
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int it = 0, tc = 0;
      bool ok = true;
      const uint32_t sf_col0 = static_cast<uint32_t>(C::ACC_COLS);
      for (int tile = pair; tile < ntiles && ok; tile += npairs, ++tc) {
        if (!mbar_wait(&aempty, (tc & 1) ^ 1, wait_ns, &ctl.abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t a0 = smem_u32(smem + s * C::STAGE_STRIDE);
          const uint32_t b0 = a0 + C::A_BYTES;
          const uint64_t adesc = sdesc_k_sw128(a0), bdesc = sdesc_k_sw128(b0);
          const uint64_t sf_desc = sdesc_plain_32x16(b0 + C::B_BYTES);
          const uint32_t sfa_t = tmem + sf_col0 + static_cast<uint32_t>(s * C::SF_COLS);
          const uint32_t sfb_t = sfa_t + 4;
          if (!mbar_wait(&full[s], (it / STAGES) & 1, wait_ns, &ctl.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // the stage's three atoms into each CTA's tensor memory right before
          // the MMAs (copies issued further ahead measured slower: 2 k-blocks
          // ahead -10 %, 4 ahead -50 %)
          tmem_cp_32x128b_warpx4_pair(sfa_t, sf_desc);
          tmem_cp_32x128b_warpx4_pair(sfb_t, sf_desc + (512 >> 4));
          tmem_cp_32x128b_warpx4_pair(sfb_t + 4, sf_desc + (1024 >> 4));
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_mxf8f6f4_pair(tmem, adesc + 2 * k, bdesc + 2 * k,
                              idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29), sfa_t,
                              sfb_t, (kb > 0 || k > 0) ? 1u : 0u);
          tc_commit_pair_mc(&empty[s], 0x3);
        }
        if (!ok) break;
        tc_commit_pair_mc(&afull, 0x3);
      }
      if (!ok) flag_abort(&ctl, dev_status);
      tc_commit_pair(&drain);
      mbar_wait(&drain, 0, kDrainTimeoutNs, nullptr);
    }
  } else {
    // ------------------------------------------------ epilogue consumers
    const int cw = warp - C::FIRST_CONSUMER_WARP;
    const int quarter = warp & 3;
    const int half = cw >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int tc = 0;
    bool ok = true;
    for (int tile = pair; tile < ntiles; tile += npairs, ++tc) {
      int mt, nt;
      tile_coords(tile, num_m, num_n, group_m, mt, nt);
      const int m = mt * C::TM + static_cast<int>(rank) * 128 + quarter * 32 + lane;
      const bool row_ok = m < M;
      const int n0 = nt * C::TN + half * 128;
      const bool got = mbar_wait(&afull, tc & 1, wait_ns, &ctl.abort);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // drain this thread's 128 accumulator columns, hand the accumulator back
      // to the even CTA, then store
      uint32_t r[4][32];
      const uint32_t taddr = tmem + lane_base + static_cast<uint32_t>(half * 128);
      tmem_ld_32x32b_x32(taddr, r[0]);
      tmem_ld_32x32b_x32(taddr + 32, r[1]);
      tmem_ld_32x32b_x32(taddr + 64, r[2]);
      tmem_ld_32x32b_x32(taddr + 96, r[3]);
      tmem_wait_ld_regs(r[0]);
      tmem_wait_ld_regs(r[1]);
      tmem_wait_ld_regs(r[2]);
      tmem_wait_ld_regs(r[3]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(aempty_lead);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int nc = n0 + 32 * c;
        if (row_ok && nc < N) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[c][i]);
          store_row32(out, static_cast<int64_t>(m) * N + nc, static_cast<int64_t>(M) * N, v, N - nc);
        }
      }
    }
    if (!ok && lane == 0) flag_abort(&ctl, dev_status);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the even CTA's MMAs and both CTAs' tensor-memory reads are done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

// =====================================================================
// Bounded-wait check: a barrier nothing ever arrives on
// =====================================================================
__global__ void wait_probe_kernel(int *dev_status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0, timeout_ns, nullptr) && dev_status != nullptr)
      atomicExch(dev_status, static_cast<int>(FP8_ERR_TIMEOUT));
  }
}

// ------------------------------------------------------------------ host
template <typename KernelT>
bool ensure_smem(KernelT kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess;
}

// X rows a raster group may hold: well inside one die's half of the L2.
#ifndef FP8BS_RASTER_MB
#define FP8BS_RASTER_MB 32
#endif
constexpr int64_t kRasterGroupBytes = int64_t{FP8BS_RASTER_MB} << 20;

int raster_group(int64_t M, int64_t K) {
  const int64_t num_m = (M + BM - 1) / BM;
  int64_t g = kRasterGroupBytes / (static_cast<int64_t>(BM) * (K > 0 ? K : 1));
  if (g < 1) g = 1;
  if (g > num_m) g = num_m;
  return static_cast<int>(g);
}

int persistent_grid(int ntiles) {
  const int sms = device_sm_count();
  return ntiles < sms ? ntiles : sms;
}

// Launch with programmatic stream serialization: the kernel may begin (and do
// its setup) while the previous kernel in the stream finishes; it waits for
// that kernel's results with grid_dependency_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// K splits for the decode kernel. Without a split, a tile is one 128-row W block
// streamed over all of K by one CTA, and when there are fewer tiles than SMs the
// idle SMs' share of HBM bandwidth is lost. With S splits the tile's K range is
// spread over a cluster of S CTAs. S minimises the largest number of CTAs any SM
// runs divided by S (the time one SM needs for its share, in units of a whole
// tile), with all CTAs resident at once (units * S <= capacity), S <= 8 (portable
// cluster size) and at least two k-blocks per CTA; ties go to the smaller S.
int swap_split(int64_t units, int64_t KB, int sms, int capacity) {
  if (units * 10 >= static_cast<int64_t>(sms) * 9) return 1;  // already fills the GPU
  int best = 1;
  double best_t = static_cast<double>((units + sms - 1) / sms);
  for (int S = 2; S <= 8; ++S) {
    if (2 * S > KB || units * S > capacity) break;
    const double t = static_cast<double>((units * S + sms - 1) / sms) / S;
    if (t < best_t - 1e-9) {
      best = S;
      best_t = t;
    }
  }
  return best;
}

template <int BX, int ST>
fp8_status_t launch_fold_swap(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb, int a_fmt,
                              int b_fmt, uint16_t *out, int64_t M, int64_t N, int64_t K, int *dev_status,
                              cudaStream_t stream, uint64_t wait_ns, bool allow_clusters) {
  CUtensorMap tx, tw;
  if (!make_tmap_u8(&tx, a, M, K, K, BX, BK) || !make_tmap_u8(&tw, b, N, K, K, BM, BK)) return FP8_ERR_CUDA;
  const int ntiles = static_cast<int>(((M + BX - 1) / BX) * ((N + BM - 1) / BM));
  // the MMA's A operand is W (format b_fmt), its B operand is X (a_fmt)
  const uint32_t idesc = idesc_f8f6f4(b_fmt, a_fmt, BM, BX);
  const int sms = device_sm_count();
  if (allow_clusters && ntiles * 10 < sms * 9 && K / BK >= 4) {
    // split-K clusters; 5 stages (the fewest the stage-barrier parity allows)
    // so that two CTAs fit on an SM where registers allow
    constexpr int STS = 5;
    using CS = SwapSplitCfg<BX, STS>;
    auto kern = gemm_fold_swap_split_kernel<BX, STS>;
    if (!ensure_smem(kern, CS::SMEM)) return FP8_ERR_CUDA;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, CS::THREADS, CS::SMEM) != cudaSuccess) occ = 1;
    const int S = swap_split(ntiles, K / BK, sms, std::max(occ, 1) * sms);
    if (S > 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(ntiles * S), 1, 1);
      cfg.blockDim = dim3(CS::THREADS, 1, 1);
      cfg.dynamicSmemBytes = CS::SMEM;
      cfg.stream = stream;
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(S);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 2;
      const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tx, tw, sa, sb, out, static_cast<int>(M),
                                               static_cast<int>(N), static_cast<int>(K), idesc, dev_status);
      note_launches(1);
      return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
    }
  }
  using C = SwapCfg<BX, ST>;
  auto kern = gemm_fold_swap_kernel<BX, ST>;
  if (!ensure_smem(kern, C::SMEM)) return FP8_ERR_CUDA;
  // the scales by tensor copies when their rows are whole 16-byte units:
  // s_x as [K/128 rows x M], s_w as [N/128 blocks x K/128]
  const int64_t KB = K / BK;
  CUtensorMap tsx = tx, tsw = tx;  // not read on the register path
  int sc_tma = M % 4 == 0 && KB % 4 == 0 && reinterpret_cast<uintptr_t>(sa) % 16 == 0 &&
               reinterpret_cast<uintptr_t>(sb) % 16 == 0;
  if (sc_tma && (!make_tmap_f32(&tsx, sa, KB, M, M, C::KBC, BX) ||
                 !make_tmap_f32(&tsw, sb, (N + BM - 1) / BM, KB, KB, 1, C::KBC)))
    return FP8_ERR_CUDA;
  if (launch_dependent(kern, static_cast<unsigned>(persistent_grid(ntiles)), C::THREADS, C::SMEM, stream, tx, tw,
                       tsx, tsw, sc_tma, sa, sb, out, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                       idesc, dev_status, wait_ns) != cudaSuccess)
    return FP8_ERR_CUDA;
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

template <int QFMT>
fp8_status_t launch_fold_pairs(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb, int a_fmt,
                               int b_fmt, uint16_t *out, uint8_t *q_out, float *q_scales, int64_t M, int64_t N,
                               int64_t K, int *dev_status, cudaStream_t stream) {
  constexpr int ST = FOLD_PAIR_STAGES;
  using C = FoldPairCfg<ST>;
  CUtensorMap ta, tb, to;
  if (!make_tmap_u8(&ta, a, M, K, K, 128, BK) || !make_tmap_u8(&tb, b, N, K, K, 128, BK)) return FP8_ERR_CUDA;
  if (QFMT < 0 ? !make_tmap_u16(&to, out, M, N, N, 32, 64) : !make_tmap_u8(&to, q_out, M, N, N, 32, 128))
    return FP8_ERR_CUDA;
  auto kern = gemm_fold_pair_kernel<ST, QFMT>;
  if (!ensure_smem(kern, C::SMEM) || !reg_split_fits(kern, C::THREADS, C::REGS_NEEDED)) return FP8_ERR_CUDA;
  const int64_t ntiles = ((M + C::TM - 1) / C::TM) * ((N + C::TN - 1) / C::TN);
  const int64_t pairs = std::min<int64_t>(ntiles, device_sm_count() / 2);
  // raster groups in units of 256-row pair tiles
  int64_t g = kRasterGroupBytes / (static_cast<int64_t>(C::TM) * K);
  g = std::max<int64_t>(1, std::min<int64_t>(g, (M + C::TM - 1) / C::TM));
  kern<<<static_cast<unsigned>(2 * pairs), C::THREADS, C::SMEM, stream>>>(
      ta, tb, to, sa, sb, q_scales, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
      idesc_f8f6f4(a_fmt, b_fmt, 256, 256), dev_status, static_cast<int>(g));
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// CTA pairs need at least 256 rows and enough pair tiles to fill the GPU.
bool use_pairs(int64_t M, int64_t N) {
  const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
  return FOLD_USE_PAIRS && M > 128 && 2 * pair_tiles >= device_sm_count();
}

template <int BN, int ST, int NBUF, int QFMT>
fp8_status_t launch_fold_cfg(const CUtensorMap &ta, const CUtensorMap &to, const uint8_t *b, const float *sa,
                             const float *sb, float *q_scales, int a_fmt, int b_fmt, int64_t M, int64_t N, int64_t K,
                             int *dev_status, cudaStream_t stream, uint64_t wait_ns) {
  using C = FoldCfg<BN, ST, NBUF>;
  CUtensorMap tb;
  if (!make_tmap_u8(&tb, b, N, K, K, BN, BK)) return FP8_ERR_CUDA;
  auto kern = gemm_fold_kernel<BN, ST, QFMT, NBUF>;
  if (!ensure_smem(kern, C::SMEM) || !reg_split_fits(kern, C::THREADS, C::REGS_NEEDED)) return FP8_ERR_CUDA;
  const int ntiles = static_cast<int>(((M + 127) / 128) * ((N + BN - 1) / BN));
  if (launch_dependent(kern, static_cast<unsigned>(persistent_grid(ntiles)), C::THREADS, C::SMEM, stream, ta, tb, to,
                       sa, sb, q_scales, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                       idesc_f8f6f4(a_fmt, b_fmt, BM, BN), dev_status, raster_group(M, K), wait_ns) != cudaSuccess)
    return FP8_ERR_CUDA;
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

template <int QFMT>
fp8_status_t launch_fold_tiles(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb, int a_fmt,
                               int b_fmt, uint16_t *out, uint8_t *q_out, float *q_scales, int64_t M, int64_t N,
                               int64_t K, int *dev_status, cudaStream_t stream, uint64_t wait_ns = kWaitTimeoutNs) {
  CUtensorMap ta, to;
  if (!make_tmap_u8(&ta, a, M, K, K, BM, BK)) return FP8_ERR_CUDA;
  // output boxes: 32 rows x 128 bytes (bf16: 64 columns; fp8 codes: 128)
  if (QFMT < 0 ? !make_tmap_u16(&to, out, M, N, N, 32, 64) : !make_tmap_u8(&to, q_out, M, N, N, 32, 128))
    return FP8_ERR_CUDA;
  if constexpr (QFMT < 0 && FOLD_BF16_BN == 128) {
    // 128-wide tiles, four partial buffers: the MMA runs up to four k-blocks
    // ahead of the fold
    return launch_fold_cfg<128, 6, 4, QFMT>(ta, to, b, sa, sb, q_scales, a_fmt, b_fmt, M, N, K, dev_status, stream,
                                            wait_ns);
  } else {
    // Wide tiles when there are enough of them to fill the GPU, else 128-wide.
    const int64_t tiles256 = ((M + 127) / 128) * ((N + 255) / 256);
    if (tiles256 >= device_sm_count())
      return launch_fold_cfg<256, FOLD_WIDE_STAGES, 2, QFMT>(ta, to, b, sa, sb, q_scales, a_fmt, b_fmt, M, N, K,
                                                             dev_status, stream, wait_ns);
    return launch_fold_cfg<128, 6, 2, QFMT>(ta, to, b, sa, sb, q_scales, a_fmt, b_fmt, M, N, K, dev_status, stream,
                                            wait_ns);
  }
}

}  // namespace

FP8BS_OOB_READER(oob_record_gemm)

fp8_status_t launch_gemm_fold(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb, int a_fmt,
                              int b_fmt, uint16_t *out, int64_t M, int64_t N, int64_t K, int *dev_status,
                              cudaStream_t stream, uint64_t wait_ns, bool allow_clusters) {
  // Few activation rows (decode): swap operands so the 128-row MMA side is W.
  // 8-stage rings (5 to 12 stages measured the same or slower)
  if (M <= 16)
    return launch_fold_swap<16, 8>(a, sa, b, sb, a_fmt, b_fmt, out, M, N, K, dev_status, stream, wait_ns,
                                   allow_clusters);
  if (M <= 32)
    return launch_fold_swap<32, 8>(a, sa, b, sb, a_fmt, b_fmt, out, M, N, K, dev_status, stream, wait_ns,
                                   allow_clusters);
  if (M <= 64)
    return launch_fold_swap<64, 8>(a, sa, b, sb, a_fmt, b_fmt, out, M, N, K, dev_status, stream, wait_ns,
                                   allow_clusters);
  if (allow_clusters && use_pairs(M, N))
    return launch_fold_pairs<-1>(a, sa, b, sb, a_fmt, b_fmt, out, nullptr, nullptr, M, N, K, dev_status, stream);
  return launch_fold_tiles<-1>(a, sa, b, sb, a_fmt, b_fmt, out, nullptr, nullptr, M, N, K, dev_status, stream,
                               wait_ns);
}

// The CTA-pair fold kernel regardless of the shape rule (M >= 1): for its tests.
fp8_status_t launch_gemm_fold_pairs(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb, int a_fmt,
                                    int b_fmt, uint16_t *out, int64_t M, int64_t N, int64_t K, int *dev_status,
                                    cudaStream_t stream) {
  return launch_fold_pairs<-1>(a, sa, b, sb, a_fmt, b_fmt, out, nullptr, nullptr, M, N, K, dev_status, stream);
}

fp8_status_t launch_gemm_fold_quantized(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb,
                                        int a_fmt, int b_fmt, int out_fmt, uint8_t *q_out, float *q_scales,
                                        int64_t M, int64_t N, int64_t K, int *dev_status, cudaStream_t stream) {
  if (use_pairs(M, N)) {
    if (out_fmt == FP8_E4M3)
      return launch_fold_pairs<FP8_E4M3>(a, sa, b, sb, a_fmt, b_fmt, nullptr, q_out, q_scales, M, N, K, dev_status,
                                         stream);
    return launch_fold_pairs<FP8_E5M2>(a, sa, b, sb, a_fmt, b_fmt, nullptr, q_out, q_scales, M, N, K, dev_status,
                                       stream);
  }
  if (out_fmt == FP8_E4M3)
    return launch_fold_tiles<FP8_E4M3>(a, sa, b, sb, a_fmt, b_fmt, nullptr, q_out, q_scales, M, N, K, dev_status,
                                       stream);
  return launch_fold_tiles<FP8_E5M2>(a, sa, b, sb, a_fmt, b_fmt, nullptr, q_out, q_scales, M, N, K, dev_status,
                                     stream);
}

fp8_status_t launch_gemm_epilogue_scaled(const uint8_t *a, const float *sa, bool a_token, const uint8_t *b,
                                         const float *sb, bool b_token, int a_fmt, int b_fmt, uint16_t *out,
                                         int64_t M, int64_t N, int64_t K, int *dev_status, cudaStream_t stream,
                                         uint64_t wait_ns) {
  constexpr int BN = 256, ST = 4, NACC = 2;
  using C = AccCfg<KIND_EPI, BN, ST, NACC>;
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, a, M, K, K, BM, BK) || !make_tmap_u8(&tb, b, N, K, K, BN, BK)) return FP8_ERR_CUDA;
  auto kern = gemm_tmem_kernel<KIND_EPI, BN, ST, NACC>;
  if (!ensure_smem(kern, C::SMEM)) return FP8_ERR_CUDA;
  const int ntiles = static_cast<int>(((M + 127) / 128) * ((N + BN - 1) / BN));
  kern<<<persistent_grid(ntiles), C::THREADS, C::SMEM, stream>>>(
      ta, tb, sa, a_token ? 1 : 0, sb, b_token ? 1 : 0, nullptr, nullptr, out, static_cast<int>(M),
      static_cast<int>(N), static_cast<int>(K), idesc_f8f6f4(a_fmt, b_fmt, BM, BN), dev_status, raster_group(M, K),
      wait_ns);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t launch_gemm_mx_pairs(const uint8_t *a, const uint8_t *sfa, const uint8_t *b, const uint8_t *sfb,
                                  int a_fmt, int b_fmt, uint16_t *out, int64_t M, int64_t N, int64_t K,
                                  int *dev_status, cudaStream_t stream, uint64_t wait_ns) {
  constexpr int ST = MX_PAIR_STAGES;
  using C = MxPairCfg<ST>;
  const int64_t KB = (K + BK - 1) / BK;
  // scale atoms as 512-byte rows: [128-row block x k-block] x 128 words
  CUtensorMap ta, tb, tsa, tsb;
  if (!make_tmap_u8(&ta, a, M, K, K, 128, BK) || !make_tmap_u8(&tb, b, N, K, K, 128, BK) ||
      !make_tmap_f32(&tsa, sfa, ((M + 127) / 128) * KB, 128, 128, 1, 128) ||
      !make_tmap_f32(&tsb, sfb, ((N + 127) / 128) * KB, 128, 128, 1, 128))
    return FP8_ERR_CUDA;
  auto kern = gemm_mx_pair_kernel<ST>;
  if (!ensure_smem(kern, C::SMEM)) return FP8_ERR_CUDA;
  const int64_t ntiles = ((M + C::TM - 1) / C::TM) * ((N + C::TN - 1) / C::TN);
  const int64_t pairs = std::min<int64_t>(ntiles, device_sm_count() / 2);
  int64_t g = kRasterGroupBytes / (static_cast<int64_t>(C::TM) * K);  // raster groups of 256-row tiles
  g = std::max<int64_t>(1, std::min<int64_t>(g, (M + C::TM - 1) / C::TM));
  kern<<<static_cast<unsigned>(2 * pairs), C::THREADS, C::SMEM, stream>>>(
      ta, tb, tsa, tsb, out, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
      idesc_mxf8f6f4(a_fmt, b_fmt, 256, 256, 0, 0), dev_status, static_cast<int>(g), wait_ns);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t launch_gemm_mx(const uint8_t *a, const uint8_t *sfa, const uint8_t *b, const uint8_t *sfb, int a_fmt,
                            int b_fmt, uint16_t *out, int64_t M, int64_t N, int64_t K, int *dev_status,
                            cudaStream_t stream, uint64_t wait_ns, int mode) {
  if (mode == 2)
    return launch_gemm_mx_pairs(a, sfa, b, sfb, a_fmt, b_fmt, out, M, N, K, dev_status, stream, wait_ns);
  constexpr int BN = MX_BN, ST = MX_STAGES, NACC = MX_NACC;
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, a, M, K, K, BM, BK) || !make_tmap_u8(&tb, b, N, K, K, BN, BK)) return FP8_ERR_CUDA;
  const int ntiles = static_cast<int>(((M + 127) / 128) * ((N + BN - 1) / BN));
  auto run = [&](auto kind) -> fp8_status_t {
    constexpr int KIND = decltype(kind)::value;
    using C = AccCfg<KIND, BN, ST, NACC>;
    auto kern = gemm_tmem_kernel<KIND, BN, ST, NACC>;
    if (!ensure_smem(kern, C::SMEM)) return FP8_ERR_CUDA;
    kern<<<persistent_grid(ntiles), C::THREADS, C::SMEM, stream>>>(
        ta, tb, nullptr, 0, nullptr, 0, sfa, sfb, out, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
        idesc_mxf8f6f4(a_fmt, b_fmt, BM, BN, 0, 0), dev_status, raster_group(M, K), wait_ns);
    note_launches(1);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
  };
  // mode 3: the scales in the staged-four-times layout
  if (mode == 3) return run(std::integral_constant<int, KIND_MX8W>{});
  return run(std::integral_constant<int, KIND_MX8>{});
}

// NVFP4: a and b are packed E2M1 [M x K/2], [N x K/2] bytes (K % 256 == 0);
// sfa, sfb the E4M3 block scales in the tiled layout (K/16 groups per row); ta,
// tb the fp32 tensor scales (device memory).
fp8_status_t launch_gemm_nvfp4(const uint8_t *a, const uint8_t *sfa, const float *ta, const uint8_t *b,
                               const uint8_t *sfb, const float *tb, uint16_t *out, int64_t M, int64_t N, int64_t K,
                               int *dev_status, cudaStream_t stream) {
  constexpr int BN = 256, ST = 4, NACC = 1;
  using C = AccCfg<KIND_NVF4, BN, ST, NACC>;
  CUtensorMap tma, tmb;
  const int64_t kbytes = K / 2;
  if (!make_tmap_u8(&tma, a, M, kbytes, kbytes, BM, BK) || !make_tmap_u8(&tmb, b, N, kbytes, kbytes, BN, BK))
    return FP8_ERR_CUDA;
  auto kern = gemm_tmem_kernel<KIND_NVF4, BN, ST, NACC>;
  if (!ensure_smem(kern, C::SMEM)) return FP8_ERR_CUDA;
  const int ntiles = static_cast<int>(((M + 127) / 128) * ((N + BN - 1) / BN));
  kern<<<persistent_grid(ntiles), C::THREADS, C::SMEM, stream>>>(
      tma, tmb, ta, 0, tb, 0, sfa, sfb, out, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
      idesc_mxf4nvf4(BM, BN), dev_status, raster_group(M, kbytes), kWaitTimeoutNs);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t launch_wait_probe(int *dev_status, uint64_t timeout_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(dev_status, timeout_ns);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8bs

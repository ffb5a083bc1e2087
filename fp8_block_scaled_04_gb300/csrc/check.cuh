// check.cuh -- store bounds checks of the FP8BS_CHECK build (a stand-in for a
// memory checker). Every plain global store of the kernels is written as
//   if (FP8BS_GUARD(offset, count, extent)) p[offset] = v;
// with offset and count in elements of the stored array and extent the number
// of elements the buffer holds for this call's shape (the caller owns at least
// that much). In the normal build the guard is the constant true and compiles
// away. In the FP8BS_CHECK build a store outside [0, extent) is skipped and the
// first one is recorded as (source line << 40) | (offset & (2^40 - 1)) in this
// translation unit's record word, read and cleared on the host by
// fp8_debug_oob_read(). No trap: the kernel runs on and the context stays usable.
#pragma once

#include <stdint.h>

namespace fp8bs {

#ifdef FP8BS_CHECK
static __device__ unsigned long long g_oob_record;

__device__ __forceinline__ bool store_in_bounds(int64_t offset, int64_t count, int64_t extent, int line) {
  if (offset >= 0 && count >= 0 && offset + count <= extent) return true;
  const unsigned long long rec =
      (static_cast<unsigned long long>(line) << 40) | (static_cast<unsigned long long>(offset) & ((1ull << 40) - 1));
  atomicCAS(&g_oob_record, 0ull, rec == 0 ? 1ull : rec);
  return false;
}
#define FP8BS_GUARD(offset, count, extent)                                                             \
  ::fp8bs::store_in_bounds(static_cast<int64_t>(offset), static_cast<int64_t>(count), static_cast<int64_t>(extent), \
                           __LINE__)
#else
#define FP8BS_GUARD(offset, count, extent) true
#endif

}  // namespace fp8bs

// Host side, one definition per translation unit that includes this header
// (quantize.cu, nvfp4.cu, gemm.cu): read and clear the record word.
#ifdef FP8BS_CHECK
#define FP8BS_OOB_READER(name)                                                                     \
  uint64_t name() {                                                                                \
    unsigned long long v = 0, z = 0;                                                              \
    if (cudaMemcpyFromSymbol(&v, ::fp8bs::g_oob_record, sizeof(v)) != cudaSuccess) return ~0ull;    \
    cudaMemcpyToSymbol(::fp8bs::g_oob_record, &z, sizeof(z));                                     \
    return v;                                                                                      \
  }
#else
#define FP8BS_OOB_READER(name) \
  uint64_t name() { return 0; }
#endif

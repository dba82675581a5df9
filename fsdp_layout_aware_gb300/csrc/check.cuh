// Checked builds (compiled with TIDE_CHECKED): every global store of the
// kernels is first compared with the byte range of the item it belongs to; a
// store outside that range is skipped and counted.  The plan guarantees that
// the items tile the caller's buffers (checked on the host), so a clean count
// over a test run means no kernel wrote outside the buffers or into another
// item.  Each translation unit keeps its own counter (internal linkage) and
// exports it through TIDE_BOUNDS_COUNTER; tide_debug_bounds_violations adds
// them up.  In normal builds store_ok is `true` and costs nothing.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace tide {

#ifdef TIDE_CHECKED
static __device__ unsigned int g_bounds_violations;

__device__ __forceinline__ bool store_ok(const void* p, size_t bytes, const void* lo, const void* hi) {
  const uintptr_t a = (uintptr_t)p;
  if (a >= (uintptr_t)lo && a + bytes <= (uintptr_t)hi) return true;
  atomicAdd(&g_bounds_violations, 1u);
  return false;
}

// Host accessor of this translation unit's counter (reads, then optionally
// clears it).
#define TIDE_BOUNDS_COUNTER(name)                                                    \
  unsigned int name(bool reset) {                                                    \
    unsigned int v = 0;                                                              \
    cudaMemcpyFromSymbol(&v, g_bounds_violations, sizeof v);                         \
    if (reset) {                                                                     \
      const unsigned int z = 0;                                                      \
      cudaMemcpyToSymbol(g_bounds_violations, &z, sizeof z);                         \
    }                                                                                \
    return v;                                                                        \
  }
#else
__device__ __forceinline__ bool store_ok(const void*, size_t, const void*, const void*) { return true; }
#define TIDE_BOUNDS_COUNTER(name) \
  unsigned int name(bool) { return 0; }
#endif

}  // namespace tide

// Device helpers shared by the reduce-scatter kernels (rs_kernel.cu,
// rs_bulk.cu, rs_staged.cu): exact bf16 widening with fp32 round-to-nearest
// adds, block-wide zero fill, and 8-output stores as aligned 16-byte vectors.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "check.cuh"

namespace tide {

// Widen the 8 bf16 values of a 16-byte vector and add them into acc (fp32,
// round to nearest even).  bf16 -> fp32 is exact: the 16 bits become the high
// half of the fp32 pattern.
__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 v) {
  acc[0] = __fadd_rn(acc[0], __uint_as_float(v.x << 16));
  acc[1] = __fadd_rn(acc[1], __uint_as_float(v.x & 0xFFFF0000u));
  acc[2] = __fadd_rn(acc[2], __uint_as_float(v.y << 16));
  acc[3] = __fadd_rn(acc[3], __uint_as_float(v.y & 0xFFFF0000u));
  acc[4] = __fadd_rn(acc[4], __uint_as_float(v.z << 16));
  acc[5] = __fadd_rn(acc[5], __uint_as_float(v.z & 0xFFFF0000u));
  acc[6] = __fadd_rn(acc[6], __uint_as_float(v.w << 16));
  acc[7] = __fadd_rn(acc[7], __uint_as_float(v.w & 0xFFFF0000u));
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Next work item from the launch's shared counter.  Every CTA keeps taking
// items until it draws an index >= n_items, so a launch of G CTAs draws
// exactly n_items + G values; the CTA that draws the last one knows that no
// other draw follows and sets the counter back to zero, ready for the next
// launch that reads the same pointer table.
__device__ __forceinline__ long long take_item(unsigned long long* counter, int64_t n_items) {
  const unsigned long long v = atomicAdd(counter, 1ull);
  if (v == (unsigned long long)n_items + gridDim.x - 1) atomicExch(counter, 0ull);
  return (long long)v;
}

// Padding rows of a destination piece: +0.0 everywhere.
__device__ __forceinline__ void zero_fill(float* dst, int n) {
  const int head = min(n, (int)(((16 - ((uintptr_t)dst & 15)) & 15) >> 2));
  if ((int)threadIdx.x < head && store_ok(dst + threadIdx.x, 4, dst, dst + n)) dst[threadIdx.x] = 0.f;
  const int nv = (n - head) >> 2;
  float4* d4 = reinterpret_cast<float4*>(dst + head);
  for (int i = threadIdx.x; i < nv; i += blockDim.x)
    if (store_ok(d4 + i, 16, dst, dst + n)) __stcs(d4 + i, make_float4(0.f, 0.f, 0.f, 0.f));
  const int t0 = head + (nv << 2);
  if ((int)threadIdx.x < n - t0 && store_ok(dst + t0 + threadIdx.x, 4, dst, dst + n)) dst[t0 + threadIdx.x] = 0.f;
}

// Store the 8 results of a vector whose lane 0 is item element e0 when the
// destination of e0 is 16-byte aligned; lanes outside [0, n) are skipped.
__device__ __forceinline__ void store8_aligned(float* dst, int e0, int n, const float (&acc)[8]) {
  if (e0 >= 0 && e0 + 8 <= n) {
    float* o = dst + e0;
    if (store_ok(o, 16, dst, dst + n)) __stcs(reinterpret_cast<float4*>(o), make_float4(acc[0], acc[1], acc[2], acc[3]));
    if (store_ok(o + 4, 16, dst, dst + n))
      __stcs(reinterpret_cast<float4*>(o + 4), make_float4(acc[4], acc[5], acc[6], acc[7]));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + i;
      if (e >= 0 && e < n && store_ok(dst + e, 4, dst, dst + n)) __stcs(dst + e, acc[i]);
    }
  }
}

__device__ __forceinline__ void store4(float* dst, int a, int n, float w0, float w1, float w2, float w3) {
  if (a >= 0 && a + 4 <= n) {
    if (store_ok(dst + a, 16, dst, dst + n)) __stcs(reinterpret_cast<float4*>(dst + a), make_float4(w0, w1, w2, w3));
  } else {
    if (a >= 0 && a < n && store_ok(dst + a, 4, dst, dst + n)) __stcs(dst + a, w0);
    if (a + 1 >= 0 && a + 1 < n && store_ok(dst + a + 1, 4, dst, dst + n)) __stcs(dst + a + 1, w1);
    if (a + 2 >= 0 && a + 2 < n && store_ok(dst + a + 2, 4, dst, dst + n)) __stcs(dst + a + 2, w2);
    if (a + 3 >= 0 && a + 3 < n && store_ok(dst + a + 3, 4, dst, dst + n)) __stcs(dst + a + 3, w3);
  }
}

// Destination of e0 is delta = 1..3 elements short of a 16-byte boundary.
// Lane t writes the 16-byte aligned elements [e0+delta, e0+delta+8): its own
// results from delta on, then the first delta results of lane t+1, which hold
// the next 8 elements (one warp holds 256 consecutive elements).  Lane 31 has
// no such neighbour and writes only its own part; lane 0 also writes its
// first delta elements, which the previous warp's lane 31 cannot.  Together
// the lanes write every element once.  Called by all 32 lanes.
__device__ __forceinline__ void store8_shifted(float* dst, int e0, int n, int delta, int lane,
                                               const float (&acc)[8]) {
  const float n0 = __shfl_down_sync(0xffffffffu, acc[0], 1);
  const float n1 = __shfl_down_sync(0xffffffffu, acc[1], 1);
  const float n2 = __shfl_down_sync(0xffffffffu, acc[2], 1);
  float w[8];
  if (delta == 1) {
    w[0] = acc[1]; w[1] = acc[2]; w[2] = acc[3]; w[3] = acc[4];
    w[4] = acc[5]; w[5] = acc[6]; w[6] = acc[7]; w[7] = n0;
  } else if (delta == 2) {
    w[0] = acc[2]; w[1] = acc[3]; w[2] = acc[4]; w[3] = acc[5];
    w[4] = acc[6]; w[5] = acc[7]; w[6] = n0; w[7] = n1;
  } else {
    w[0] = acc[3]; w[1] = acc[4]; w[2] = acc[5]; w[3] = acc[6];
    w[4] = acc[7]; w[5] = n0; w[6] = n1; w[7] = n2;
  }
  const int a = e0 + delta;
  store4(dst, a, n, w[0], w[1], w[2], w[3]);   // always this lane's own results
  if (lane != 31) {
    store4(dst, a + 4, n, w[4], w[5], w[6], w[7]);
  } else {
#pragma unroll
    for (int i = 4; i < 8; ++i) {
      const int j = a + i;
      if (j < e0 + 8 && j >= 0 && j < n && store_ok(dst + j, 4, dst, dst + n)) __stcs(dst + j, w[i]);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int j = e0 + i;
      if (i < delta && j >= 0 && j < n && store_ok(dst + j, 4, dst, dst + n)) __stcs(dst + j, acc[i]);
    }
  }
}

// Result variants of the reduce-scatter (tide_plan_set_option): the sum is
// divided by N (fp32, correctly rounded) when averaging, then added to the
// shard's previous value when accumulating.
enum : int { EPI_AVERAGE = 1, EPI_ACCUMULATE = 2 };

__device__ __forceinline__ float epilogue1(float acc, const float* dst, int flags, int N) {
  if (flags & EPI_AVERAGE) acc = __fdiv_rn(acc, (float)N);
  if (flags & EPI_ACCUMULATE) acc = __fadd_rn(*dst, acc);
  return acc;
}

// Apply the variants to the 8 results of a vector whose lane 0 is element e0
// of dst (elements outside [0, n) are left alone).
__device__ __forceinline__ void epilogue8(float (&acc)[8], const float* dst, int e0, int n, int flags, int N) {
  if (!flags) return;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = e0 + i;
    if (e >= 0 && e < n) acc[i] = epilogue1(acc[i], dst + e, flags, N);
  }
}

// Padding rows: +0.0, or the previous value plus +0.0 when accumulating.
__device__ __forceinline__ void pad_fill(float* dst, int n, int flags, int tid, int nthreads) {
  if (!(flags & EPI_ACCUMULATE)) {
    const int head = min(n, (int)(((16 - ((uintptr_t)dst & 15)) & 15) >> 2));
    if (tid < head && store_ok(dst + tid, 4, dst, dst + n)) dst[tid] = 0.f;
    const int nv = (n - head) >> 2;
    float4* d4 = reinterpret_cast<float4*>(dst + head);
    for (int i = tid; i < nv; i += nthreads)
      if (store_ok(d4 + i, 16, dst, dst + n)) __stcs(d4 + i, make_float4(0.f, 0.f, 0.f, 0.f));
    const int t0 = head + (nv << 2);
    if (tid < n - t0 && store_ok(dst + t0 + tid, 4, dst, dst + n)) dst[t0 + tid] = 0.f;
  } else {
    for (int i = tid; i < n; i += nthreads)
      if (store_ok(dst + i, 4, dst, dst + n)) dst[i] = __fadd_rn(dst[i], 0.f);
  }
}

}  // namespace tide

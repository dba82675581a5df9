// TIDE-RS hot loop on one GPU: every emulated rank's bf16 gradients are read
// in place and reduced in fp32 straight into each destination rank's packed
// fp32 shard ("What shipped" in the TIDE news post; "Reduce-scatter: two
// levels of addition, the last one done by NVSwitch" in "The Endgame of FSDP
// Communication"; Figure 6 of the preprint).
//
// What the pages split across copy engines, summing CTAs, RDMA and an
// NVSwitch read-and-add is fused here into one pass over HBM, because every
// rank's gradients already sit in this GPU's memory: per output element, the
// N contributions are loaded once, summed per source node over l = 0..L-1
// (level 1, an fp32 node partial), and the M partials are added in the
// Latin-square landing order of that element's slice (level 2).  The order of
// the fp32 additions is exactly that one, so the result is bit-reproducible.
//
// Work decomposition: a persistent grid of CTAs walks the plan's item list
// round-robin; an item is one contiguous range (<= 8192 elements) of one
// (parameter, destination rank) piece inside one level-2 slice.  Each thread
// owns 8 consecutive outputs, so each contributor is read with one 16-byte
// load per thread and a warp reads 512 contiguous bytes of each contributor.

#include <cuda_runtime.h>

#include <cstdint>

#include "tide_internal.h"

namespace tide {
namespace {

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

// Padding rows of a destination piece: +0.0 everywhere.
__device__ __forceinline__ void zero_fill(float* dst, int n) {
  const int head = min(n, (int)(((16 - ((uintptr_t)dst & 15)) & 15) >> 2));
  if ((int)threadIdx.x < head) dst[threadIdx.x] = 0.f;
  const int nv = (n - head) >> 2;
  float4* d4 = reinterpret_cast<float4*>(dst + head);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) __stcs(d4 + i, make_float4(0.f, 0.f, 0.f, 0.f));
  const int t0 = head + (nv << 2);
  if ((int)threadIdx.x < n - t0) dst[t0 + threadIdx.x] = 0.f;
}

// Store the 8 results of a vector whose lane 0 is item element e0 when the
// destination of e0 is 16-byte aligned; lanes outside [0, n) are skipped.
__device__ __forceinline__ void store8_aligned(float* dst, int e0, int n, const float (&acc)[8]) {
  if (e0 >= 0 && e0 + 8 <= n) {
    float* o = dst + e0;
    __stcs(reinterpret_cast<float4*>(o), make_float4(acc[0], acc[1], acc[2], acc[3]));
    __stcs(reinterpret_cast<float4*>(o + 4), make_float4(acc[4], acc[5], acc[6], acc[7]));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + i;
      if (e >= 0 && e < n) __stcs(dst + e, acc[i]);
    }
  }
}

__device__ __forceinline__ void store4(float* dst, int a, int n, float w0, float w1, float w2, float w3) {
  if (a >= 0 && a + 4 <= n) {
    __stcs(reinterpret_cast<float4*>(dst + a), make_float4(w0, w1, w2, w3));
  } else {
    if (a >= 0 && a < n) __stcs(dst + a, w0);
    if (a + 1 >= 0 && a + 1 < n) __stcs(dst + a + 1, w1);
    if (a + 2 >= 0 && a + 2 < n) __stcs(dst + a + 2, w2);
    if (a + 3 >= 0 && a + 3 < n) __stcs(dst + a + 3, w3);
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
      if (j < e0 + 8 && j >= 0 && j < n) __stcs(dst + j, w[i]);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int j = e0 + i;
      if (i < delta && j >= 0 && j < n) __stcs(dst + j, acc[i]);
    }
  }
}

// All N contributors of the item's parameter share their address phase mod 16:
// every thread loads whole aligned 16-byte granules.  The first and last
// granules may extend past the item's range; they never leave the 16-byte
// granule of a valid element, so they stay inside mapped memory, and the
// extra lanes are never stored.
template <int L>
__device__ __forceinline__ void reduce_aligned(const uint16_t* const* src, const uint8_t* ord, int M, float* dst,
                                               int n) {
  const int ph = (int)(((uintptr_t)src[0] >> 1) & 7);
  const int nvec = (ph + n + 7) >> 3;
  // elements from a vector's first element to the next 16-byte boundary of dst
  const int delta = (int)(((unsigned)ph - (unsigned)((uintptr_t)dst >> 2)) & 3u);
  const int lane = threadIdx.x & 31;
  // The loop condition is uniform per warp (the warp's first vector), so all
  // 32 lanes reach the shuffles in store8_shifted.
  for (int v = threadIdx.x; v - lane < nvec; v += blockDim.x) {
    const int e0 = v * 8 - ph;
    float acc2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc2[i] = 0.f;
    if (v < nvec) {
      for (int k = 0; k < M; ++k) {
        const int node = ord[k];
        uint4 x[L];
#pragma unroll
        for (int l = 0; l < L; ++l) x[l] = __ldcs(reinterpret_cast<const uint4*>(src[node * L + l] + e0));
        float acc1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc1[i] = 0.f;
#pragma unroll
        for (int l = 0; l < L; ++l) add_bf16x8(acc1, x[l]);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc2[i] = __fadd_rn(acc2[i], acc1[i]);
      }
    }
    if (delta == 0)
      store8_aligned(dst, e0, n, acc2);
    else
      store8_shifted(dst, e0, n, delta, lane, acc2);
  }
}

// Contributors at different address phases: element-wise loads, same order.
template <int L>
__device__ __forceinline__ void reduce_unaligned(const uint16_t* const* src, const uint8_t* ord, int M, float* dst,
                                                 int n) {
  const int nvec = (n + 7) >> 3;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const int e0 = v * 8;
    const int cnt = min(8, n - e0);
    float acc2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc2[i] = 0.f;
    for (int k = 0; k < M; ++k) {
      const int node = ord[k];
      float acc1[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc1[i] = 0.f;
#pragma unroll
      for (int l = 0; l < L; ++l) {
        const uint16_t* s = src[node * L + l] + e0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < cnt) acc1[i] = __fadd_rn(acc1[i], bf16_to_f32(__ldcs(s + i)));
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) acc2[i] = __fadd_rn(acc2[i], acc1[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < cnt) __stcs(dst + e0 + i, acc2[i]);
  }
}

// CTAs take items in list order from a shared counter (one atomicAdd per
// item, issued one item ahead so its latency is hidden): the work balances
// whatever the items' sizes, and at any moment the CTAs are on neighbouring
// items, so the contributors are read in nearly address order across the GPU.
// Without a counter (noalloc entry point) CTA b takes items b, b+G, b+2G, ...
template <int L>
__global__ void __launch_bounds__(kRsThreads, 4) rs_fused_kernel(const __grid_constant__ RsArgs a) {
  __shared__ const uint16_t* src[kMaxN];
  __shared__ long long next_item[2];
  unsigned long long* counter = a.counter;
  if (threadIdx.x == 0)
    next_item[0] = counter ? (long long)atomicAdd(counter, 1ull) : (long long)blockIdx.x;
  __syncthreads();
  int slot = 0;
  for (int64_t it = next_item[0]; it < a.n_items; it = next_item[slot]) {
    slot ^= 1;
    if (threadIdx.x == 0)
      next_item[slot] = counter ? (long long)atomicAdd(counter, 1ull) : (long long)(it + gridDim.x);
    const RsItem item = a.items[it];
    float* dst = a.shard_tab[item.r] + item.dst_off;
    if (item.kind == RS_PAD) {
      zero_fill(dst, item.n);
    } else {
      if ((int)threadIdx.x < a.N)
        src[threadIdx.x] = a.grad_tab[(int64_t)item.p * a.N + threadIdx.x] + item.src_off;
      __syncthreads();
      const uint8_t* ord = a.order + ((item.r / L) * L + item.slice) * a.M;
      if (a.uniform_phase[item.p])
        reduce_aligned<L>(src, ord, a.M, dst, item.n);
      else
        reduce_unaligned<L>(src, ord, a.M, dst, item.n);
    }
    __syncthreads();  // next_item[slot] is visible; this item's readers of src[] are done
  }
}

template <int L>
int launch_rs_t(const RsArgs& a, int grid, cudaStream_t s) {
  rs_fused_kernel<L><<<grid, kRsThreads, 0, s>>>(a);
  return (int)cudaGetLastError();
}

template <int L>
int occupancy_t() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rs_fused_kernel<L>, kRsThreads, 0) != cudaSuccess) return 0;
  return n;
}

}  // namespace

int launch_rs(const RsArgs& a, int grid, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  switch (a.L) {
    case 1: return launch_rs_t<1>(a, grid, s);
    case 2: return launch_rs_t<2>(a, grid, s);
    case 3: return launch_rs_t<3>(a, grid, s);
    case 4: return launch_rs_t<4>(a, grid, s);
    case 5: return launch_rs_t<5>(a, grid, s);
    case 6: return launch_rs_t<6>(a, grid, s);
    case 7: return launch_rs_t<7>(a, grid, s);
    case 8: return launch_rs_t<8>(a, grid, s);
  }
  return (int)cudaErrorInvalidValue;
}

int rs_blocks_per_sm(int L) {
  switch (L) {
    case 1: return occupancy_t<1>();
    case 2: return occupancy_t<2>();
    case 3: return occupancy_t<3>();
    case 4: return occupancy_t<4>();
    case 5: return occupancy_t<5>();
    case 6: return occupancy_t<6>();
    case 7: return occupancy_t<7>();
    case 8: return occupancy_t<8>();
  }
  return 0;
}

}  // namespace tide

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

#include "rs_device.cuh"
#include "tide_internal.h"

namespace tide {
namespace {

// All N contributors of the item's parameter share their address phase mod 16:
// every thread loads whole aligned 16-byte granules.  The first and last
// granules may extend past the item's range; they never leave the 16-byte
// granule of a valid element, so they stay inside mapped memory, and the
// extra lanes are never stored.
// tid / nthr: this thread's index among the nthr threads (a whole CTA, or one
// warp) sharing the item.
template <int L, bool kBatched>
__device__ __forceinline__ void reduce_aligned(const uint16_t* const* src, int M, float* dst, int n, int epi, int N,
                                               int tid, int nthr) {
  const int ph = (int)(((uintptr_t)src[0] >> 1) & 7);
  const int nvec = (ph + n + 7) >> 3;
  // elements from a vector's first element to the next 16-byte boundary of dst
  const int delta = (int)(((unsigned)ph - (unsigned)((uintptr_t)dst >> 2)) & 3u);
  const int lane = threadIdx.x & 31;
  // The loop condition is uniform per warp (the warp's first vector), so all
  // 32 lanes reach the shuffles in store8_shifted.
  for (int v = tid; v - lane < nvec; v += nthr) {
    const int e0 = v * 8 - ph;
    float acc2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc2[i] = 0.f;
    if (v < nvec) {
      // With M <= L there is one batch and acc2 is its sum (+0.0 + b == b:
      // a sum started at +0.0 is never -0.0), so only M > L keeps a batch sum.
      float bsum[kBatched ? 8 : 1];
#pragma unroll
      for (int i = 0; i < (kBatched ? 8 : 1); ++i) bsum[i] = 0.f;
      for (int k = 0; k < M; ++k) {
        uint4 x[L];
#pragma unroll
        for (int l = 0; l < L; ++l) x[l] = __ldcs(reinterpret_cast<const uint4*>(src[k * L + l] + e0));
        float acc1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc1[i] = 0.f;
#pragma unroll
        for (int l = 0; l < L; ++l) add_bf16x8(acc1, x[l]);
        if constexpr (kBatched) {
#pragma unroll
          for (int i = 0; i < 8; ++i) bsum[i] = __fadd_rn(bsum[i], acc1[i]);
          if ((k + 1) % L == 0 || k + 1 == M) {  // end of a batch of L sources
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              acc2[i] = __fadd_rn(acc2[i], bsum[i]);
              bsum[i] = 0.f;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc2[i] = __fadd_rn(acc2[i], acc1[i]);
        }
      }
    }
    epilogue8(acc2, dst, e0, n, epi, N);
    if (delta == 0)
      store8_aligned(dst, e0, n, acc2);
    else
      store8_shifted(dst, e0, n, delta, lane, acc2);
  }
}

// Contributors at different address phases: element-wise loads, same order.
template <int L, bool kBatched>
__device__ __forceinline__ void reduce_unaligned(const uint16_t* const* src, int M, float* dst, int n, int epi, int N,
                                                 int tid, int nthr) {
  const int nvec = (n + 7) >> 3;
  for (int v = tid; v < nvec; v += nthr) {
    const int e0 = v * 8;
    const int cnt = min(8, n - e0);
    float acc2[8], bsum[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc2[i] = bsum[i] = 0.f;
    for (int k = 0; k < M; ++k) {
      float acc1[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc1[i] = 0.f;
#pragma unroll
      for (int l = 0; l < L; ++l) {
        const uint16_t* s = src[k * L + l] + e0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < cnt) acc1[i] = __fadd_rn(acc1[i], bf16_to_f32(__ldcs(s + i)));
      }
      if constexpr (kBatched) {
#pragma unroll
        for (int i = 0; i < 8; ++i) bsum[i] = __fadd_rn(bsum[i], acc1[i]);
        if ((k + 1) % L == 0 || k + 1 == M) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            acc2[i] = __fadd_rn(acc2[i], bsum[i]);
            bsum[i] = 0.f;
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc2[i] = __fadd_rn(acc2[i], acc1[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < cnt) __stcs(dst + e0 + i, epilogue1(acc2[i], dst + e0 + i, epi, N));
  }
}

// src[k * L + l] = contributor l of the k-th node in the item's level-2 order,
// written by the nthr threads sharing the item.
template <int L>
__device__ __forceinline__ void fill_sources(const RsArgs& a, const RsItem& item, const uint16_t** src, int tid,
                                             int nthr) {
  const uint8_t* ord = a.order + ((item.r / L) * L + item.slice) * a.M;
  for (int t = tid; t < a.N; t += nthr) {
    const int node = ord[t / L];
    src[t] = a.grad_tab[(int64_t)item.p * a.N + node * L + t % L] + item.src_off;
  }
}

template <int L, bool kBatched>
__device__ __forceinline__ void run_item(const RsArgs& a, const RsItem& item, const uint16_t* const* src, int tid,
                                         int nthr) {
  float* dst = a.shard_tab[item.r] + item.dst_off;
  if (a.uniform_phase[item.p])
    reduce_aligned<L, kBatched>(src, a.M, dst, item.n, a.epilogue, a.N, tid, nthr);
  else
    reduce_unaligned<L, kBatched>(src, a.M, dst, item.n, a.epilogue, a.N, tid, nthr);
}

// CTAs take work units in list order from a shared counter (one atomicAdd per
// unit, issued one unit ahead so its latency is hidden): the work balances
// whatever the items' sizes, and at any moment the CTAs are on neighbouring
// items, so the contributors are read in nearly address order across the GPU.
// A unit is one item, reduced by the whole CTA, or a run of up to eight small
// items, one per warp.  Without a counter (noalloc entry point) CTA b takes
// units b, b+G, b+2G, ...
template <int L, bool kBatched>
__global__ void __launch_bounds__(kRsThreads, 4) rs_fused_kernel(const __grid_constant__ RsArgs a) {
  __shared__ const uint16_t* src[kRsBundle][kMaxN];  // one pointer table per warp; the CTA uses [0]
  __shared__ long long next_unit[2];
  unsigned long long* counter = a.counter;
  const int64_t n_units = a.units ? a.n_units : a.n_items;
  if (threadIdx.x == 0) next_unit[0] = counter ? take_item(counter, n_units) : (long long)blockIdx.x;
  __syncthreads();
  int slot = 0;
  for (int64_t u = next_unit[0]; u < n_units; u = next_unit[slot]) {
    slot ^= 1;
    if (threadIdx.x == 0) next_unit[slot] = counter ? take_item(counter, n_units) : (long long)(u + gridDim.x);
    const int64_t lo = a.units ? a.units[u] : u;
    const int64_t hi = a.units ? a.units[u + 1] : u + 1;
    if (hi - lo == 1) {
      const RsItem item = a.items[lo];
      if (item.kind == RS_PAD) {
        pad_fill(a.shard_tab[item.r] + item.dst_off, item.n, a.epilogue, threadIdx.x, blockDim.x);
      } else {
        fill_sources<L>(a, item, src[0], threadIdx.x, blockDim.x);
        __syncthreads();
        run_item<L, kBatched>(a, item, src[0], threadIdx.x, blockDim.x);
      }
    } else {
      const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
      if (lo + w < hi) {
        const RsItem item = a.items[lo + w];
        if (item.kind == RS_PAD) {
          pad_fill(a.shard_tab[item.r] + item.dst_off, item.n, a.epilogue, lane, 32);
        } else {
          fill_sources<L>(a, item, src[w], lane, 32);
          __syncwarp();
          run_item<L, kBatched>(a, item, src[w], lane, 32);
        }
      }
    }
    __syncthreads();  // next_unit[slot] is visible; this unit's readers of src[] are done
  }
}

// M > L (sources in batches) takes its own instantiation, so the usual
// M <= L kernel keeps its registers for loads in flight.
template <int L>
int launch_rs_t(const RsArgs& a, int grid, cudaStream_t s) {
  if (a.M > L)
    rs_fused_kernel<L, true><<<grid, kRsThreads, 0, s>>>(a);
  else
    rs_fused_kernel<L, false><<<grid, kRsThreads, 0, s>>>(a);
  return (int)cudaGetLastError();
}

template <int L>
int occupancy_t() {
  int n = 0, nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rs_fused_kernel<L, false>, kRsThreads, 0) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, rs_fused_kernel<L, true>, kRsThreads, 0) != cudaSuccess)
    return 0;
  return n < nb ? n : nb;
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

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
// from a shared counter; an item is one contiguous range (2048-8192 elements,
// fewer the more ranks read it) of one (parameter, destination rank) piece
// inside one level-2 slice.  Each thread
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
template <int L, bool kBatched>
__device__ __forceinline__ void reduce_aligned(const uint16_t* const* src, int M, float* dst, int n, int epi, int N) {
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
__device__ __forceinline__ void reduce_unaligned(const uint16_t* const* src, int M, float* dst, int n, int epi,
                                                 int N) {
  const int nvec = (n + 7) >> 3;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
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
      if (i < cnt && store_ok(dst + e0 + i, 4, dst, dst + n))
        __stcs(dst + e0 + i, epilogue1(acc2[i], dst + e0 + i, epi, N));
  }
}

// CTAs take items in list order from a shared counter (one atomicAdd per
// item, issued one item ahead so its latency is hidden): the work balances
// whatever the items' sizes, and at any moment the CTAs are on neighbouring
// items, so the contributors are read in nearly address order across the GPU.
template <int L, bool kBatched>
__global__ void __launch_bounds__(kRsThreads, 4) rs_fused_kernel(const __grid_constant__ RsArgs a) {
  __shared__ const uint16_t* src[kMaxN];
  __shared__ long long next_item[2];
  if (threadIdx.x == 0) next_item[0] = take_item(a.counter, a.n_items);
  __syncthreads();
  int slot = 0;
  for (int64_t it = next_item[0]; it < a.n_items; it = next_item[slot]) {
    slot ^= 1;
    if (threadIdx.x == 0) next_item[slot] = take_item(a.counter, a.n_items);
    const RsItem item = a.items[it];
    float* dst = a.shard_tab[item.r] + item.dst_off;
    if (item.kind == RS_PAD) {
      pad_fill(dst, item.n, a.epilogue, threadIdx.x, blockDim.x);
    } else {
      // src[k * L + l]: contributor l of the k-th node in level-2 order
      if ((int)threadIdx.x < a.N) {
        const int k = (int)threadIdx.x / L, l = (int)threadIdx.x % L;
        const int node = a.order[((item.r / L) * L + item.slice) * a.M + k];
        src[threadIdx.x] = a.grad_tab[(int64_t)item.p * a.N + node * L + l] + item.src_off;
      }
      __syncthreads();
      if (a.uniform_phase[item.p])
        reduce_aligned<L, kBatched>(src, a.M, dst, item.n, a.epilogue, a.N);
      else
        reduce_unaligned<L, kBatched>(src, a.M, dst, item.n, a.epilogue, a.N);
    }
    __syncthreads();  // next_item[slot] is visible; this item's readers of src[] are done
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

TIDE_BOUNDS_COUNTER(rs_kernel_bounds)

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

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

// Store the 8 results of a vector whose lane 0 is item element e0; lanes
// outside [0, n) are skipped.  dmis is the address phase (bytes mod 16) of
// lane 0's output, the same for every vector of an item.
__device__ __forceinline__ void store8(float* dst, int e0, int n, int dmis, const float (&acc)[8]) {
  if (e0 >= 0 && e0 + 8 <= n) {
    float* o = dst + e0;
    if (dmis == 0) {
      __stcs(reinterpret_cast<float4*>(o), make_float4(acc[0], acc[1], acc[2], acc[3]));
      __stcs(reinterpret_cast<float4*>(o + 4), make_float4(acc[4], acc[5], acc[6], acc[7]));
    } else if (dmis == 8) {
#pragma unroll
      for (int j = 0; j < 4; ++j) __stcs(reinterpret_cast<float2*>(o + 2 * j), make_float2(acc[2 * j], acc[2 * j + 1]));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) __stcs(o + i, acc[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + i;
      if (e >= 0 && e < n) __stcs(dst + e, acc[i]);
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
  const int dmis = (int)(((uintptr_t)dst - 4u * (unsigned)ph) & 15);
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const int e0 = v * 8 - ph;
    float acc2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc2[i] = 0.f;
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
    store8(dst, e0, n, dmis, acc2);
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

template <int L>
__global__ void __launch_bounds__(kRsThreads) rs_fused_kernel(const __grid_constant__ RsArgs a) {
  __shared__ const uint16_t* src[kMaxN];
  for (int64_t it = blockIdx.x; it < a.n_items; it += gridDim.x) {
    const RsItem item = a.items[it];
    float* dst = a.shard_tab[item.r] + item.dst_off;
    if (item.kind == RS_PAD) {
      zero_fill(dst, item.n);
      continue;
    }
    __syncthreads();  // the previous item's readers of src[] are done
    if ((int)threadIdx.x < a.N)
      src[threadIdx.x] = a.grad_tab[(int64_t)item.p * a.N + threadIdx.x] + item.src_off;
    __syncthreads();
    const uint8_t* ord = a.order + ((item.r / L) * L + item.slice) * a.M;
    if (a.uniform_phase[item.p])
      reduce_aligned<L>(src, ord, a.M, dst, item.n);
    else
      reduce_unaligned<L>(src, ord, a.M, dst, item.n);
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

// TIDE-RS in the pages' two stages, emulated on one GPU ("Reduce-scatter:
// two levels of addition, the last one done by NVSwitch" in "The Endgame of
// FSDP Communication"; Figure 6 of the preprint).
//
// Stage 1, the summing CTAs: for every destination rank r (node n_d, local
// GPU l_d) and every source node n_s, the fp32 partial of n_s's L local bf16
// copies (l ascending) is written to the inbox slot it lands in.  On the
// pages the GPU of n_s that owns slice s sends its partial over its own line,
// so it arrives on destination GPU g = (s - c) mod L with c = (n_d - n_s)
// mod M; the emulated inbox is laid out [n_d][g][c][L * B] floats, rank
// l_d's block of the slice at l_d * B (B = ceil(S / L)).
//
// Stage 2, the landing CTAs (the NVSwitch read-and-add plus the CTAs that
// accumulate into the shard): every destination element adds the partials of
// its slice in the plan's level-2 order (by default landing GPUs g = 0..L-1
// in turn), batch by batch when M > L, and stores the sum.
//
// The additions happen in the same order as in rs_fused, so the shards are
// bit-identical; the price is 8*M extra bytes per shard element (every
// partial written once and read once).  CTA counts can be set per emulated
// rank to reproduce the pages' budget (16 summing, 4 landing CTAs per GPU).

#include <cuda_runtime.h>

#include <cstdint>

#include "rs_device.cuh"
#include "tide_internal.h"

namespace tide {
namespace {

__device__ __forceinline__ float* inbox_block(const RsArgs& a, int n_dest, int l_dest, int n_src, int slice,
                                             int64_t dst_off) {
  const int M = a.M, L = a.L;
  const int c = ((n_dest - n_src) % M + M) % M;
  const int g = ((slice - c) % L + L) % L;
  const int64_t slot = (int64_t)L * a.slice_len;
  return a.inbox + ((int64_t)(n_dest * L + g) * M + c) * slot + (int64_t)l_dest * a.slice_len +
         (dst_off - (int64_t)slice * a.slice_len);
}

// Stage 1 for one item whose contributors share their address phase mod 16.
template <int L>
__device__ __forceinline__ void sum_aligned(const RsArgs& a, const uint16_t* const* src, const RsItem& item) {
  const int ph = (int)(((uintptr_t)src[0] >> 1) & 7);
  const int n = item.n;
  const int nvec = (ph + n + 7) >> 3;
  const int lane = threadIdx.x & 31;
  const int n_dest = item.r / L, l_dest = item.r % L;
  for (int v = threadIdx.x; v - lane < nvec; v += blockDim.x) {
    const int e0 = v * 8 - ph;
    for (int n_src = 0; n_src < a.M; ++n_src) {
      float acc1[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc1[i] = 0.f;
      if (v < nvec) {
        uint4 x[L];
#pragma unroll
        for (int l = 0; l < L; ++l) x[l] = __ldcs(reinterpret_cast<const uint4*>(src[n_src * L + l] + e0));
#pragma unroll
        for (int l = 0; l < L; ++l) add_bf16x8(acc1, x[l]);
      }
      float* dst = inbox_block(a, n_dest, l_dest, n_src, item.slice, item.dst_off);
      const int delta = (int)(((unsigned)ph - (unsigned)((uintptr_t)dst >> 2)) & 3u);
      if (delta == 0)
        store8_aligned(dst, e0, n, acc1);
      else
        store8_shifted(dst, e0, n, delta, lane, acc1);
    }
  }
}

// The same with two vectors per thread per round (v and v + blockDim.x), both
// vectors' loads issued before either is added: for summing grids too small
// to fill the GPU (the pages' 16 summing CTAs per GPU), where the bytes each
// thread keeps in flight set the speed.  The stores, and so the partials,
// are those of sum_aligned.  128 registers, 2 CTAs per SM; used when the
// summing grid is below the full one and fits one wave at that residency.
// Against sum_aligned on one box, alternating (whole staged reduce-scatter
// with 16 + 4 CTAs): llama70b 9.71 vs 10.27 ms, qwen3moe 6.28 vs 6.49.
template <int L>
__device__ __forceinline__ void sum_aligned_wide(const RsArgs& a, const uint16_t* const* src, const RsItem& item) {
  const int ph = (int)(((uintptr_t)src[0] >> 1) & 7);
  const int n = item.n;
  const int nvec = (ph + n + 7) >> 3;
  const int lane = threadIdx.x & 31;
  const int n_dest = item.r / L, l_dest = item.r % L;
  for (int v = threadIdx.x; v - lane < nvec; v += 2 * blockDim.x) {
    const int v2 = v + blockDim.x;
    const int e0 = v * 8 - ph, e1 = v2 * 8 - ph;
    const bool second = v2 - lane < nvec;  // uniform per warp, like the loop condition
    for (int n_src = 0; n_src < a.M; ++n_src) {
      float acc1[8], acc2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc1[i] = acc2[i] = 0.f;
      uint4 x[L], y[L];
#pragma unroll
      for (int l = 0; l < L; ++l) {
        x[l] = v < nvec ? __ldcs(reinterpret_cast<const uint4*>(src[n_src * L + l] + e0)) : make_uint4(0, 0, 0, 0);
        y[l] = v2 < nvec ? __ldcs(reinterpret_cast<const uint4*>(src[n_src * L + l] + e1)) : make_uint4(0, 0, 0, 0);
      }
      if (v < nvec) {
#pragma unroll
        for (int l = 0; l < L; ++l) add_bf16x8(acc1, x[l]);
      }
      if (v2 < nvec) {
#pragma unroll
        for (int l = 0; l < L; ++l) add_bf16x8(acc2, y[l]);
      }
      float* dst = inbox_block(a, n_dest, l_dest, n_src, item.slice, item.dst_off);
      const int delta = (int)(((unsigned)ph - (unsigned)((uintptr_t)dst >> 2)) & 3u);
      if (delta == 0) {
        store8_aligned(dst, e0, n, acc1);
        if (second) store8_aligned(dst, e1, n, acc2);
      } else {
        store8_shifted(dst, e0, n, delta, lane, acc1);
        if (second) store8_shifted(dst, e1, n, delta, lane, acc2);
      }
    }
  }
}

// Stage 1 for contributors at different address phases: element-wise loads.
template <int L>
__device__ __forceinline__ void sum_unaligned(const RsArgs& a, const uint16_t* const* src, const RsItem& item) {
  const int n = item.n;
  const int n_dest = item.r / L, l_dest = item.r % L;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    for (int n_src = 0; n_src < a.M; ++n_src) {
      float acc1 = 0.f;
#pragma unroll
      for (int l = 0; l < L; ++l) acc1 = __fadd_rn(acc1, bf16_to_f32(__ldcs(src[n_src * L + l] + e)));
      float* blk = inbox_block(a, n_dest, l_dest, n_src, item.slice, item.dst_off);
      if (store_ok(blk + e, 4, blk, blk + n)) __stcs(blk + e, acc1);
    }
  }
}

template <int L, bool kWide>
__global__ void __launch_bounds__(kRsThreads, kWide ? 2 : 4) rs_sum_kernel(const __grid_constant__ RsArgs a) {
  __shared__ const uint16_t* src[kMaxN];
  __shared__ long long next_item[2];
  if (threadIdx.x == 0) next_item[0] = take_item(a.counter, a.n_items);
  __syncthreads();
  int slot = 0;
  for (int64_t it = next_item[0]; it < a.n_items; it = next_item[slot]) {
    slot ^= 1;
    if (threadIdx.x == 0) next_item[slot] = take_item(a.counter, a.n_items);
    const RsItem item = a.items[it];
    if (item.kind == RS_PAD) {
      // padding rows: every source's partial is +0.0
      for (int n_src = 0; n_src < a.M; ++n_src)
        zero_fill(inbox_block(a, item.r / L, item.r % L, n_src, item.slice, item.dst_off), item.n);
    } else {
      if ((int)threadIdx.x < a.N)
        src[threadIdx.x] = a.grad_tab[(int64_t)item.p * a.N + threadIdx.x] + item.src_off;
      __syncthreads();
      if (!a.uniform_phase[item.p])
        sum_unaligned<L>(a, src, item);
      else if constexpr (kWide)
        sum_aligned_wide<L>(a, src, item);
      else
        sum_aligned<L>(a, src, item);
    }
    __syncthreads();
  }
}

// Stage 2.  blockIdx.y is the destination rank.  For each slice, the first
// M threads list where the slice's partials landed, in the plan's level-2
// order, in shared memory.
__device__ __forceinline__ void list_partials(const RsArgs& a, const float** part, int n_dest, int l_dest, int s,
                                              int64_t lo) {
  const int M = a.M, L = a.L;
  if ((int)threadIdx.x < M) {
    const int k = threadIdx.x;
    const int node = a.order[(n_dest * L + s) * M + k];
    const int c = ((n_dest - node) % M + M) % M;  // relative index of the k-th source
    const int g = ((s - c) % L + L) % L;            // the GPU its slice s landed on
    part[k] = a.inbox + ((int64_t)(n_dest * L + g) * M + c) * (int64_t)L * a.slice_len +
              (int64_t)l_dest * a.slice_len - lo;
  }
}

// The threads then stream the slice, four outputs each per round, adding the
// partials in that order.  Keeping the list in shared memory keeps the kernel
// at 32 registers, so eight CTAs fit per SM (five when M > L, where the batch
// sums take 48 registers).  Used for M = 1 and M > L.
template <bool kBatched>
__global__ void __launch_bounds__(256, kBatched ? 5 : 8) rs_land_kernel(const __grid_constant__ RsArgs a) {
  __shared__ const float* part[kMaxM];
  const int M = a.M, L = a.L;
  const int64_t S = a.S, B = a.slice_len;
  const int r = blockIdx.y;
  const int n_dest = r / L, l_dest = r % L;
  float* out = a.shard_tab[r];
  const int64_t step = (int64_t)gridDim.x * blockDim.x * 4;
  for (int s = 0; s < L; ++s) {
    const int64_t lo = (int64_t)s * B, hi = min(S, lo + B);
    if (lo >= hi) break;
    __syncthreads();  // the previous slice's readers of part[] are done
    list_partials(a, part, n_dest, l_dest, s, lo);
    __syncthreads();
    const int np = M;
    for (int64_t x0 = lo + (int64_t)blockIdx.x * blockDim.x * 4 + threadIdx.x; x0 < hi; x0 += step) {
      // With M <= L there is one batch and acc is its sum directly.
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, bsum[kBatched ? 4 : 1] = {0.f};
      for (int j = 0; j < np; ++j) {
        const float* pj = part[j];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t x = x0 + (int64_t)u * blockDim.x;
          if (x < hi) {
            if constexpr (kBatched)
              bsum[u] = __fadd_rn(bsum[u], __ldcs(pj + x));
            else
              acc[u] = __fadd_rn(acc[u], __ldcs(pj + x));
          }
        }
        if constexpr (kBatched) {
          if ((j + 1) % L == 0 || j + 1 == np) {  // end of a batch
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              acc[u] = __fadd_rn(acc[u], bsum[u]);
              bsum[u] = 0.f;
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t x = x0 + (int64_t)u * blockDim.x;
        if (x < hi && store_ok(out + x, 4, out + lo, out + hi))
          __stcs(out + x, epilogue1(acc[u], out + x, a.epilogue, M * L));
      }
    }
  }
}

// The same for 2 <= M <= L, with the partials loaded kGroup at a time into
// registers before any of them is added: with kGroup = 2 a thread has eight
// loads in flight instead of waiting for one partial's loads before issuing
// the next one's.  The additions still run partial by partial in the plan's
// order.  Still 32 registers and eight CTAs per SM.  Measured against the
// one-partial-at-a-time loop on one box, alternating (whole staged
// reduce-scatter, filling the GPU / with the pages' 16 + 4 CTAs): qwen3moe
// (M = 2) 4.591 vs 4.672 ms / 12.29 vs 16.84 ms; wan22dit (M = 8) 9.871 vs
// 9.924 / 11.89 vs 14.35 ms; uneven (M = 6) 2.324 vs 2.323 / 3.10 vs 3.53 ms.
// With M = 1 or M > L it was slower, so those keep rs_land_kernel.  (Written as a template over the
// batching flag and group size: the same loop as a plain kernel measured
// slower.)
template <bool kBatched, int kGroup>
__global__ void __launch_bounds__(256, kBatched ? 5 : 8) rs_land_grouped_kernel(const __grid_constant__ RsArgs a) {
  __shared__ const float* part[kMaxM];
  const int M = a.M, L = a.L;
  const int64_t S = a.S, B = a.slice_len;
  const int r = blockIdx.y;
  const int n_dest = r / L, l_dest = r % L;
  float* out = a.shard_tab[r];
  const int64_t slot = (int64_t)L * B;
  const int64_t step = (int64_t)gridDim.x * blockDim.x * 4;
  for (int s = 0; s < L; ++s) {
    const int64_t lo = (int64_t)s * B, hi = min(S, lo + B);
    if (lo >= hi) break;
    __syncthreads();  // the previous slice's readers of part[] are done
    if ((int)threadIdx.x < M) {
      const int k = threadIdx.x;
      const int node = a.order[(n_dest * L + s) * M + k];
      const int c = ((n_dest - node) % M + M) % M;  // relative index of the k-th source
      const int g = ((s - c) % L + L) % L;            // the GPU its slice s landed on
      part[k] = a.inbox + ((int64_t)(n_dest * L + g) * M + c) * slot + (int64_t)l_dest * B - lo;
    }
    __syncthreads();
    for (int64_t x0 = lo + (int64_t)blockIdx.x * blockDim.x * 4 + threadIdx.x; x0 < hi; x0 += step) {
      // With M <= L there is one batch and acc is its sum directly.
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, bsum[kBatched ? 4 : 1] = {0.f};
      for (int j0 = 0; j0 < M; j0 += kGroup) {
        float v[kGroup][4];
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          const float* pj = part[min(j0 + q, M - 1)];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int64_t x = x0 + (int64_t)u * blockDim.x;
            v[q][u] = (j0 + q < M && x < hi) ? __ldcs(pj + x) : 0.f;
          }
        }
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          const int j = j0 + q;
          if (j >= M) break;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if constexpr (kBatched)
              bsum[u] = __fadd_rn(bsum[u], v[q][u]);
            else
              acc[u] = __fadd_rn(acc[u], v[q][u]);
          }
          if constexpr (kBatched) {
            if ((j + 1) % L == 0 || j + 1 == M) {  // end of a batch
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                acc[u] = __fadd_rn(acc[u], bsum[u]);
                bsum[u] = 0.f;
              }
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t x = x0 + (int64_t)u * blockDim.x;
        if (x < hi && store_ok(out + x, 4, out + lo, out + hi))
          __stcs(out + x, epilogue1(acc[u], out + x, a.epilogue, M * L));
      }
    }
  }
}

__device__ __forceinline__ void add_v(float4& a, const float4 b) {
  a.x = __fadd_rn(a.x, b.x);
  a.y = __fadd_rn(a.y, b.y);
  a.z = __fadd_rn(a.z, b.z);
  a.w = __fadd_rn(a.w, b.w);
}
__device__ __forceinline__ void add_v(float2& a, const float2 b) {
  a.x = __fadd_rn(a.x, b.x);
  a.y = __fadd_rn(a.y, b.y);
}
__device__ __forceinline__ void set_zero(float4& z) { z = make_float4(0.f, 0.f, 0.f, 0.f); }
__device__ __forceinline__ void set_zero(float2& z) { z = make_float2(0.f, 0.f); }
// the variants applied to each component (d: the vector's first element)
__device__ __forceinline__ float4 epilogue_v(float4 v, const float* d, int flags, int N) {
  return make_float4(epilogue1(v.x, d, flags, N), epilogue1(v.y, d + 1, flags, N), epilogue1(v.z, d + 2, flags, N),
                     epilogue1(v.w, d + 3, flags, N));
}
__device__ __forceinline__ float2 epilogue_v(float2 v, const float* d, int flags, int N) {
  return make_float2(epilogue1(v.x, d, flags, N), epilogue1(v.y, d + 1, flags, N));
}

// The landing kernels again, with vector loads and stores of V (float4 or
// float2), for plans whose slice length B is a multiple of the vector's
// width W (4: llama70b, qwen3moe, uneven and wan22dit as 16 x 4; 2: wan22dit
// as 8 x 8) when the inbox and every shard start on a 4*W-byte boundary:
// then slice s starts at element s*B of a shard and at a multiple of B in the
// inbox, so every partial of the slice and the shard share one vector phase.
// Each thread takes kVecs vectors per round (kVecs * kGroup vector loads in
// flight); the last W - 1 or fewer elements of a slice, past its whole
// vectors, are added element by element.  The additions are the scalar
// kernels', component by component, in the same order.  Measured (float4)
// against the 4-byte kernels on one box, alternating (whole staged
// reduce-scatter, filling the GPU / with the pages' 16 + 4 CTAs): llama70b
// 3.374 vs 3.464 ms / 15.70 vs 25.74 ms, qwen3moe 4.581 vs 4.590 / 10.21 vs
// 12.28, uneven 2.284 vs 2.324 / 2.77 vs 3.09, wan22dit as 16 x 4 13.26 vs
// 13.54 / 15.93 vs 16.69; float2 on wan22dit 9.646 vs 9.770 / 10.95 vs
// 11.94.  The M = 1 and float2 instances take 40 registers (6 CTAs per SM);
// at 32 they spilled.
//
// kVecs = 8 is the instance for landing grids too small to fill the GPU (the
// pages' 4 landing CTAs per GPU): with at most a CTA or two per SM, the bytes
// each thread keeps in flight set the speed, and registers are plentiful.
// Against kVecs = 2 on one box, alternating (whole staged reduce-scatter with
// 16 + 4 CTAs): llama70b 10.28 vs 15.69 ms, qwen3moe 6.49 vs 10.21, wan22dit
// 9.86 vs 10.94, uneven 2.49 vs 2.77.
template <bool kBatched, int kGroup, class V, int kVecs>
__global__ void __launch_bounds__(256, kVecs > 2 ? 1 : (kBatched ? 5 : ((kGroup == 1 || sizeof(V) == 8) ? 6 : 8)))
    rs_land_vec_kernel(const __grid_constant__ RsArgs a) {
  constexpr int W = (int)(sizeof(V) / 4);
  __shared__ const float* part[kMaxM];
  const int M = a.M, L = a.L;
  const int64_t S = a.S, B = a.slice_len;
  const int r = blockIdx.y;
  const int n_dest = r / L, l_dest = r % L;
  float* out = a.shard_tab[r];
  const int64_t slot = (int64_t)L * B;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  V zv;
  set_zero(zv);
  for (int s = 0; s < L; ++s) {
    const int64_t lo = (int64_t)s * B, hi = min(S, lo + B);
    if (lo >= hi) break;
    __syncthreads();  // the previous slice's readers of part[] are done
    if ((int)threadIdx.x < M) {
      const int k = threadIdx.x;
      const int node = a.order[(n_dest * L + s) * M + k];
      const int c = ((n_dest - node) % M + M) % M;  // relative index of the k-th source
      const int g = ((s - c) % L + L) % L;            // the GPU its slice s landed on
      part[k] = a.inbox + ((int64_t)(n_dest * L + g) * M + c) * slot + (int64_t)l_dest * B;  // element lo
    }
    __syncthreads();
    const int64_t nv = (hi - lo) / W;  // whole vectors of the slice
    float* const o = out + lo;
    for (int64_t v0 = tid; v0 < nv; v0 += kVecs * nthr) {
      V acc[kVecs], bsum[kBatched ? kVecs : 1];
#pragma unroll
      for (int u = 0; u < kVecs; ++u) acc[u] = zv;
#pragma unroll
      for (int u = 0; u < (kBatched ? kVecs : 1); ++u) bsum[u] = zv;
      for (int j0 = 0; j0 < M; j0 += kGroup) {
        V v[kGroup][kVecs];
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          const V* pj = reinterpret_cast<const V*>(part[min(j0 + q, M - 1)]);
#pragma unroll
          for (int u = 0; u < kVecs; ++u) {
            const int64_t vi = v0 + u * nthr;
            v[q][u] = (j0 + q < M && vi < nv) ? __ldcs(pj + vi) : zv;
          }
        }
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          const int j = j0 + q;
          if (j >= M) break;
#pragma unroll
          for (int u = 0; u < kVecs; ++u) {
            if constexpr (kBatched)
              add_v(bsum[u], v[q][u]);
            else
              add_v(acc[u], v[q][u]);
          }
          if constexpr (kBatched) {
            if ((j + 1) % L == 0 || j + 1 == M) {  // end of a batch
#pragma unroll
              for (int u = 0; u < kVecs; ++u) {
                add_v(acc[u], bsum[u]);
                bsum[u] = zv;
              }
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kVecs; ++u) {
        const int64_t vi = v0 + u * nthr;
        if (vi < nv) {
          float* d = o + W * vi;
          const V res = epilogue_v(acc[u], d, a.epilogue, M * L);
          if (store_ok(d, 4 * W, out + lo, out + hi)) __stcs(reinterpret_cast<V*>(d), res);
        }
      }
    }
    // the elements past the slice's whole vectors
    const int64_t x = lo + W * nv + tid;
    if (x < hi) {
      float acc = 0.f, bsum = 0.f;
      for (int j = 0; j < M; ++j) {
        const float pv = __ldcs(part[j] + (x - lo));
        if constexpr (kBatched) {
          bsum = __fadd_rn(bsum, pv);
          if ((j + 1) % L == 0 || j + 1 == M) {
            acc = __fadd_rn(acc, bsum);
            bsum = 0.f;
          }
        } else {
          acc = __fadd_rn(acc, pv);
        }
      }
      if (store_ok(out + x, 4, out + lo, out + hi)) __stcs(out + x, epilogue1(acc, out + x, a.epilogue, M * L));
    }
  }
}

using LandKernel = void (*)(RsArgs);

template <class V, int kVecs>
LandKernel land_vec_kernel_for(int M, int L) {
  if (M > L) return rs_land_vec_kernel<true, 1, V, kVecs>;
  return M == 1 ? rs_land_vec_kernel<false, 1, V, kVecs> : rs_land_vec_kernel<false, 2, V, kVecs>;
}

// vec: vector width of the landing (4, 2, or 0 for 4-byte accesses); wide:
// the landing grid is too small to fill the GPU (8 vectors per thread).
LandKernel land_kernel_for(int M, int L, int vec, bool wide) {
  if (vec == 4) return wide ? land_vec_kernel_for<float4, 8>(M, L) : land_vec_kernel_for<float4, 2>(M, L);
  if (vec == 2) return wide ? land_vec_kernel_for<float2, 8>(M, L) : land_vec_kernel_for<float2, 2>(M, L);
  if (M > L) return rs_land_kernel<true>;
  return M == 1 ? rs_land_kernel<false> : rs_land_grouped_kernel<false, 2>;
}

template <int L>
int launch_sum_t(const RsArgs& a, int grid, bool wide, cudaStream_t s) {
  if (wide)
    rs_sum_kernel<L, true><<<grid, kRsThreads, 0, s>>>(a);
  else
    rs_sum_kernel<L, false><<<grid, kRsThreads, 0, s>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace

TIDE_BOUNDS_COUNTER(rs_staged_bounds)

int launch_rs_staged(const RsArgs& a, int sum_grid, bool sum_wide, int land_grid_x, int land_vec, bool land_wide,
                     void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  int err = (int)cudaErrorInvalidValue;
  switch (a.L) {
    case 1: err = launch_sum_t<1>(a, sum_grid, sum_wide, s); break;
    case 2: err = launch_sum_t<2>(a, sum_grid, sum_wide, s); break;
    case 3: err = launch_sum_t<3>(a, sum_grid, sum_wide, s); break;
    case 4: err = launch_sum_t<4>(a, sum_grid, sum_wide, s); break;
    case 5: err = launch_sum_t<5>(a, sum_grid, sum_wide, s); break;
    case 6: err = launch_sum_t<6>(a, sum_grid, sum_wide, s); break;
    case 7: err = launch_sum_t<7>(a, sum_grid, sum_wide, s); break;
    case 8: err = launch_sum_t<8>(a, sum_grid, sum_wide, s); break;
  }
  if (err != cudaSuccess) return err;
  land_kernel_for(a.M, a.L, land_vec, land_wide)<<<dim3(land_grid_x, a.N), 256, 0, s>>>(a);
  return (int)cudaGetLastError();
}

int rs_land_blocks_per_sm(int M, int L, int vec) {
  int n = 0;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, land_kernel_for(M, L, vec, false), 256, 0) == cudaSuccess
             ? n
             : 0;
}

}  // namespace tide

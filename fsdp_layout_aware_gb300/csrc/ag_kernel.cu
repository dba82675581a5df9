// TIDE-AG direct landing on one GPU: every rank's packed shard piece of every
// parameter is written once, at its final parameter-major address, with no
// rank-major temporary ("All-gather: parameters land at their final address"
// in "The Endgame of FSDP Communication"; "What shipped" in the TIDE news
// post; Figure 1 of the preprint).  On the pages a copy engine multicasts the
// piece through NVSwitch; here both ends are in this GPU's HBM, so the copy is
// an SM kernel that streams each piece with 16-byte loads and stores.
//
// Piece (p, r) is e_p contiguous elements at shard_r + op going to
// param_p + r*e_p.  When the two addresses agree mod 16 the body moves as
// aligned 16-byte vectors.  When they do not (odd row lengths make op and
// r*e_p arbitrary), each thread builds one destination-aligned 16-byte word
// from the two source granules that overlap it and a funnel shift, so loads
// and stores both stay 16-byte wide.

#include <cuda_runtime.h>

#include <cstdint>

#include "check.cuh"
#include "tide_internal.h"

namespace tide {
namespace {

union Vec16 {
  uint4 v;
  uint32_t w[4];
  uint16_t h[8];
};

__device__ __forceinline__ void copy_elem(unsigned char* d, const unsigned char* s, int eb, const void* lo,
                                          const void* hi) {
  if (!store_ok(d, eb, lo, hi)) return;
  if (eb == 4)
    *reinterpret_cast<uint32_t*>(d) = *reinterpret_cast<const uint32_t*>(s);
  else
    *reinterpret_cast<uint16_t*>(d) = *reinterpret_cast<const uint16_t*>(s);
}

// One warp copies one item.  Source and destination at the same address
// phase mod 16: a short element-wise head, then 16-byte vectors, four in
// flight per lane, then an element-wise tail.
__device__ __forceinline__ void warp_copy_same_phase(unsigned char* dst, const unsigned char* src, int64_t nbytes,
                                                     int eb, int lane) {
  const int64_t head = min(nbytes, (int64_t)((16 - ((uintptr_t)dst & 15)) & 15));
  const unsigned char* const end = dst + nbytes;
  for (int64_t i = (int64_t)lane * eb; i < head; i += 32 * eb) copy_elem(dst + i, src + i, eb, dst, end);
  const int64_t nv = (nbytes - head) >> 4;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + head);
  uint4* d4 = reinterpret_cast<uint4*>(dst + head);
  int64_t i = lane;
  for (; i + 96 < nv; i += 128) {
    const uint4 a = __ldcs(s4 + i), b = __ldcs(s4 + i + 32), c = __ldcs(s4 + i + 64), d = __ldcs(s4 + i + 96);
    if (store_ok(d4 + i, 16, dst, end)) __stcs(d4 + i, a);
    if (store_ok(d4 + i + 32, 16, dst, end)) __stcs(d4 + i + 32, b);
    if (store_ok(d4 + i + 64, 16, dst, end)) __stcs(d4 + i + 64, c);
    if (store_ok(d4 + i + 96, 16, dst, end)) __stcs(d4 + i + 96, d);
  }
  for (; i < nv; i += 32)
    if (store_ok(d4 + i, 16, dst, end)) __stcs(d4 + i, __ldcs(s4 + i));
  for (int64_t j = head + (nv << 4) + (int64_t)lane * eb; j < nbytes; j += 32 * eb)
    copy_elem(dst + j, src + j, eb, dst, end);
}

// Bytes [sh, sh + 16) of the 32-byte concatenation lo || hi (sh even).
__device__ __forceinline__ uint4 extract16(const uint4 lo, const uint4 hi, int sh) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint4 o;
  const bool half = (sh & 2) != 0;
#define TIDE_PICK(Q)                                                             \
  if (half) {                                                                    \
    o.x = __funnelshift_r(w[Q + 0], w[Q + 1], 16);                               \
    o.y = __funnelshift_r(w[Q + 1], w[Q + 2], 16);                               \
    o.z = __funnelshift_r(w[Q + 2], w[Q + 3], 16);                               \
    o.w = __funnelshift_r(w[Q + 3], w[Q + 4], 16);                               \
  } else {                                                                       \
    o.x = w[Q + 0];                                                              \
    o.y = w[Q + 1];                                                              \
    o.z = w[Q + 2];                                                              \
    o.w = w[Q + 3];                                                              \
  }
  switch (sh >> 2) {
    case 0: TIDE_PICK(0) break;
    case 1: TIDE_PICK(1) break;
    case 2: TIDE_PICK(2) break;
    default: TIDE_PICK(3) break;
  }
#undef TIDE_PICK
  return o;
}

__device__ __forceinline__ uint4 shfl16(const uint4 v, int src_lane) {
  uint4 o;
  o.x = __shfl_sync(0xffffffffu, v.x, src_lane);
  o.y = __shfl_sync(0xffffffffu, v.y, src_lane);
  o.z = __shfl_sync(0xffffffffu, v.z, src_lane);
  o.w = __shfl_sync(0xffffffffu, v.w, src_lane);
  return o;
}

__device__ __forceinline__ uint4 load_granule(uintptr_t g, uintptr_t s_lo, uintptr_t s_hi) {
  return (g + 16 > s_lo && g < s_hi) ? __ldcs(reinterpret_cast<const uint4*>(g)) : make_uint4(0, 0, 0, 0);
}

// Source and destination at different phases.  Destination word w covers
// bytes [d0 + 16w, d0 + 16w + 16); its bytes come from source address
// (that + src - dst), which straddles the aligned source granules g(w) and
// g(w) + 16 = g(w + 1).  In a round the warp handles words base + 32j + lane
// (j = 0..3, four in flight per lane); lane t loads g(w) for its words and
// takes g(w + 1) from lane t + 1 by a rotating shuffle -- lane 31's next
// granule is lane 0's granule of the following group, and lane 0 loads the
// one after the round.  Every granule is read once, and only if it holds a
// byte of the source range.  Called by all 32 lanes of the warp.
__device__ __forceinline__ void warp_copy_shifted(unsigned char* dst, const unsigned char* src, int64_t nbytes, int eb,
                                                  int lane) {
  const uintptr_t d_lo = (uintptr_t)dst, d_hi = d_lo + (uintptr_t)nbytes;
  const uintptr_t s_lo = (uintptr_t)src, s_hi = s_lo + (uintptr_t)nbytes;
  const uintptr_t d0 = d_lo & ~(uintptr_t)15;
  const int nw = (int)((d_hi + 15 - d0) >> 4);  // items are at most 64 KiB
  const uintptr_t delta = s_lo - d_lo;  // modular: source address = destination address + delta
  const int sh = (int)(delta & 15);
  const unsigned char* g_first = (const unsigned char*)((d0 + delta) & ~(uintptr_t)15);  // granule of word 0
  unsigned char* const dbase = (unsigned char*)d0;
  const int next_lane = (lane + 1) & 31;
  for (int base = 0; base < nw; base += 128) {
    uint4 lo[5];
#pragma unroll
    for (int j = 0; j < 4; ++j) lo[j] = load_granule((uintptr_t)(g_first + 16 * (base + 32 * j + lane)), s_lo, s_hi);
    lo[4] = lane == 0 ? load_granule((uintptr_t)(g_first + 16 * (base + 128)), s_lo, s_hi) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 hi = shfl16(lane == 0 ? lo[j + 1] : lo[j], next_lane);
      const int w = base + 32 * j + lane;
      if (w >= nw) continue;
      unsigned char* dw = dbase + 16 * w;
      Vec16 out;
      out.v = extract16(lo[j], hi, sh);
      const void* rng_lo = (const void*)d_lo;
      const void* rng_hi = (const void*)d_hi;
      if ((uintptr_t)dw >= d_lo && (uintptr_t)dw + 16 <= d_hi) {
        if (store_ok(dw, 16, rng_lo, rng_hi)) __stcs(reinterpret_cast<uint4*>(dw), out.v);
      } else if (eb == 2) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const uintptr_t addr = (uintptr_t)dw + 2 * b;
          if (addr >= d_lo && addr < d_hi && store_ok((void*)addr, 2, rng_lo, rng_hi))
            *reinterpret_cast<uint16_t*>(addr) = out.h[b];
        }
      } else {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uintptr_t addr = (uintptr_t)dw + 4 * b;
          if (addr >= d_lo && addr < d_hi && store_ok((void*)addr, 4, rng_lo, rng_hi))
            *reinterpret_cast<uint32_t*>(addr) = out.w[b];
        }
      }
    }
  }
}

// Warp w of W processes units w, w + W, ...; the plan cut the units to equal
// cost (bytes copied plus a per-item start-up charge), so a small or ragged
// item never leaves one warp with more than its share, and neighbouring warps
// copy neighbouring parts of the item list.
__global__ void __launch_bounds__(kAgThreads, 4) ag_place_kernel(const __grid_constant__ AgArgs a) {
  const int eb = a.elem_bytes;
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t u = warp; u < a.n_units; u += nwarps) {
    const UnitStart s = a.units[u], e = a.units[u + 1];
    const int64_t last = e.off > 0 ? e.item : (int64_t)e.item - 1;
    for (int64_t i = s.item; i <= last; ++i) {
      const AgItem item = a.items[i];
      const int32_t ea = i == s.item ? s.off : 0;
      const int32_t ee = i == e.item ? e.off : item.n;
      if (ea >= ee) continue;
      const unsigned char* src = a.shard_tab[item.r] + (item.src_off + ea) * eb;
      unsigned char* dst = a.param_tab[item.p] + (item.dst_off + ea) * eb;
      const int64_t nbytes = (int64_t)(ee - ea) * eb;
      if ((((uintptr_t)src ^ (uintptr_t)dst) & 15) == 0)
        warp_copy_same_phase(dst, src, nbytes, eb, lane);
      else
        warp_copy_shifted(dst, src, nbytes, eb, lane);
    }
  }
}

}  // namespace

TIDE_BOUNDS_COUNTER(ag_kernel_bounds)

namespace {
// Positive control of the store checks: asks about an address outside a
// made-up range, without touching memory; a checked build counts one.
__global__ void bounds_selftest_kernel() {
  if (threadIdx.x == 0) (void)store_ok((const void*)64, 4, (const void*)0, (const void*)32);
}
}  // namespace

int ag_bounds_selftest() {
  bounds_selftest_kernel<<<1, 32>>>();
  return (int)cudaGetLastError();
}

int launch_ag(const AgArgs& a, int grid, void* stream) {
  ag_place_kernel<<<grid, kAgThreads, 0, (cudaStream_t)stream>>>(a);
  return (int)cudaGetLastError();
}

int ag_blocks_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ag_place_kernel, kAgThreads, 0) != cudaSuccess) return 0;
  return n;
}

}  // namespace tide

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

#include "tide_internal.h"

namespace tide {
namespace {

union Vec16 {
  uint4 v;
  uint32_t w[4];
  uint16_t h[8];
};

__device__ __forceinline__ void copy_elem(unsigned char* d, const unsigned char* s, int eb) {
  if (eb == 4)
    *reinterpret_cast<uint32_t*>(d) = *reinterpret_cast<const uint32_t*>(s);
  else
    *reinterpret_cast<uint16_t*>(d) = *reinterpret_cast<const uint16_t*>(s);
}

// Source and destination at the same address phase mod 16.
__device__ __forceinline__ void copy_same_phase(unsigned char* dst, const unsigned char* src, int64_t nbytes,
                                                int eb) {
  const int64_t head = min(nbytes, (int64_t)((16 - ((uintptr_t)dst & 15)) & 15));
  for (int64_t i = (int64_t)threadIdx.x * eb; i < head; i += (int64_t)blockDim.x * eb) copy_elem(dst + i, src + i, eb);
  const int64_t nv = (nbytes - head) >> 4;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + head);
  uint4* d4 = reinterpret_cast<uint4*>(dst + head);
  const int64_t T = blockDim.x;
  int64_t i = threadIdx.x;
  for (; i + 3 * T < nv; i += 4 * T) {
    const uint4 a = __ldcs(s4 + i), b = __ldcs(s4 + i + T), c = __ldcs(s4 + i + 2 * T), d = __ldcs(s4 + i + 3 * T);
    __stcs(d4 + i, a);
    __stcs(d4 + i + T, b);
    __stcs(d4 + i + 2 * T, c);
    __stcs(d4 + i + 3 * T, d);
  }
  for (; i < nv; i += T) __stcs(d4 + i, __ldcs(s4 + i));
  for (int64_t j = head + (nv << 4) + (int64_t)threadIdx.x * eb; j < nbytes; j += T * eb) copy_elem(dst + j, src + j, eb);
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

// Source and destination at different phases.  Destination word w covers
// bytes [d0 + 16w, d0 + 16w + 16); its source bytes start at that address +
// (src - dst) and straddle two aligned source granules.  A granule is loaded
// only if it holds at least one byte of the source range.
__device__ __forceinline__ void copy_shifted(unsigned char* dst, const unsigned char* src, int64_t nbytes, int eb) {
  const uintptr_t d_lo = (uintptr_t)dst, d_hi = d_lo + (uintptr_t)nbytes;
  const uintptr_t s_lo = (uintptr_t)src, s_hi = s_lo + (uintptr_t)nbytes;
  const uintptr_t d0 = d_lo & ~(uintptr_t)15;
  const int64_t nw = (int64_t)((d_hi + 15 - d0) >> 4);
  const uintptr_t delta = s_lo - d_lo;  // modular; source address = destination address + delta
  const int sh = (int)(delta & 15);
  for (int64_t w = threadIdx.x; w < nw; w += blockDim.x) {
    const uintptr_t dw = d0 + 16 * (uintptr_t)w;
    const uintptr_t g0 = (dw + delta) & ~(uintptr_t)15, g1 = g0 + 16;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
    if (g0 + 16 > s_lo && g0 < s_hi) lo = __ldg(reinterpret_cast<const uint4*>(g0));
    if (g1 + 16 > s_lo && g1 < s_hi) hi = __ldg(reinterpret_cast<const uint4*>(g1));
    Vec16 out;
    out.v = extract16(lo, hi, sh);
    if (dw >= d_lo && dw + 16 <= d_hi) {
      __stcs(reinterpret_cast<uint4*>(dw), out.v);
    } else if (eb == 2) {
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const uintptr_t addr = dw + 2 * b;
        if (addr >= d_lo && addr < d_hi) *reinterpret_cast<uint16_t*>(addr) = out.h[b];
      }
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uintptr_t addr = dw + 4 * b;
        if (addr >= d_lo && addr < d_hi) *reinterpret_cast<uint32_t*>(addr) = out.w[b];
      }
    }
  }
}

__global__ void __launch_bounds__(kAgThreads) ag_place_kernel(const __grid_constant__ AgArgs a) {
  const int eb = a.elem_bytes;
  for (int64_t it = blockIdx.x; it < a.n_items; it += gridDim.x) {
    const AgItem item = a.items[it];
    const unsigned char* src = a.shard_tab[item.r] + item.src_off * eb;
    unsigned char* dst = a.param_tab[item.p] + item.dst_off * eb;
    const int64_t nbytes = (int64_t)item.n * eb;
    if ((((uintptr_t)src ^ (uintptr_t)dst) & 15) == 0)
      copy_same_phase(dst, src, nbytes, eb);
    else
      copy_shifted(dst, src, nbytes, eb);
  }
}

}  // namespace

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

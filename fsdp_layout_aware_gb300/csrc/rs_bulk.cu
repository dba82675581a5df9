// TIDE-RS hot loop, bulk-copy pipeline (sm_103a).
//
// Same result as rs_fused (bit for bit: identical fp32 addition order) but the
// contributors' bf16 data reach the SM through the Tensor Memory Accelerator
// instead of per-thread loads, so the bytes in flight per SM are set by the
// shared-memory rings, not by registers:
//
//   * four CTAs per SM (four independent pipelines), each a producer warp and
//     4 consumer warps;
//   * per CTA a ring of S stages (3 of 16 KiB with L = 8); a stage holds,
//     for one tile of T = 8*V = 1024 outputs of one item and one source
//     node, the aligned 16-byte windows of that node's L contributors (L
//     windows of at most 2 KiB), so a tile takes M stages;
//   * the producer walks the CTA's items (round-robin over the grid: the
//     consumers follow the producer's order without a shared counter) and,
//     per tile, fills one stage per source node in the tile's level-2 order
//     (the Latin-square landing order of its slice): it arms the stage's
//     "full" mbarrier with the expected byte count and issues one
//     cp.async.bulk per contributor.  Every request moves a whole window, so
//     the request count per byte does not grow with the number of nodes;
//   * consumer thread v owns vector v (outputs 8v .. 8v+7) of every tile: per
//     stage it sums the node's L contributions from shared memory (level 1,
//     l ascending) and adds the partial to its running level-2 sum in
//     registers (batches of L nodes when M > L); after the tile's last node
//     it stores its 8 finished outputs (16-byte stores, realigned across
//     lanes when the shard is not 16-byte aligned there);
//   * a consumer warp releases the stage ("empty" mbarrier) as soon as its
//     level-1 loads are done, so the producer refills it while the sums run.
//
// Padding ranges are zero-filled by the consumers; parameters whose N
// gradients do not share an address phase mod 16 (bulk copies need 16-byte
// aligned sources) are reduced by the consumers with element-wise loads.
//
// Every wait is bounded by %globaltimer.  On timeout a thread records
// TIDE_DEVICE_TIMEOUT in the plan's status word and raises the CTA's abort
// flag; all loops stop, the CTA waits (again bounded) until every bulk copy it
// issued has landed, and returns.  tide_plan_check reports the status word.

#include <cuda_runtime.h>

#include <cstdint>

#include "bulk_ptx.cuh"
#include "rs_device.cuh"
#include "tide_internal.h"

namespace tide {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;

enum TileKind : int32_t { TILE_BULK = 0, TILE_PAD = 1, TILE_DIRECT = 2, TILE_END = 3 };

struct TileDesc {
  float* dst;        // first output of the tile
  int64_t src_off;   // DIRECT: element offset inside the contributors' gradients
  int32_t n;         // outputs in the tile
  int32_t ph;        // BULK: elements of the first granule before the first output
  int32_t kind;
  int32_t p;         // DIRECT: parameter
  uint32_t ord_lo;   // level-2 source-node order, one byte per node: nodes 0..3
  uint32_t ord_hi;   //   and 4..7 (M <= 8)
  int32_t k;         // BULK: the stage holds the windows of the k-th node in the level-2 order
  int32_t pad_;
};

__device__ __forceinline__ void consumer_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

__device__ __forceinline__ uint4 lds16(const unsigned char* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

// Shared-memory carve-up, computed on the host (rs_bulk_layout).
struct Smem {
  unsigned char* stages;
  TileDesc* desc;        // [S]
  uint64_t* full;        // [S]
  uint64_t* empty;       // [S]
  int* ctl;              // [0] abort flag, [1 + s] rounds issued on stage s,
                         // [1 + kMaxBulkStages + s] consumers' wait result for stage s
};

__device__ __forceinline__ Smem carve(unsigned char* base, const RsArgs& a) {
  Smem m;
  m.stages = base;
  m.desc = reinterpret_cast<TileDesc*>(base + a.bulk.off_desc);
  m.full = reinterpret_cast<uint64_t*>(base + a.bulk.off_bar);
  m.empty = m.full + a.bulk.stages;
  m.ctl = reinterpret_cast<int*>(base + a.bulk.off_ctl);
  return m;
}

// Bounded wait for the phase of `bar` with the given parity.  False on
// timeout (recorded in the plan's status word, abort raised) or when the CTA
// is already aborting.
__device__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag, const RsArgs& a) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > a.bulk.wait_limit_ns) {
      atomicOr(a.bulk.status, TIDE_DEVICE_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// A phase another thread has already seen complete: acquire it in this thread
// too (returns at once; bounded all the same).
__device__ __forceinline__ void acquire_completed(uint64_t* bar, uint32_t parity) {
  for (int i = 0; i < (1 << 20) && !mbar_try_wait(bar, parity); ++i) {
  }
}

// The producer warp decides as one: lane 0 waits, the warp follows its answer.
__device__ __forceinline__ bool warp_wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                const RsArgs& a) {
  const int lane = threadIdx.x & 31;
  int ok = 0;
  if (lane == 0) ok = wait_phase(bar, parity, abort_flag, a) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok && lane != 0) acquire_completed(bar, parity);
  return ok != 0;
}

template <int L>
__device__ void producer(const RsArgs& a, const Smem& m) {
  const int lane = threadIdx.x & 31;
  const int N = a.N;
  const int V = a.bulk.V;
  const int T = 8 * V;
  volatile int* abort_flag = m.ctl;
  uint32_t stage = 0, round = 0;
  int64_t tile = 0;
  bool ok = true;
  // Claim the next stage: wait until the consumers have released its previous use.
  auto acquire = [&]() -> bool { return warp_wait_phase(&m.empty[stage], (round & 1) ^ 1, abort_flag, a); };
  auto advance = [&]() {
    if (++stage == (uint32_t)a.bulk.stages) {
      stage = 0;
      ++round;
    }
    ++tile;
  };
  for (int64_t it = blockIdx.x; ok && it < a.n_items; it += gridDim.x) {
    const RsItem item = a.items[it];
    float* dst = a.shard_tab[item.r] + item.dst_off;
    uint32_t ord_lo = 0, ord_hi = 0;
    {
      const uint8_t* ord = a.order + ((item.r / L) * L + item.slice) * a.M;
      for (int k = 0; k < a.M; ++k) {
        if (k < 4) ord_lo |= (uint32_t)ord[k] << (8 * k);
        else ord_hi |= (uint32_t)ord[k] << (8 * (k - 4));
      }
    }
    if (item.kind == RS_PAD || !a.uniform_phase[item.p]) {
      if (!(ok = acquire())) break;
      if (lane == 0) {
        TileDesc d;
        d.dst = dst;
        d.src_off = item.src_off;
        d.n = item.n;
        d.ph = 0;
        d.kind = item.kind == RS_PAD ? TILE_PAD : TILE_DIRECT;
        d.p = item.p;
        d.ord_lo = ord_lo;
        d.ord_hi = ord_hi;
        m.desc[stage] = d;
        if (tile != a.bulk.test_drop_tile) mbar_arrive(&m.full[stage]);
      }
      __syncwarp();
      advance();
      continue;
    }
    // Lane c holds contributor c's pointer (g0) and contributor c + 32's (g1).
    const uint16_t* g0 = lane < N ? a.grad_tab[(int64_t)item.p * N + lane] + item.src_off : nullptr;
    const uint16_t* g1 = lane + 32 < N ? a.grad_tab[(int64_t)item.p * N + lane + 32] + item.src_off : nullptr;
    const uintptr_t first = __shfl_sync(0xffffffffu, (unsigned long long)(uintptr_t)g0, 0);
    const int ph0 = (int)((first >> 1) & 7);
    for (int e = 0; ok && e < item.n;) {
      const int ph = e == 0 ? ph0 : 0;
      const int nt = min(item.n - e, T - ph);
      const uint32_t bytes = (uint32_t)((2 * (ph + nt) + 15) & ~15);
      for (int k = 0; k < a.M; ++k) {
        if (!(ok = acquire())) break;
        // the k-th node of the level-2 order; lane l < L loads its contributor node*L + l
        const int node = (int)(((k < 4 ? ord_lo >> (8 * k) : ord_hi >> (8 * (k - 4)))) & 0xFFu);
        const int c = node * L + (lane < L ? lane : 0);
        const uintptr_t p0 = __shfl_sync(0xffffffffu, (unsigned long long)(uintptr_t)g0, c & 31);
        const uintptr_t p1 = __shfl_sync(0xffffffffu, (unsigned long long)(uintptr_t)g1, c & 31);
        const uint16_t* gsrc = reinterpret_cast<const uint16_t*>(c < 32 ? p0 : p1);
        unsigned char* sbuf = m.stages + (size_t)stage * a.bulk.stage_bytes;
        const bool drop = tile == a.bulk.test_drop_tile;
        if (lane == 0) {
          TileDesc d;
          d.dst = dst + e;
          d.src_off = 0;
          d.n = nt;
          d.ph = ph;
          d.kind = TILE_BULK;
          d.p = item.p;
          d.ord_lo = ord_lo;
          d.ord_hi = ord_hi;
          d.k = k;
          d.pad_ = 0;
          m.desc[stage] = d;
          if (!drop) {
            mbar_arrive_expect_tx(&m.full[stage], bytes * (uint32_t)L);
            m.ctl[1 + stage] = (int)round + 1;
          }
        }
        __syncwarp();
        if (!drop && lane < L) bulk_load(sbuf + (size_t)lane * 16 * V, gsrc + e - ph, bytes, &m.full[stage]);
        advance();
      }
      e += nt;
    }
  }
  if (ok && acquire()) {
    if (lane == 0) {
      m.desc[stage].kind = TILE_END;
      mbar_arrive(&m.full[stage]);
    }
  }
  __syncwarp();
}

template <int L>
__device__ void consumers(const RsArgs& a, const Smem& m) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int M = a.M;
  const int V = a.bulk.V;
  volatile int* abort_flag = m.ctl;
  uint32_t stage = 0, round = 0;
  // Level-2 state of this thread's vector, carried across the M stages of a
  // tile: the running batch sum and the running total.
  float acc2[8], bsum[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc2[i] = bsum[i] = 0.f;
  for (;;) {
    // The consumer warps decide as one (a named barrier must never lose a
    // participant): thread 0 waits, publishes the answer in this stage's slot,
    // and every thread then acquires the completed phase itself.  (Every warp
    // waiting on the mbarrier by itself measured 3-5% slower.)
    if (tid == 0) m.ctl[1 + kMaxBulkStages + stage] = wait_phase(&m.full[stage], round & 1, abort_flag, a) ? 1 : 0;
    consumer_barrier();
    if (!m.ctl[1 + kMaxBulkStages + stage]) break;
    if (tid != 0) acquire_completed(&m.full[stage], round & 1);
    const TileDesc d = m.desc[stage];
    if (d.kind == TILE_END) break;
    if (d.kind == TILE_BULK) {
      const unsigned char* sbuf = m.stages + (size_t)stage * a.bulk.stage_bytes;
      const int nvec = (d.ph + d.n + 7) >> 3;
      if (tid < nvec) {
        // level 1: the node's L contributions, l ascending
        float acc1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc1[i] = 0.f;
        uint4 x[L];
#pragma unroll
        for (int l = 0; l < L; ++l) x[l] = lds16(sbuf + (size_t)l * 16 * V + 16 * tid);
#pragma unroll
        for (int l = 0; l < L; ++l) add_bf16x8(acc1, x[l]);
        // level 2: this node is the d.k-th of the tile's order; a batch of L
        // ends after every L-th node and at the last
#pragma unroll
        for (int i = 0; i < 8; ++i) bsum[i] = __fadd_rn(bsum[i], acc1[i]);
        if ((d.k + 1) % L == 0 || d.k + 1 == M) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            acc2[i] = __fadd_rn(acc2[i], bsum[i]);
            bsum[i] = 0.f;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.empty[stage]);  // this warp is done reading the stage
      if (d.k + 1 == M) {
        // the tile's last node: thread v holds the finished sums of its 8 outputs
        if (tid - lane < nvec) {  // warp-uniform: the shuffles need every lane
          const int delta = (int)(((unsigned)d.ph - (unsigned)((uintptr_t)d.dst >> 2)) & 3u);
          const int e0 = tid * 8 - d.ph;
          epilogue8(acc2, d.dst, e0, d.n, a.epilogue, a.N);
          if (delta == 0)
            store8_aligned(d.dst, e0, d.n, acc2);
          else
            store8_shifted(d.dst, e0, d.n, delta, lane, acc2);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) acc2[i] = bsum[i] = 0.f;
      }
    } else if (d.kind == TILE_PAD) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.empty[stage]);
      pad_fill(d.dst, d.n, a.epilogue, tid, kConsumers);
    } else {  // TILE_DIRECT: contributors at different address phases
      __syncwarp();
      if (lane == 0) mbar_arrive(&m.empty[stage]);
      const uint16_t* const* gtab = a.grad_tab + (int64_t)d.p * a.N;
      for (int e0 = tid * 8; e0 < d.n; e0 += kConsumers * 8) {
        const int cnt = min(8, d.n - e0);
        float sum2[8], bs[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) sum2[i] = bs[i] = 0.f;
        for (int k = 0; k < M; ++k) {
          const int node = (int)(((k < 4 ? d.ord_lo >> (8 * k) : d.ord_hi >> (8 * (k - 4)))) & 0xFFu);
          float acc1[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc1[i] = 0.f;
#pragma unroll
          for (int l = 0; l < L; ++l) {
            const uint16_t* src = gtab[node * L + l] + d.src_off + e0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (i < cnt) acc1[i] = __fadd_rn(acc1[i], __uint_as_float((uint32_t)__ldcs(src + i) << 16));
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) bs[i] = __fadd_rn(bs[i], acc1[i]);
          if ((k + 1) % L == 0 || k + 1 == M) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              sum2[i] = __fadd_rn(sum2[i], bs[i]);
              bs[i] = 0.f;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < cnt && store_ok(d.dst + e0 + i, 4, d.dst, d.dst + d.n))
            __stcs(d.dst + e0 + i, epilogue1(sum2[i], d.dst + e0 + i, a.epilogue, a.N));
      }
    }
    if (++stage == (uint32_t)a.bulk.stages) {
      stage = 0;
      ++round;
    }
  }
}

template <int L>
__global__ void __launch_bounds__(kConsumers + 32, kBulkCtasPerSm) rs_bulk_kernel(const __grid_constant__ RsArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const Smem m = carve(smem, a);
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.bulk.stages; ++s) {
      mbar_init(&m.full[s], 1);
      mbar_init(&m.empty[s], kConsumerWarps);
      m.ctl[1 + s] = 0;
      m.ctl[1 + kMaxBulkStages + s] = 0;
    }
    m.ctl[0] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x >= kConsumers)
    producer<L>(a, m);
  else
    consumers<L>(a, m);
  __syncthreads();
  // After an abort, wait (bounded) until every bulk copy this CTA issued has
  // landed, so that none writes into shared memory after the CTA exits.
  if (threadIdx.x == 0 && m.ctl[0]) {
    for (int s = 0; s < a.bulk.stages; ++s) {
      const int issued = m.ctl[1 + s];
      if (issued == 0) continue;
      const uint32_t parity = (uint32_t)(issued - 1) & 1;
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(&m.full[s], parity) && global_ns() - t0 < a.bulk.wait_limit_ns) {
      }
    }
  }
  __syncthreads();
}

template <int L>
int launch_t(const RsArgs& a, int grid, cudaStream_t s) {
  rs_bulk_kernel<L><<<grid, kConsumers + 32, a.bulk.smem_bytes, s>>>(a);
  return (int)cudaGetLastError();
}

template <int L>
int occupancy_t(int smem_bytes) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rs_bulk_kernel<L>, kConsumers + 32, smem_bytes) != cudaSuccess)
    return 0;
  return n;
}

template <int L>
int setup_t(int smem_bytes) {
  return (int)cudaFuncSetAttribute(rs_bulk_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

}  // namespace

TIDE_BOUNDS_COUNTER(rs_bulk_bounds)

BulkLayout rs_bulk_layout(int N, int M, int L, int smem_budget) {
  BulkLayout b{};
  b.V = 128;
  b.stage_bytes = 16 * L * b.V;
  const int fixed = kMaxBulkStages * (int)sizeof(TileDesc) + 2 * kMaxBulkStages * 8 + (1 + 2 * kMaxBulkStages) * 4 + 256;
  int stages = (smem_budget - fixed) / b.stage_bytes;
  stages = stages < 2 ? 2 : (stages > kMaxBulkStages ? kMaxBulkStages : stages);
  b.stages = stages;
  b.off_desc = stages * b.stage_bytes;
  b.off_bar = b.off_desc + kMaxBulkStages * (int)sizeof(TileDesc);
  b.off_ctl = b.off_bar + 2 * kMaxBulkStages * 8;
  b.smem_bytes = b.off_ctl + (1 + 2 * kMaxBulkStages) * 4;
  (void)N;
  (void)M;
  return b;
}

int rs_bulk_setup(int L, int smem_bytes) {
  switch (L) {
    case 1: return setup_t<1>(smem_bytes);
    case 2: return setup_t<2>(smem_bytes);
    case 3: return setup_t<3>(smem_bytes);
    case 4: return setup_t<4>(smem_bytes);
    case 5: return setup_t<5>(smem_bytes);
    case 6: return setup_t<6>(smem_bytes);
    case 7: return setup_t<7>(smem_bytes);
    case 8: return setup_t<8>(smem_bytes);
  }
  return (int)cudaErrorInvalidValue;
}

int rs_bulk_blocks_per_sm(int L, int smem_bytes) {
  switch (L) {
    case 1: return occupancy_t<1>(smem_bytes);
    case 2: return occupancy_t<2>(smem_bytes);
    case 3: return occupancy_t<3>(smem_bytes);
    case 4: return occupancy_t<4>(smem_bytes);
    case 5: return occupancy_t<5>(smem_bytes);
    case 6: return occupancy_t<6>(smem_bytes);
    case 7: return occupancy_t<7>(smem_bytes);
    case 8: return occupancy_t<8>(smem_bytes);
  }
  return 0;
}

int launch_rs_bulk(const RsArgs& a, int grid, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  switch (a.L) {
    case 1: return launch_t<1>(a, grid, s);
    case 2: return launch_t<2>(a, grid, s);
    case 3: return launch_t<3>(a, grid, s);
    case 4: return launch_t<4>(a, grid, s);
    case 5: return launch_t<5>(a, grid, s);
    case 6: return launch_t<6>(a, grid, s);
    case 7: return launch_t<7>(a, grid, s);
    case 8: return launch_t<8>(a, grid, s);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace tide

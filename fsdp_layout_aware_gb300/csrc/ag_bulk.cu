// TIDE-AG direct landing through the Tensor Memory Accelerator: one thread
// per SM moves the aligned middle of every piece global -> shared -> global
// with bulk copies ("All-gather: parameters land at their final address" in
// "The Endgame of FSDP Communication"; "What shipped" in the TIDE news post:
// the pages' all-gather uses no SM threads; here one thread per SM issues
// the copies and the rest of the SM is left idle).
//
// The plan cuts every all-gather item whose source and destination share
// their address phase mod 16 into a head, a 16-byte aligned middle and a tail;
// the middles, in chunks of at most 32 KiB, are this kernel's work list, and
// heads, tails and phase-mismatched items go to ag_place_kernel.
//
// Pipeline per CTA (one per SM, a single thread): a ring of kStages 32 KiB
// shared-memory stages.  Chunk j is loaded into stage j mod kStages with its
// completion counted on that stage's mbarrier; kLookahead chunks later the
// thread waits for the load and issues the bulk store of the stage to the
// chunk's destination (one bulk async-group per store).  Before a stage is
// loaded again, the store that last read it must be done reading, which is
// "at most kStages - kLookahead newer groups pending".  So kLookahead loads
// and kStages - kLookahead stores are in flight per SM.
//
// Loads and stores carry an evict-first L2 policy.  Without it the stores
// leave L2 full of dirty lines that the next kernel (the reduce-scatter in a
// training step) has to write back: measured on llama70b, this kernel took
// 0.496 ms against the SM kernel's 0.520 ms, but the reduce-scatter after it
// slowed from 2.365 to 2.418 ms; with the policy the two take 0.516 and
// 2.374 ms and the step is level with the SM kernel's.
//
// Every wait is bounded by %globaltimer.  On timeout the thread records
// TIDE_DEVICE_TIMEOUT in the plan's status word, stops issuing, waits
// (bounded again) for the loads it issued, waits for its stores, and returns.
// A test hook (TIDE_OPT_TEST_DROP_TILE) arms one stage without issuing its
// load, so that path runs without any fault.

#include <cuda_runtime.h>

#include <cstdint>

#include "bulk_ptx.cuh"
#include "tide_internal.h"

namespace tide {
namespace {

constexpr int kStages = 7;
constexpr int kLookahead = 4;
constexpr uint32_t kChunkBytes = 2 * kAgBulkChunkElems;
constexpr int kSmemBytes = kStages * (int)kChunkBytes + kStages * 8;

__device__ __forceinline__ bool wait_loaded(uint64_t* bar, int64_t i, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(&bar[i % kStages], (uint32_t)((i / kStages) & 1)))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}

__global__ void __launch_bounds__(32, 1) ag_bulk_kernel(const __grid_constant__ AgBulkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kStages * kChunkBytes);
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

  const uint64_t pol = policy_evict_first();  // every byte is read once and written once
  unsigned char* pend_dst[kStages];
  uint32_t pend_bytes[kStages];
  int64_t issued = 0, retired = 0;
  bool ok = true;
  for (int64_t c = blockIdx.x; c < a.n_items; c += gridDim.x) {
    if (issued - retired == kLookahead) {
      // retire the oldest load: wait for it, then store its stage
      const int s = (int)(retired % kStages);
      if (!wait_loaded(bar, retired, a.wait_limit_ns)) {
        ok = false;
        break;
      }
      fence_proxy_async_smem();
      bulk_store_policy(pend_dst[s], smem + s * kChunkBytes, pend_bytes[s], pol);
      bulk_commit();
      ++retired;
    }
    // the stage about to be loaded was last read by the store of chunk
    // issued - kStages; at most kStages - kLookahead stores are newer
    if (issued >= kStages) bulk_wait_read<kStages - kLookahead>();
    const AgItem it = a.items[c];
    const int s = (int)(issued % kStages);
    const uint32_t bytes = 2u * (uint32_t)it.n;
    mbar_arrive_expect_tx(&bar[s], bytes);
    if (issued != a.test_drop_chunk)  // test hook: an armed stage whose data never comes
      bulk_load_policy(smem + s * kChunkBytes, a.shard_tab[it.r] + 2 * it.src_off, bytes, &bar[s], pol);
    pend_dst[s] = a.param_tab[it.p] + 2 * it.dst_off;
    pend_bytes[s] = bytes;
    ++issued;
  }
  while (ok && retired < issued) {
    const int s = (int)(retired % kStages);
    if (!wait_loaded(bar, retired, a.wait_limit_ns)) {
      ok = false;
      break;
    }
    fence_proxy_async_smem();
    bulk_store_policy(pend_dst[s], smem + s * kChunkBytes, pend_bytes[s], pol);
    bulk_commit();
    ++retired;
  }
  if (!ok) {
    atomicOr(a.status, TIDE_DEVICE_TIMEOUT);
    // The loads still in flight write this CTA's shared memory: let them land.
    for (int64_t i = retired; i < issued; ++i) wait_loaded(bar, i, a.wait_limit_ns);
  }
  bulk_wait_all();  // every store has written global memory
}

}  // namespace

int ag_bulk_smem_bytes() { return kSmemBytes; }

int ag_bulk_setup() {
  return (int)cudaFuncSetAttribute(ag_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

int launch_ag_bulk(const AgBulkArgs& a, int grid, void* stream) {
  ag_bulk_kernel<<<grid, 32, kSmemBytes, (cudaStream_t)stream>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace tide

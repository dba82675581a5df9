// tide_rs_reduce_noalloc: the reduce-scatter for callers that cannot allocate
// device memory.
//
// tide_rs_reduce keeps its work list and per-call pointer tables in device
// memory that the plan allocates on first use (cudaMalloc, cudaHostAlloc).
// Some callers cannot do that: a process whose device memory is all owned by
// a caching allocator (so a cudaMalloc outside it fails or forces the cache to
// be emptied), a runtime that must not add the implicit device
// synchronisation cudaMalloc/cudaFree can bring, or code that runs under a
// fixed, pre-reserved memory budget.  This entry point allocates nothing: the
// same data live in one file-scope __device__ array of fixed size (below),
// which the CUDA module loader places in every GPU that loads this library and
// which stays there until the process exits.  The reduction itself is the
// unchanged rs_fused kernel, so the results are bit-identical to
// tide_rs_reduce.
//
// Sharing rules: every call on a device uses the same array, and the array
// keeps whatever the last call left in it.  The host remembers, per device,
// which plan's work list the array holds and which gradient and shard
// pointers its tables were built from; a call uploads only what differs
// (nothing, when a plan is called again on the same buffers, as FSDP2 does
// step after step).  The work counter of the kernel's dynamic item order
// lives in the array too: it is zeroed (cudaMemsetAsync, no allocation) when
// a plan's work list is uploaded, and every launch leaves it at zero.  Two
// calls whose work overlaps on the GPU (different streams, no ordering
// between them) race on the array; issue them on one stream or order them.
// A call on a stream that is being captured is refused: a captured launch
// would keep reading whatever a later call leaves in the array.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "tide_internal.h"

namespace tide {
namespace {

// Largest static scratch: work items (32 bytes each), the caller's pointer
// array, the transposed gradient table, the shard table and the phase flags.
// The five measured workloads need at most 5.3 MiB (wan22dit: 172,166 items
// of 32 bytes are 5.25 MiB of it).
constexpr size_t kNoallocScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// One lock per device guards that device's record below, so callers on
// different devices never wait for one another; callers on one device are
// serialised, including the waits for their streams that the uploads from
// pageable memory can bring.
std::mutex g_device_mutex[kMaxDevices];
unsigned char* g_scratch_addr[kMaxDevices] = {};

// What the array on a device holds: the plan whose work list and counter are
// in place (0: unknown), and the pointer arrays its tables were built from.
struct DeviceRecord {
  uint64_t plan_uid = 0;
  std::vector<const void*> grads;
  std::vector<const void*> shards;
};
DeviceRecord g_record[kMaxDevices];

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The caller passes gradient pointers rank-major ([r][p]); the kernel reads
// them parameter-major ([p][r]).  Also flags each parameter whose N gradients
// share one address phase mod 16 (the kernel's 16-byte load path).
__global__ void noalloc_tables_kernel(const uint16_t* const* grads_rp, int N, int P, const uint16_t** gtab,
                                      uint8_t* flags) {
  const int64_t total = (int64_t)N * P;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t p = i / N, r = i % N;
    gtab[i] = grads_rp[r * P + p];
  }
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < P; p += stride) {
    const uintptr_t phase0 = (uintptr_t)grads_rp[p] & 15;
    uint8_t uniform = 1;
    for (int r = 1; r < N; ++r)
      if (((uintptr_t)grads_rp[(int64_t)r * P + p] & 15) != phase0) uniform = 0;
    flags[p] = uniform;
  }
}

tide_status cuda_status(cudaError_t err, const char* what) {
  return fail(err == cudaErrorMemoryAllocation ? TIDE_ERR_OUT_OF_MEMORY : TIDE_ERR_CUDA,
              std::string(what) + ": " + cudaGetErrorString(err));
}

}  // namespace
}  // namespace tide

using namespace tide;

extern "C" tide_status tide_rs_reduce_noalloc(const tide_plan* pl, const void* const* grads, float* const* shards,
                                              void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  pl->last_launches = 0;
  if (pl->rs_items.empty()) return TIDE_OK;
  const tide_status st = check_rs_call(pl, grads, shards, nullptr);
  if (st != TIDE_OK) return st;

  // Scratch layout: items | caller's [r][p] pointers | [p][r] table | shards | flags | work counter.
  const size_t n_ptr = (size_t)pl->N * pl->P;
  const size_t items_bytes = pl->rs_items.size() * sizeof(RsItem);
  const size_t off_grads_rp = align256(items_bytes);
  const size_t off_gtab = align256(off_grads_rp + 8 * n_ptr);
  const size_t off_shards = align256(off_gtab + 8 * n_ptr);
  const size_t off_flags = align256(off_shards + 8 * (size_t)pl->N);
  const size_t off_counter = align256(off_flags + (size_t)pl->P);
  const size_t need = off_counter + 8;
  if (need > kNoallocScratchBytes)
    return fail(TIDE_ERR_INVALID_ARG, "this group needs " + std::to_string(need) +
                                          " bytes of static scratch; tide_rs_reduce_noalloc is limited to " +
                                          std::to_string(kNoallocScratchBytes) + " bytes (use tide_rs_reduce)");

  cudaStream_t s = (cudaStream_t)stream;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t err = cudaStreamIsCapturing(s, &cap);
  if (err != cudaSuccess) return cuda_status(err, "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone)
    return fail(TIDE_ERR_INVALID_ARG,
                "tide_rs_reduce_noalloc called on a stream under capture (its tables live in one shared array "
                "that later calls rewrite; use tide_rs_reduce in graphs)");

  int dev = -1;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_status(err, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(TIDE_ERR_INVALID_ARG, "device ordinal beyond 63");
  std::lock_guard<std::mutex> lock(g_device_mutex[dev]);
  if (!g_scratch_addr[dev]) {
    // First call on this device: where the module loader put the array on
    // this device (the address differs per device).
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (err != cudaSuccess) return cuda_status(err, "cudaGetSymbolAddress(static scratch)");
    g_scratch_addr[dev] = (unsigned char*)ptr;
  }
  unsigned char* const base = g_scratch_addr[dev];
  DeviceRecord& rec = g_record[dev];
  const std::vector<const void*> gv(grads, grads + n_ptr);
  const std::vector<const void*> sv((const void* const*)shards, (const void* const*)shards + pl->N);
  int launches = 0;
  // On any failure below the record is cleared, so the next call uploads everything.
  auto cuda_fail_rec = [&](cudaError_t e, const char* what) {
    rec = DeviceRecord();
    return cuda_status(e, what);
  };
  if (rec.plan_uid != pl->uid) {
    rec = DeviceRecord();
    if ((err = cudaMemcpyAsync(base, pl->rs_items.data(), items_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return cuda_fail_rec(err, "work-list upload");
    if ((err = cudaMemsetAsync(base + off_counter, 0, 8, s)) != cudaSuccess)
      return cuda_fail_rec(err, "work-counter reset");
    rec.plan_uid = pl->uid;
  }
  if (rec.grads != gv) {
    if ((err = cudaMemcpyAsync(base + off_grads_rp, grads, 8 * n_ptr, cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return cuda_fail_rec(err, "gradient pointer upload");
    const int tgrid = (int)std::min<int64_t>(1024, ((int64_t)n_ptr + 255) / 256);
    noalloc_tables_kernel<<<tgrid, 256, 0, s>>>((const uint16_t* const*)(base + off_grads_rp), pl->N, pl->P,
                                                 (const uint16_t**)(base + off_gtab), base + off_flags);
    if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail_rec(err, "pointer-table kernel launch");
    ++launches;
    rec.grads = gv;
  }
  if (rec.shards != sv) {
    if ((err = cudaMemcpyAsync(base + off_shards, shards, 8 * (size_t)pl->N, cudaMemcpyHostToDevice, s)) !=
        cudaSuccess)
      return cuda_fail_rec(err, "shard pointer upload");
    rec.shards = sv;
  }

  int sms = 0;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail_rec(err, "cudaDeviceGetAttribute");
  const int occ = rs_blocks_per_sm(pl->L);
  if (occ <= 0) {
    rec = DeviceRecord();
    return fail(TIDE_ERR_CUDA, "occupancy query failed");
  }

  RsArgs a;
  a.items = (const RsItem*)base;
  a.counter = (unsigned long long*)(base + off_counter);  // zero at launch; the kernel leaves it at zero
  a.n_items = (int64_t)pl->rs_items.size();
  a.grad_tab = (const uint16_t* const*)(base + off_gtab);
  a.shard_tab = (float* const*)(base + off_shards);
  a.uniform_phase = base + off_flags;
  a.N = pl->N;
  a.M = pl->M;
  a.L = pl->L;
  a.P = pl->P;
  a.S = pl->S;
  a.epilogue = pl->rs_epilogue;
  a.inbox = nullptr;
  a.slice_len = pl->S > 0 ? (pl->S + pl->L - 1) / pl->L : 0;
  std::memcpy(a.order, pl->order, sizeof(a.order));
  const int grid = (int)std::min<int64_t>((int64_t)sms * occ, a.n_items);
  const int lerr = launch_rs(a, grid, stream);
  if (lerr != cudaSuccess) return cuda_fail_rec((cudaError_t)lerr, "rs_fused launch");
  pl->last_launches = launches + 1;  // the table kernel when the tables changed, and rs_fused
  return TIDE_OK;
}

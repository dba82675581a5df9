// Compute entry points of libtide: device set-up of a plan, the per-call
// pointer-table upload through an event-guarded pinned ring, and the kernel
// launches on the caller's stream.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>

#include "tide_internal.h"

using namespace tide;

namespace {

tide_status cuda_fail(cudaError_t err, const char* what) {
  return fail(err == cudaErrorMemoryAllocation ? TIDE_ERR_OUT_OF_MEMORY : TIDE_ERR_CUDA,
              std::string(what) + ": " + cudaGetErrorString(err));
}

#define TIDE_CUDA(call, what)                          \
  do {                                                 \
    cudaError_t err_ = (call);                         \
    if (err_ != cudaSuccess) return cuda_fail(err_, what); \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bytes of one per-call pointer table: RS needs [P][N] gradient pointers, [N]
// shard pointers, [P] phase flags and its 8-byte work counter; AG needs [N]
// shard and [P] param pointers.
size_t rs_table_bytes(const tide_plan* pl) {
  return align_up((size_t)pl->P * pl->N * 8 + (size_t)pl->N * 8, 16) + align_up((size_t)pl->P, 16) + 16;
}
size_t ag_table_bytes(const tide_plan* pl) { return (size_t)pl->N * 8 + (size_t)pl->P * 8; }

void release_device_state(tide_plan* pl) {
  for (auto& s : pl->ring) {
    if (s.done) {
      if (s.in_flight) cudaEventSynchronize((cudaEvent_t)s.done);
      cudaEventDestroy((cudaEvent_t)s.done);
    }
    if (s.host) cudaFreeHost(s.host);
    if (s.dev) cudaFree(s.dev);
    s = tide_plan::Slot();
  }
  for (int k = 0; k < tide_plan::kTableKinds; ++k) pl->cached_slot[k] = -1;
  for (auto& s : pl->captured) {
    if (s.host) cudaFreeHost(s.host);
    if (s.dev) cudaFree(s.dev);
    s = tide_plan::Slot();
  }
  pl->n_captured = 0;
  if (pl->d_rs_items) cudaFree(pl->d_rs_items);
  if (pl->d_ag_items) cudaFree(pl->d_ag_items);
  if (pl->d_ag_units) cudaFree(pl->d_ag_units);
  for (int l = 0; l < kMaxL; ++l) {
    if (pl->d_rail_items[l]) cudaFree(pl->d_rail_items[l]);
    if (pl->d_rail_units[l]) cudaFree(pl->d_rail_units[l]);
    pl->d_rail_items[l] = nullptr;
    pl->d_rail_units[l] = nullptr;
    pl->rail_n_items[l] = pl->rail_n_units[l] = 0;
  }
  for (int d = 0; d < tide_plan::kMaxRounds; ++d) {
    for (void* q : {(void*)pl->d_rd_items[d], (void*)pl->d_rd_units[d], (void*)pl->d_rdr_items[d],
                    (void*)pl->d_rdr_units[d]})
      if (q) cudaFree(q);
    pl->d_rd_items[d] = pl->d_rdr_items[d] = nullptr;
    pl->d_rd_units[d] = pl->d_rdr_units[d] = nullptr;
    pl->rd_n_items[d] = pl->rd_n_units[d] = pl->rdr_n_items[d] = pl->rdr_n_units[d] = 0;
  }
  for (void* q : {(void*)pl->d_init_items, (void*)pl->d_init_units})
    if (q) cudaFree(q);
  pl->d_init_items = nullptr;
  pl->d_init_units = nullptr;
  pl->init_n_items = pl->init_units = 0;
  if (pl->d_status) cudaFree(pl->d_status);
  pl->d_status = nullptr;
  for (void* q : {(void*)pl->d_agu_items, (void*)pl->d_agu_units, (void*)pl->d_pack_items, (void*)pl->d_pack_units})
    if (q) cudaFree(q);
  for (void* q : {(void*)pl->d_agb_items, (void*)pl->d_agr_items, (void*)pl->d_agr_units})
    if (q) cudaFree(q);
  pl->d_agb_items = pl->d_agr_items = nullptr;
  pl->d_agr_units = nullptr;
  pl->agb_n_items = pl->agr_n_items = pl->agr_units = 0;
  pl->ag_bulk_ok = false;
  pl->d_agu_items = nullptr;
  pl->d_agu_units = nullptr;
  pl->d_pack_items = nullptr;
  pl->d_pack_units = nullptr;
  pl->agu_units = pl->pack_units = 0;
  pl->d_rs_items = nullptr;
  pl->d_ag_items = nullptr;
  pl->d_ag_units = nullptr;
  pl->device = -1;
}

// First compute call: bind the plan to the current device, upload its work
// lists and build the pointer-table ring.  Synchronous; allocates.
tide_status ensure_device(tide_plan* pl) {
  int dev = -1;
  TIDE_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (pl->device >= 0) {
    if (dev != pl->device)
      return fail(TIDE_ERR_DEVICE_MISMATCH, "plan was set up on device " + std::to_string(pl->device) +
                                                " but device " + std::to_string(dev) + " is current");
    return TIDE_OK;
  }
  pl->device = dev;
  tide_status st = TIDE_OK;
  auto bail = [&](cudaError_t err, const char* what) {
    st = cuda_fail(err, what);
    release_device_state(pl);
    return st;
  };
  cudaError_t err = cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return bail(err, "cudaDeviceGetAttribute");
  if (!pl->rs_items.empty()) {
    const size_t bytes = pl->rs_items.size() * sizeof(RsItem);
    if ((err = cudaMalloc(&pl->d_rs_items, bytes)) != cudaSuccess) return bail(err, "cudaMalloc(rs items)");
    if ((err = cudaMemcpy(pl->d_rs_items, pl->rs_items.data(), bytes, cudaMemcpyHostToDevice)) != cudaSuccess)
      return bail(err, "cudaMemcpy(rs items)");
  }
  if (!pl->ag_items.empty()) {
    const size_t bytes = pl->ag_items.size() * sizeof(AgItem);
    if ((err = cudaMalloc(&pl->d_ag_items, bytes)) != cudaSuccess) return bail(err, "cudaMalloc(ag items)");
    if ((err = cudaMemcpy(pl->d_ag_items, pl->ag_items.data(), bytes, cudaMemcpyHostToDevice)) != cudaSuccess)
      return bail(err, "cudaMemcpy(ag items)");
  }
  pl->slot_bytes = align_up(std::max(rs_table_bytes(pl), ag_table_bytes(pl)), 256);
  pl->table_scratch.assign(pl->slot_bytes, 0);
  for (auto& s : pl->ring) {
    if ((err = cudaHostAlloc((void**)&s.host, pl->slot_bytes, cudaHostAllocDefault)) != cudaSuccess)
      return bail(err, "cudaHostAlloc(pointer ring)");
    if ((err = cudaMalloc((void**)&s.dev, pl->slot_bytes)) != cudaSuccess) return bail(err, "cudaMalloc(pointer ring)");
    cudaEvent_t ev;
    if ((err = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
      return bail(err, "cudaEventCreate");
    s.done = ev;
  }
  for (auto& s : pl->captured) {
    if ((err = cudaHostAlloc((void**)&s.host, pl->slot_bytes, cudaHostAllocDefault)) != cudaSuccess)
      return bail(err, "cudaHostAlloc(captured tables)");
    if ((err = cudaMalloc((void**)&s.dev, pl->slot_bytes)) != cudaSuccess)
      return bail(err, "cudaMalloc(captured tables)");
    s.fixed = true;
  }
  if ((err = cudaMalloc(&pl->d_status, sizeof(int))) != cudaSuccess) return bail(err, "cudaMalloc(status)");
  if ((err = cudaMemset(pl->d_status, 0, sizeof(int))) != cudaSuccess) return bail(err, "cudaMemset(status)");
  if (pl->M <= 8) {
    // Bulk-copy pipeline (M <= 8 only): kBulkCtasPerSm CTAs per SM, each with
    // as many stages as its share of the SM's shared memory allows (a little
    // is left for the per-block reservation and the static allocations).
    // Independent pipelines per SM set the speed: one CTA of 8 consumer
    // warps with a 6-stage ring of 32 KiB reached 0.76-0.95 of the copy
    // bandwidth, two such CTAs with 3 stages each 0.99-1.04, four CTAs of 4
    // consumer warps with 3 stages of 16 KiB each 1.015-1.067 (kept); five
    // spill registers and are 3-4% slower.
    int optin = 0, per_sm = 0;
    if ((err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return bail(err, "cudaDeviceGetAttribute(smem)");
    if ((err = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
      return bail(err, "cudaDeviceGetAttribute(smem per SM)");
    const int budget = std::min(optin, per_sm / kBulkCtasPerSm - 1024) - 2048;
    pl->bulk = rs_bulk_layout(pl->N, pl->M, pl->L, budget);
    if (pl->bulk.smem_bytes > optin) {
      release_device_state(pl);
      return fail(TIDE_ERR_UNIMPLEMENTED, "device has too little shared memory for the bulk-copy pipeline");
    }
    if ((err = (cudaError_t)rs_bulk_setup(pl->L, pl->bulk.smem_bytes)) != cudaSuccess)
      return bail(err, "cudaFuncSetAttribute(rs_bulk)");
    const int bulk_occ = rs_bulk_blocks_per_sm(pl->L, pl->bulk.smem_bytes);
    if (bulk_occ <= 0) {
      release_device_state(pl);
      return fail(TIDE_ERR_CUDA, "occupancy query of the bulk-copy pipeline failed");
    }
    pl->bulk_grid = (int)std::min<int64_t>((int64_t)pl->num_sms * std::min(bulk_occ, kBulkCtasPerSm),
                                           std::max<int64_t>(1, pl->rs_items.size()));
  }
  const int rs_occ = rs_blocks_per_sm(pl->L);
  const int ag_occ = ag_blocks_per_sm();
  if (rs_occ <= 0 || ag_occ <= 0) {
    release_device_state(pl);
    return fail(TIDE_ERR_CUDA, "occupancy query failed (is this an sm_103 device?)");
  }
  pl->rs_grid = (int)std::min<int64_t>((int64_t)pl->num_sms * rs_occ, std::max<int64_t>(1, pl->rs_items.size()));
  // The all-gather's units are dealt to warps statically, so every SM gets
  // the same number of CTAs: with fewer CTAs than SMs x occupancy, SMs with
  // more CTAs give each warp less bandwidth and set the tail.  Warps left
  // without units exit at once.
  pl->ag_grid = pl->num_sms * ag_occ;
  // Equal-cost all-gather units: about 8 KiB each, at most 64 per warp (a sweep
  // of 4-32 KiB and 2-4 CTAs per SM on the four full-size workloads put the
  // best here).
  try {
    const std::vector<UnitStart> au = ag_unit_starts(pl, (int64_t)pl->ag_grid * (kAgThreads / 32), 8 << 10, 64);
    pl->ag_units = (int64_t)au.size() - 1;
    // Unpadded all-gather and Slot-Reuse packing lists.
    auto upload = [&](const std::vector<AgItem>& v, AgItem** d_items, UnitStart** d_units,
                      int64_t* n_units) -> cudaError_t {
      if (v.empty()) return cudaSuccess;
      const std::vector<UnitStart> u = ag_unit_starts_of(v, (int64_t)pl->ag_grid * (kAgThreads / 32), 8 << 10, 64);
      *n_units = (int64_t)u.size() - 1;
      cudaError_t e2 = cudaMalloc(d_items, v.size() * sizeof(AgItem));
      if (e2 == cudaSuccess) e2 = cudaMemcpy(*d_items, v.data(), v.size() * sizeof(AgItem), cudaMemcpyHostToDevice);
      if (e2 == cudaSuccess) e2 = cudaMalloc(d_units, u.size() * sizeof(UnitStart));
      if (e2 == cudaSuccess) e2 = cudaMemcpy(*d_units, u.data(), u.size() * sizeof(UnitStart), cudaMemcpyHostToDevice);
      return e2;
    };
    if ((err = upload(pl->ag_items_unpadded, &pl->d_agu_items, &pl->d_agu_units, &pl->agu_units)) != cudaSuccess)
      return bail(err, "uploading the unpadded all-gather list");
    if ((err = upload(pl->pack_items, &pl->d_pack_items, &pl->d_pack_units, &pl->pack_units)) != cudaSuccess)
      return bail(err, "uploading the Slot-Reuse packing list");
    // Per-rail item lists for tide_ag_stage_place.
    for (int l = 0; l < pl->L; ++l) {
      std::vector<AgItem> ri;
      for (const AgItem& it : pl->ag_items)
        if (it.r % pl->L == l) ri.push_back(it);
      pl->rail_n_items[l] = (int64_t)ri.size();
      if (ri.empty()) continue;
      const std::vector<UnitStart> ru = ag_unit_starts_of(ri, (int64_t)pl->ag_grid * (kAgThreads / 32), 8 << 10, 64);
      pl->rail_n_units[l] = (int64_t)ru.size() - 1;
      if ((err = cudaMalloc(&pl->d_rail_items[l], ri.size() * sizeof(AgItem))) != cudaSuccess)
        return bail(err, "cudaMalloc(rail items)");
      if ((err = cudaMemcpy(pl->d_rail_items[l], ri.data(), ri.size() * sizeof(AgItem), cudaMemcpyHostToDevice)) !=
          cudaSuccess)
        return bail(err, "cudaMemcpy(rail items)");
      if ((err = cudaMalloc(&pl->d_rail_units[l], ru.size() * sizeof(UnitStart))) != cudaSuccess)
        return bail(err, "cudaMalloc(rail units)");
      if ((err = cudaMemcpy(pl->d_rail_units[l], ru.data(), ru.size() * sizeof(UnitStart), cudaMemcpyHostToDevice)) !=
          cudaSuccess)
        return bail(err, "cudaMemcpy(rail units)");
    }
    // Recursive-doubling rounds for the SM exchange: in round d node n copies
    // the first c = min(2^d, M - 2^d) pieces of node (n + 2^d) mod M's stage
    // buffer to its own slots [2^d, 2^d + c), in 32768-element items.  The
    // lists count elements, so they serve both element sizes.
    const int32_t rounds = tide_rd_rounds(pl->M);
    for (int32_t d = 0; d < rounds && d < tide_plan::kMaxRounds && pl->S > 0; ++d) {
      const int64_t have = (int64_t)1 << d, c = tide_rd_send_count(pl->M, d);
      std::vector<AgItem> v;
      for (int32_t n = 0; n < pl->M; ++n)
        for (int64_t e = 0; e < c * pl->S; e += 32768)
          v.push_back(AgItem{e, have * pl->S + e, (int32_t)std::min<int64_t>(32768, c * pl->S - e), n,
                             (int32_t)((n + have) % pl->M), 0});
      pl->rd_n_items[d] = (int64_t)v.size();
      if ((err = upload(v, &pl->d_rd_items[d], &pl->d_rd_units[d], &pl->rd_n_units[d])) != cudaSuccess)
        return bail(err, "uploading the exchange rounds");
      // The same round on every rail: buffer l*M + n is rail l's node n.
      std::vector<AgItem> vr;
      vr.reserve(v.size() * pl->L);
      for (int32_t l = 0; l < pl->L; ++l)
        for (const AgItem& it : v) {
          AgItem x = it;
          x.p = l * pl->M + it.p;
          x.r = l * pl->M + it.r;
          vr.push_back(x);
        }
      pl->rdr_n_items[d] = (int64_t)vr.size();
      if ((err = upload(vr, &pl->d_rdr_items[d], &pl->d_rdr_units[d], &pl->rdr_n_units[d])) != cudaSuccess)
        return bail(err, "uploading the exchange rounds of all rails");
    }
    // Stage init: rank r = n*L + l's shard to slot 0 of stage buffer l*M + n.
    if (pl->S > 0) {
      std::vector<AgItem> v;
      for (int32_t r = 0; r < pl->N; ++r)
        for (int64_t e = 0; e < pl->S; e += 32768)
          v.push_back(AgItem{e, e, (int32_t)std::min<int64_t>(32768, pl->S - e), (r % pl->L) * pl->M + r / pl->L, r, 0});
      pl->init_n_items = (int64_t)v.size();
      if ((err = upload(v, &pl->d_init_items, &pl->d_init_units, &pl->init_units)) != cudaSuccess)
        return bail(err, "uploading the stage-init list");
    }
    // Bulk-copy all-gather lists, for bf16 and 16-byte aligned base pointers.
    {
      int optin = 0;
      if ((err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return bail(err, "cudaDeviceGetAttribute(smem)");
      pl->ag_bulk_ok = optin >= ag_bulk_smem_bytes();
      if (pl->ag_bulk_ok && (err = (cudaError_t)ag_bulk_setup()) != cudaSuccess)
        return bail(err, "cudaFuncSetAttribute(ag_bulk)");
    }
    if (pl->ag_bulk_ok) {
      const std::vector<AgItem>& bulk = pl->ag_bulk_items;
      pl->agb_n_items = (int64_t)bulk.size();
      pl->agr_n_items = (int64_t)pl->ag_rest_items.size();
      if (!bulk.empty()) {
        if ((err = cudaMalloc(&pl->d_agb_items, bulk.size() * sizeof(AgItem))) != cudaSuccess)
          return bail(err, "cudaMalloc(bulk all-gather items)");
        if ((err = cudaMemcpy(pl->d_agb_items, bulk.data(), bulk.size() * sizeof(AgItem),
                              cudaMemcpyHostToDevice)) != cudaSuccess)
          return bail(err, "cudaMemcpy(bulk all-gather items)");
      }
      if ((err = upload(pl->ag_rest_items, &pl->d_agr_items, &pl->d_agr_units, &pl->agr_units)) != cudaSuccess)
        return bail(err, "uploading the bulk all-gather's remainder");
    }
    if ((err = cudaMalloc(&pl->d_ag_units, au.size() * sizeof(UnitStart))) != cudaSuccess)
      return bail(err, "cudaMalloc(ag units)");
    if ((err = cudaMemcpy(pl->d_ag_units, au.data(), au.size() * sizeof(UnitStart), cudaMemcpyHostToDevice)) !=
        cudaSuccess)
      return bail(err, "cudaMemcpy(ag units)");
  } catch (const std::bad_alloc&) {
    release_device_state(pl);
    return fail(TIDE_ERR_OUT_OF_MEMORY, "host allocation failed while building work units");
  }
  return TIDE_OK;
}

// Claim the next ring slot, waiting for the call that used it last.
tide_status acquire_slot(tide_plan* pl, tide_plan::Slot** out) {
  tide_plan::Slot& s = pl->ring[pl->next_slot];
  if (s.in_flight) {
    TIDE_CUDA(cudaEventSynchronize((cudaEvent_t)s.done), "waiting for a pointer-table slot");
    s.in_flight = false;
  }
  pl->next_slot = (pl->next_slot + 1) % tide_plan::kRing;
  *out = &s;
  return TIDE_OK;
}

enum TableKind { TABLE_RS = 0, TABLE_AG = 1, TABLE_PACK = 2, TABLE_STAGE = 3, TABLE_RD = 4, TABLE_RDR = 5, TABLE_INIT = 6 };

// Puts the pointer table just built in pl->table_scratch (its first `bytes`)
// on the device.  If the previous table of this kind is byte-for-byte the
// same, its slot has not taken other content since, and its last use was on
// this stream (stream order) or has finished, that device copy is used as it
// is: persistent buffers cost no upload per call.  Otherwise the next ring
// slot is taken (waiting for its last use) and the table uploaded.  A reused
// RS table is valid because the kernels leave their work counter at zero.
tide_status commit_table(tide_plan* pl, TableKind kind, size_t bytes, cudaStream_t stream, tide_plan::Slot** out) {
  const unsigned char* tab = pl->table_scratch.data();
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  TIDE_CUDA(cudaStreamIsCapturing(stream, &cap), "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone) {
    // Graph capture: no event queries or waits (not capturable); the table
    // goes to a slot of its own and the upload becomes a node of the graph.
    if (cap != cudaStreamCaptureStatusActive) return fail(TIDE_ERR_CUDA, "stream capture was invalidated");
    if (pl->n_captured == tide_plan::kCaptureSlots)
      return fail(TIDE_ERR_INVALID_ARG, "more than " + std::to_string(tide_plan::kCaptureSlots) +
                                            " calls of this plan captured into CUDA graphs");
    tide_plan::Slot* s = &pl->captured[pl->n_captured++];
    std::memcpy(s->host, tab, bytes);
    TIDE_CUDA(cudaMemcpyAsync(s->dev, s->host, bytes, cudaMemcpyHostToDevice, stream), "pointer-table upload");
    s->bytes = bytes;
    *out = s;
    return TIDE_OK;
  }
  const int c = pl->cached_slot[kind];
  if (c >= 0) {
    tide_plan::Slot& s = pl->ring[c];
    if (s.gen == pl->cached_gen[kind] && s.bytes == bytes && std::memcmp(s.host, tab, bytes) == 0) {
      bool usable = !s.in_flight || s.stream == (void*)stream;
      if (!usable) {
        const cudaError_t q = cudaEventQuery((cudaEvent_t)s.done);
        if (q == cudaSuccess) {
          s.in_flight = false;
          usable = true;
        } else if (q != cudaErrorNotReady) {
          return cuda_fail(q, "cudaEventQuery(pointer-table slot)");
        }
      }
      if (usable) {
        s.stream = (void*)stream;
        *out = &s;
        return TIDE_OK;
      }
    }
  }
  tide_plan::Slot* s = nullptr;
  tide_status st = acquire_slot(pl, &s);
  if (st != TIDE_OK) return st;
  std::memcpy(s->host, tab, bytes);
  TIDE_CUDA(cudaMemcpyAsync(s->dev, s->host, bytes, cudaMemcpyHostToDevice, stream), "pointer-table upload");
  s->gen = ++pl->next_gen;
  s->bytes = bytes;
  s->stream = (void*)stream;
  pl->cached_slot[kind] = (int)(s - pl->ring);
  pl->cached_gen[kind] = s->gen;
  *out = s;
  return TIDE_OK;
}

tide_status finish(tide_plan::Slot* s, int launch_err, cudaStream_t stream, const char* what) {
  if (launch_err != cudaSuccess) return cuda_fail((cudaError_t)launch_err, what);
  if (s->fixed) return TIDE_OK;  // captured: the slot is never recycled
  TIDE_CUDA(cudaEventRecord((cudaEvent_t)s->done, stream), "cudaEventRecord");
  s->in_flight = true;
  return TIDE_OK;
}

}  // namespace

extern "C" {

void tide_plan_destroy(tide_plan* pl) {
  if (!pl) return;
  if (pl->device >= 0) {
    int cur = -1;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    if (!have_cur || cur != pl->device) cudaSetDevice(pl->device);
    release_device_state(pl);
    if (have_cur && cur != pl->device) cudaSetDevice(cur);
  }
  delete pl;
}

tide_status tide_plan_set_option(tide_plan* pl, int32_t option, int64_t value) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  switch (option) {
    case TIDE_OPT_RS_KERNEL:
      if (value != 0 && value != 1) return fail(TIDE_ERR_INVALID_ARG, "TIDE_OPT_RS_KERNEL must be 0 or 1");
      pl->rs_kernel = (int32_t)value;
      return TIDE_OK;
    case TIDE_OPT_WAIT_LIMIT_NS:
      if (value <= 0) return fail(TIDE_ERR_INVALID_ARG, "TIDE_OPT_WAIT_LIMIT_NS must be positive");
      pl->wait_limit_ns = (uint64_t)value;
      return TIDE_OK;
    case TIDE_OPT_RS_AVERAGE:
    case TIDE_OPT_RS_ACCUMULATE: {
      if (value != 0 && value != 1) return fail(TIDE_ERR_INVALID_ARG, "option value must be 0 or 1");
      const int bit = option == TIDE_OPT_RS_AVERAGE ? 1 : 2;
      pl->rs_epilogue = value ? (pl->rs_epilogue | bit) : (pl->rs_epilogue & ~bit);
      return TIDE_OK;
    }
    case TIDE_OPT_AG_UNPADDED:
      if (value != 0 && value != 1) return fail(TIDE_ERR_INVALID_ARG, "TIDE_OPT_AG_UNPADDED must be 0 or 1");
      pl->ag_unpadded = value != 0;
      return TIDE_OK;
    case TIDE_OPT_SUM_ORDER:
      if (value != TIDE_SUM_LANDING && value != TIDE_SUM_RELATIVE)
        return fail(TIDE_ERR_INVALID_ARG, "TIDE_OPT_SUM_ORDER must be TIDE_SUM_LANDING or TIDE_SUM_RELATIVE");
      pl->sum_order = (int32_t)value;
      build_order_table(pl);  // read by every later call (passed by value at launch)
      return TIDE_OK;
    case TIDE_OPT_AG_TRANSPORT:
      if (value < TIDE_AG_SM || value > TIDE_AG_BULK)
        return fail(TIDE_ERR_INVALID_ARG, "TIDE_OPT_AG_TRANSPORT must be a tide_ag_transport");
      pl->ag_transport = (int32_t)value;
      return TIDE_OK;
    case TIDE_OPT_RD_EXCHANGE:
      if (value != 0 && value != 1) return fail(TIDE_ERR_INVALID_ARG, "TIDE_OPT_RD_EXCHANGE must be 0 or 1");
      pl->rd_exchange = (int32_t)value;
      return TIDE_OK;
    case TIDE_OPT_CHECK_OVERLAP:
      if (value != 0 && value != 1) return fail(TIDE_ERR_INVALID_ARG, "TIDE_OPT_CHECK_OVERLAP must be 0 or 1");
      pl->check_overlap = value != 0;
      return TIDE_OK;
    case TIDE_OPT_TEST_DROP_TILE:
      if (value < -1) return fail(TIDE_ERR_INVALID_ARG, "TIDE_OPT_TEST_DROP_TILE must be >= -1");
      pl->test_drop_tile = value;
      return TIDE_OK;
  }
  return fail(TIDE_ERR_INVALID_ARG, "unknown option " + std::to_string(option));
}

int32_t tide_plan_last_launches(const tide_plan* pl) { return pl ? pl->last_launches : -1; }

tide_status tide_debug_bounds_selftest(void) {
  clear_error();
  TIDE_CUDA((cudaError_t)ag_bounds_selftest(), "bounds self-test launch");
  TIDE_CUDA(cudaDeviceSynchronize(), "bounds self-test");
  return TIDE_OK;
}

int64_t tide_debug_bounds_violations(int32_t reset) {
#ifdef TIDE_CHECKED
  if (cudaDeviceSynchronize() != cudaSuccess) return -2;
  return (int64_t)rs_kernel_bounds(reset != 0) + rs_staged_bounds(reset != 0) + rs_bulk_bounds(reset != 0) +
         ag_kernel_bounds(reset != 0);
#else
  (void)reset;
  return -1;
#endif
}

tide_status tide_plan_check(tide_plan* pl) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  if (pl->device < 0 || !pl->d_status) return TIDE_OK;
  int cur = -1;
  TIDE_CUDA(cudaGetDevice(&cur), "cudaGetDevice");
  if (cur != pl->device) TIDE_CUDA(cudaSetDevice(pl->device), "cudaSetDevice");
  cudaError_t err = cudaDeviceSynchronize();
  int word = 0;
  if (err == cudaSuccess) err = cudaMemcpy(&word, pl->d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (err == cudaSuccess && word) err = cudaMemset(pl->d_status, 0, sizeof(int));
  if (cur != pl->device) cudaSetDevice(cur);
  if (err != cudaSuccess) return cuda_fail(err, "reading the plan's status word");
  if (word & TIDE_DEVICE_TIMEOUT)
    return fail(TIDE_ERR_TIMEOUT, "a kernel of this plan gave up a bounded wait; its outputs are undefined");
  return TIDE_OK;
}

}  // extern "C"

namespace {
// Validate a reduce-scatter call, set up the device on first use, fill and
// upload the call's pointer table, and return the kernel arguments.
// Byte ranges for TIDE_OPT_CHECK_OVERLAP.
void add_grad_ranges(const tide_plan* pl, const void* const* grads, std::vector<ByteRange>* v) {
  for (int32_t r = 0; r < pl->N; ++r)
    for (int32_t p = 0; p < pl->P; ++p) {
      const uintptr_t g = (uintptr_t)grads[(size_t)r * pl->P + p];
      v->push_back({g, g + (uintptr_t)(2 * pl->rows[p] * pl->Kp[p]), "grads", (int64_t)r * pl->P + p});
    }
}
void add_ranges(const void* const* ptrs, int32_t n, size_t bytes, const char* what, std::vector<ByteRange>* v) {
  for (int32_t i = 0; i < n; ++i) v->push_back({(uintptr_t)ptrs[i], (uintptr_t)ptrs[i] + bytes, what, i});
}
void add_param_ranges(const tide_plan* pl, void* const* params, int32_t eb, bool unpadded, std::vector<ByteRange>* v) {
  for (int32_t p = 0; p < pl->P; ++p) {
    const int64_t n = unpadded ? pl->rows[p] * pl->Kp[p] : (int64_t)pl->N * pl->e[p];
    v->push_back({(uintptr_t)params[p], (uintptr_t)params[p] + (uintptr_t)(n * eb), "params", p});
  }
}

// The constant stride of `count` buffers (buffer i at ptrs[0] + i*stride), if
// they have one of at least min_stride bytes that a strided copy can take;
// else 0.
int64_t constant_stride(const void* const* ptrs, int32_t count, int64_t min_stride) {
  if (count < 2) return 0;
  const int64_t stride = (int64_t)((intptr_t)ptrs[1] - (intptr_t)ptrs[0]);
  if (stride < min_stride) return 0;
  for (int32_t i = 2; i < count; ++i)
    if ((int64_t)((intptr_t)ptrs[i] - (intptr_t)ptrs[0]) != i * stride) return 0;
  int dev = -1, max_pitch = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&max_pitch, cudaDevAttrMaxPitch, dev) != cudaSuccess ||
      stride > max_pitch)
    return 0;
  return stride;
}

// Rows of at most this many bytes go as strided copies in the exchange (its
// rows are c whole shards); larger ones copy faster one by one.  Measured
// every rail at once on copy engines, stage buffers as rows of one buffer:
// uneven (rows of 4.5-9 MB) 3086 GB/s strided against 1925 one by one;
// wan22dit as 32 x 2 (rows of 11-176 MB) 3820 against 5028 all strided.
constexpr size_t kExchangeStridedMaxRow = size_t(16) << 20;

// One exchange round of one rail whose M stage buffers lie at stride T from
// `rail` (node n's buffer at rail + n*T), as two strided copies: nodes
// n < M - have take the first c pieces of node n + have, the last `have`
// nodes those of nodes 0 .. have - 1; every node writes slots
// [have, have + c) and reads slots [0, c) of another, so no byte is both read
// and written in the round.
cudaError_t rd_round_strided(unsigned char* rail, int64_t T, int32_t M, int32_t have, int32_t c, size_t piece,
                             cudaStream_t s) {
  const size_t w = (size_t)c * piece;
  cudaError_t e = cudaMemcpy2DAsync(rail + (size_t)have * piece, (size_t)T, rail + (size_t)have * T, (size_t)T, w,
                                    (size_t)(M - have), cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaMemcpy2DAsync(rail + (size_t)(M - have) * T + (size_t)have * piece, (size_t)T, rail, (size_t)T, w,
                           (size_t)have, cudaMemcpyDeviceToDevice, s);
}

}  // namespace

tide_status tide::check_rs_call(const tide_plan* pl, const void* const* grads, float* const* shards,
                                const float* inbox) {
  if (!grads || !shards) return fail(TIDE_ERR_INVALID_ARG, "grads or shards array is NULL");
  for (int32_t r = 0; r < pl->N; ++r) {
    if (!shards[r]) return fail(TIDE_ERR_INVALID_ARG, "shards[" + std::to_string(r) + "] is NULL");
    if ((uintptr_t)shards[r] & 3) return fail(TIDE_ERR_ALIGNMENT, "shard pointer not 4-byte aligned");
  }
  for (int32_t p = 0; p < pl->P; ++p) {
    if (pl->e[p] == 0) continue;
    for (int32_t r = 0; r < pl->N; ++r) {
      const void* g = grads[(size_t)r * pl->P + p];
      if (!g) return fail(TIDE_ERR_INVALID_ARG, "grads[" + std::to_string(r * pl->P + p) + "] is NULL");
      if ((uintptr_t)g & 1) return fail(TIDE_ERR_ALIGNMENT, "gradient pointer not 2-byte aligned");
    }
  }
  if (pl->check_overlap) {
    std::vector<ByteRange> in, out;
    add_grad_ranges(pl, grads, &in);
    add_ranges((const void* const*)shards, pl->N, (size_t)pl->S * 4, "shards", &out);
    if (inbox) out.push_back({(uintptr_t)inbox, (uintptr_t)(inbox + tide_plan_inbox_elems(pl)), "inbox", 0});
    return check_overlap(in, out);
  }
  return TIDE_OK;
}

namespace {

tide_status prepare_rs(tide_plan* pl, const void* const* grads, float* const* shards, void* stream, RsArgs* a,
                       tide_plan::Slot** out_slot, const float* inbox = nullptr) {
  tide_status st = check_rs_call(pl, grads, shards, inbox);
  if (st != TIDE_OK) return st;
  st = ensure_device(pl);
  if (st != TIDE_OK) return st;
  tide_plan::Slot* slot = nullptr;

  // Pointer table: [P][N] gradients, [N] shards, [P] phase flags, work counter.
  unsigned char* tab = pl->table_scratch.data();
  const size_t n_grad = (size_t)pl->P * pl->N;
  const uint16_t** gtab = (const uint16_t**)tab;
  float** stab = (float**)(tab + n_grad * 8);
  const size_t flags_at = align_up(n_grad * 8 + (size_t)pl->N * 8, 16);
  uint8_t* flags = tab + flags_at;
  std::memset(tab + n_grad * 8 + (size_t)pl->N * 8, 0, flags_at - (n_grad * 8 + (size_t)pl->N * 8));
  for (int32_t p = 0; p < pl->P; ++p) {
    const uintptr_t phase0 = (uintptr_t)grads[p] & 15;
    uint8_t uniform = 1;
    for (int32_t r = 0; r < pl->N; ++r) {
      const void* g = grads[(size_t)r * pl->P + p];
      gtab[(size_t)p * pl->N + r] = (const uint16_t*)g;
      if (((uintptr_t)g & 15) != phase0) uniform = 0;
    }
    flags[p] = uniform;
  }
  for (int32_t r = 0; r < pl->N; ++r) stab[r] = shards[r];
  const size_t counter_at = flags_at + align_up((size_t)pl->P, 16);
  std::memset(flags + pl->P, 0, counter_at + 8 - (flags_at + pl->P));  // pad bytes; work counter = 0
  const size_t bytes = counter_at + 8;
  if ((st = commit_table(pl, TABLE_RS, bytes, (cudaStream_t)stream, &slot)) != TIDE_OK) return st;

  a->items = pl->d_rs_items;
  a->n_items = (int64_t)pl->rs_items.size();
  a->counter = (unsigned long long*)(slot->dev + counter_at);
  a->grad_tab = (const uint16_t* const*)slot->dev;
  a->shard_tab = (float* const*)(slot->dev + n_grad * 8);
  a->uniform_phase = (const uint8_t*)(slot->dev + flags_at);
  a->N = pl->N;
  a->M = pl->M;
  a->L = pl->L;
  a->P = pl->P;
  a->S = pl->S;
  a->epilogue = pl->rs_epilogue;
  a->inbox = nullptr;
  a->slice_len = pl->S > 0 ? (pl->S + pl->L - 1) / pl->L : 0;
  std::memcpy(a->order, pl->order, sizeof(a->order));
  a->bulk = pl->bulk;
  a->bulk.status = pl->d_status;
  a->bulk.wait_limit_ns = pl->wait_limit_ns;
  a->bulk.test_drop_tile = pl->test_drop_tile;
  *out_slot = slot;
  return TIDE_OK;
}
}  // namespace

extern "C" {

tide_status tide_rs_reduce(tide_plan* pl, const void* const* grads, float* const* shards, void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  pl->last_launches = 0;
  if (pl->rs_items.empty()) return TIDE_OK;  // S == 0: nothing to write
  if (pl->rs_kernel == 1 && pl->M > 8)
    return fail(TIDE_ERR_UNIMPLEMENTED, "the bulk-copy kernel handles at most 8 nodes (TIDE_OPT_RS_KERNEL = 0 does)");
  RsArgs a;
  tide_plan::Slot* slot = nullptr;
  tide_status st = prepare_rs(pl, grads, shards, stream, &a, &slot);
  if (st != TIDE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  pl->last_launches = 1;
  if (pl->rs_kernel == 1) return finish(slot, launch_rs_bulk(a, pl->bulk_grid, stream), s, "rs_bulk launch");
  return finish(slot, launch_rs(a, pl->rs_grid, stream), s, "rs_fused launch");
}

int64_t tide_plan_inbox_elems(const tide_plan* pl) {
  if (!pl) return -1;
  if (pl->S == 0) return 0;
  const int64_t B = (pl->S + pl->L - 1) / pl->L;
  return (int64_t)pl->M * pl->L * pl->M * pl->L * B;
}

tide_status tide_rs_staged(tide_plan* pl, const void* const* grads, float* const* shards, float* inbox,
                           int32_t sum_ctas_per_rank, int32_t landing_ctas_per_rank, void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  pl->last_launches = 0;
  if (sum_ctas_per_rank < 0 || landing_ctas_per_rank < 0) return fail(TIDE_ERR_INVALID_ARG, "negative CTA count");
  if (pl->rs_items.empty()) return TIDE_OK;
  if (!inbox) return fail(TIDE_ERR_INVALID_ARG, "inbox is NULL");
  if ((uintptr_t)inbox & 3) return fail(TIDE_ERR_ALIGNMENT, "inbox not 4-byte aligned");
  RsArgs a;
  tide_plan::Slot* slot = nullptr;
  tide_status st = prepare_rs(pl, grads, shards, stream, &a, &slot, inbox);
  if (st != TIDE_OK) return st;
  a.inbox = inbox;
  const int64_t sum_grid =
      sum_ctas_per_rank > 0 ? std::min<int64_t>((int64_t)sum_ctas_per_rank * pl->N, 1 << 20) : pl->rs_grid;
  // Vector landing (16- or 8-byte accesses) when every slice starts on such a
  // boundary of the inbox and of each shard.
  int land_vec = 0;
  for (const int w : {4, 2}) {
    bool ok = a.slice_len % w == 0 && ((uintptr_t)inbox % (4 * w)) == 0;
    for (int32_t r = 0; ok && r < pl->N; ++r) ok = ((uintptr_t)shards[r] % (4 * w)) == 0;
    if (ok) {
      land_vec = w;
      break;
    }
  }
  const int land_per_sm = std::max(1, rs_land_blocks_per_sm(pl->M, pl->L, land_vec));  // resident landing CTAs per SM
  const int land_x =
      landing_ctas_per_rank > 0 ? landing_ctas_per_rank : std::max(1, pl->num_sms * land_per_sm / pl->N);
  const bool land_wide = land_vec != 0 && (int64_t)land_x * pl->N < 2 * (int64_t)pl->num_sms;
  // a summing grid below the full one that fits one wave at 2 CTAs per SM
  const bool sum_wide = sum_grid < pl->rs_grid && sum_grid <= 2 * (int64_t)pl->num_sms;
  pl->last_launches = 2;
  return finish(slot, launch_rs_staged(a, (int)sum_grid, sum_wide, land_x, land_vec, land_wide, stream), (cudaStream_t)stream, "rs_staged launch");
}

tide_status tide_ag_place(tide_plan* pl, const void* const* shards, void* const* params, int32_t elem_bytes,
                          void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  pl->last_launches = 0;
  if (elem_bytes != 2 && elem_bytes != 4) return fail(TIDE_ERR_INVALID_ARG, "elem_bytes must be 2 or 4");
  if (pl->ag_items.empty()) return TIDE_OK;
  if (!shards || !params) return fail(TIDE_ERR_INVALID_ARG, "shards or params array is NULL");
  for (int32_t r = 0; r < pl->N; ++r) {
    if (!shards[r]) return fail(TIDE_ERR_INVALID_ARG, "shards[" + std::to_string(r) + "] is NULL");
    if ((uintptr_t)shards[r] % elem_bytes) return fail(TIDE_ERR_ALIGNMENT, "shard pointer not element-aligned");
  }
  for (int32_t p = 0; p < pl->P; ++p) {
    if (pl->e[p] == 0) continue;
    if (!params[p]) return fail(TIDE_ERR_INVALID_ARG, "params[" + std::to_string(p) + "] is NULL");
    if ((uintptr_t)params[p] % elem_bytes) return fail(TIDE_ERR_ALIGNMENT, "param pointer not element-aligned");
  }
  if (pl->check_overlap) {
    std::vector<ByteRange> in, out;
    add_ranges(shards, pl->N, (size_t)pl->S * elem_bytes, "shards", &in);
    add_param_ranges(pl, params, elem_bytes, pl->ag_unpadded, &out);
    tide_status st = check_overlap(in, out);
    if (st != TIDE_OK) return st;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (pl->ag_transport == TIDE_AG_COPY_ENGINES) {
    // The pages' transport: copy-engine copies straight to the final
    // addresses; no kernel, no device state.  When the N shards lie at one
    // constant stride (rows of one buffer), parameter p's N pieces can go as
    // one strided copy: row r from shards[0] + r*stride + op to
    // params[p] + r*e_p.  That replaces N host calls by one, which is what
    // limits small pieces; pieces above kCeStridedMaxPiece go one by one, as
    // plain copies move large rows faster.  Measured with the shards as rows
    // of one buffer, against every piece on its own: qwen3moe 2.41 / 25.6 ms,
    // uneven 1.20 / 45.1 ms, wan22dit 0.74 / 3.30 ms, llama70b 0.67 / 0.76 ms
    // (its 17-58 MB pieces one by one; all strided it took 0.95 ms).
    constexpr size_t kCeStridedMaxPiece = size_t(4) << 20;
    const int64_t stride =
        pl->ag_unpadded ? 0 : constant_stride((const void* const*)shards, pl->N, pl->S * (int64_t)elem_bytes);
    const bool strided = stride > 0;
    for (int32_t p = 0; p < pl->P; ++p) {
      const size_t width = (size_t)pl->e[p] * elem_bytes;
      if (strided && width > 0 && width <= kCeStridedMaxPiece) {
        TIDE_CUDA(cudaMemcpy2DAsync(params[p], width, (const unsigned char*)shards[0] + (size_t)pl->o[p] * elem_bytes,
                                    (size_t)stride, width, (size_t)pl->N, cudaMemcpyDeviceToDevice, s),
                  "all-gather strided copy");
        continue;
      }
      for (int32_t r = 0; r < pl->N; ++r) {
        const int64_t n = pl->ag_unpadded ? std::min(pl->Rp[p], std::max<int64_t>(0, pl->rows[p] - r * pl->Rp[p])) *
                                                pl->Kp[p]
                                          : pl->e[p];
        if (n == 0) continue;
        TIDE_CUDA(cudaMemcpyAsync((unsigned char*)params[p] + (size_t)r * pl->e[p] * elem_bytes,
                                  (const unsigned char*)shards[r] + (size_t)pl->o[p] * elem_bytes,
                                  (size_t)n * elem_bytes, cudaMemcpyDeviceToDevice, s),
                  "all-gather piece copy");
      }
    }
    return TIDE_OK;
  }
  tide_status st = ensure_device(pl);
  if (st != TIDE_OK) return st;
  tide_plan::Slot* slot = nullptr;
  const void** stab = (const void**)pl->table_scratch.data();
  void** ptab = (void**)(pl->table_scratch.data() + (size_t)pl->N * 8);
  for (int32_t r = 0; r < pl->N; ++r) stab[r] = shards[r];
  for (int32_t p = 0; p < pl->P; ++p) ptab[p] = params[p];
  if ((st = commit_table(pl, TABLE_AG, ag_table_bytes(pl), s, &slot)) != TIDE_OK) return st;

  // Bulk copies need bf16, the padded layout and 16-byte aligned bases.
  bool bulk = pl->ag_transport == TIDE_AG_BULK && pl->ag_bulk_ok && elem_bytes == 2 && !pl->ag_unpadded;
  for (int32_t r = 0; bulk && r < pl->N; ++r) bulk = ((uintptr_t)shards[r] & 15) == 0;
  for (int32_t p = 0; bulk && p < pl->P; ++p) bulk = pl->e[p] == 0 || ((uintptr_t)params[p] & 15) == 0;
  if (bulk) {
    // Remainder (heads, tails, phase-mismatched pieces) on the SM kernel,
    // then the aligned middles by bulk copies; disjoint bytes, any order.
    if (pl->agr_n_items > 0) {
      AgArgs r;
      r.items = pl->d_agr_items;
      r.n_items = pl->agr_n_items;
      r.units = pl->d_agr_units;
      r.n_units = pl->agr_units;
      r.shard_tab = (const unsigned char* const*)slot->dev;
      r.param_tab = (unsigned char* const*)(slot->dev + (size_t)pl->N * 8);
      r.elem_bytes = 2;
      const int lerr = launch_ag(r, pl->ag_grid, stream);
      if (lerr != cudaSuccess) return cuda_fail((cudaError_t)lerr, "ag_place (remainder) launch");
      pl->last_launches = 1;
    }
    if (pl->agb_n_items == 0) return finish(slot, cudaSuccess, s, "bulk all-gather");
    AgBulkArgs b;
    b.items = pl->d_agb_items;
    b.n_items = pl->agb_n_items;
    b.shard_tab = (const unsigned char* const*)slot->dev;
    b.param_tab = (unsigned char* const*)(slot->dev + (size_t)pl->N * 8);
    b.status = pl->d_status;
    b.wait_limit_ns = pl->wait_limit_ns;
    b.test_drop_chunk = pl->test_drop_tile;
    const int grid = (int)std::min<int64_t>(pl->num_sms, pl->agb_n_items);
    ++pl->last_launches;
    return finish(slot, launch_ag_bulk(b, grid, stream), s, "bulk all-gather launch");
  }

  AgArgs a;
  if (pl->ag_unpadded) {
    a.items = pl->d_agu_items;
    a.n_items = (int64_t)pl->ag_items_unpadded.size();
    a.units = pl->d_agu_units;
    a.n_units = pl->agu_units;
  } else {
    a.items = pl->d_ag_items;
    a.n_items = (int64_t)pl->ag_items.size();
    a.units = pl->d_ag_units;
    a.n_units = pl->ag_units;
  }
  a.shard_tab = (const unsigned char* const*)slot->dev;
  a.param_tab = (unsigned char* const*)(slot->dev + (size_t)pl->N * 8);
  a.elem_bytes = elem_bytes;
  pl->last_launches = 1;
  return finish(slot, launch_ag(a, pl->ag_grid, stream), s, "ag_place launch");
}

tide_status tide_slot_pack(tide_plan* pl, const void* const* grads, void* const* slots, void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  pl->last_launches = 0;
  if (pl->pack_items.empty()) return TIDE_OK;
  if (!grads || !slots) return fail(TIDE_ERR_INVALID_ARG, "grads or slots array is NULL");
  for (int32_t r = 0; r < pl->N; ++r) {
    if (!slots[r]) return fail(TIDE_ERR_INVALID_ARG, "slots[" + std::to_string(r) + "] is NULL");
    if ((uintptr_t)slots[r] & 1) return fail(TIDE_ERR_ALIGNMENT, "slot pointer not 2-byte aligned");
    for (int32_t p = 0; p < pl->P; ++p) {
      if (pl->rows[p] * pl->Kp[p] == 0) continue;
      const void* g = grads[(size_t)r * pl->P + p];
      if (!g) return fail(TIDE_ERR_INVALID_ARG, "grads[" + std::to_string(r * pl->P + p) + "] is NULL");
      if ((uintptr_t)g & 1) return fail(TIDE_ERR_ALIGNMENT, "gradient pointer not 2-byte aligned");
    }
  }
  if (pl->check_overlap) {
    std::vector<ByteRange> in, out;
    add_grad_ranges(pl, grads, &in);
    add_ranges((const void* const*)slots, pl->N, (size_t)2 * pl->N * pl->S, "slots", &out);
    tide_status st = check_overlap(in, out);
    if (st != TIDE_OK) return st;
  }
  tide_status st = ensure_device(pl);
  if (st != TIDE_OK) return st;
  tide_plan::Slot* slot = nullptr;
  const size_t n_grad = (size_t)pl->N * pl->P;
  const void** gtab = (const void**)pl->table_scratch.data();  // indexed by r*P + p
  void** stab = (void**)(pl->table_scratch.data() + n_grad * 8);
  for (size_t i = 0; i < n_grad; ++i) gtab[i] = grads[i];
  for (int32_t r = 0; r < pl->N; ++r) stab[r] = slots[r];
  cudaStream_t s = (cudaStream_t)stream;
  if ((st = commit_table(pl, TABLE_PACK, (n_grad + (size_t)pl->N) * 8, s, &slot)) != TIDE_OK) return st;
  AgArgs a;
  a.items = pl->d_pack_items;
  a.n_items = (int64_t)pl->pack_items.size();
  a.units = pl->d_pack_units;
  a.n_units = pl->pack_units;
  a.shard_tab = (const unsigned char* const*)slot->dev;
  a.param_tab = (unsigned char* const*)(slot->dev + n_grad * 8);
  a.elem_bytes = 2;
  pl->last_launches = 1;
  return finish(slot, launch_ag(a, pl->ag_grid, stream), s, "slot pack launch");
}

tide_status tide_rs_reduce_slots(tide_plan* pl, const void* const* slots, float* const* shards, void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  if (!slots) return fail(TIDE_ERR_INVALID_ARG, "slots array is NULL");
  for (int32_t r = 0; r < pl->N; ++r) {
    if (!slots[r]) return fail(TIDE_ERR_INVALID_ARG, "slots[" + std::to_string(r) + "] is NULL");
    for (int32_t p = 0; p < pl->P; ++p)
      pl->slot_grads[(size_t)r * pl->P + p] = (const unsigned char*)slots[r] + (size_t)2 * pl->N * pl->o[p];
  }
  return tide_rs_reduce(pl, pl->slot_grads.data(), shards, stream);
}

tide_status tide_ag_rd_exchange(tide_plan* pl, void* const* stages, int32_t elem_bytes, void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  pl->last_launches = 0;
  if (elem_bytes != 2 && elem_bytes != 4) return fail(TIDE_ERR_INVALID_ARG, "elem_bytes must be 2 or 4");
  if (pl->S == 0 || pl->M == 1) return TIDE_OK;
  if (!stages) return fail(TIDE_ERR_INVALID_ARG, "stages array is NULL");
  for (int32_t n = 0; n < pl->M; ++n) {
    if (!stages[n]) return fail(TIDE_ERR_INVALID_ARG, "stages[" + std::to_string(n) + "] is NULL");
    for (int32_t m = 0; m < n; ++m)
      if (stages[m] == stages[n]) return fail(TIDE_ERR_INVALID_ARG, "two nodes share a stage buffer");
  }
  const size_t piece = (size_t)pl->S * elem_bytes;
  cudaStream_t s = (cudaStream_t)stream;
  const int32_t rounds = tide_rd_rounds(pl->M);
  if (pl->rd_exchange == 1) {
    // SM kernel: one all-gather launch per round over that round's M copies
    // (rounds stay in stream order; within a round node n reads slots below
    // 2^d of another buffer and writes slots from 2^d up of its own).
    tide_status st = ensure_device(pl);
    if (st != TIDE_OK) return st;
    if (rounds > tide_plan::kMaxRounds) return fail(TIDE_ERR_UNIMPLEMENTED, "more than 5 exchange rounds");
    void** tab = (void**)pl->table_scratch.data();
    for (int32_t n = 0; n < pl->M; ++n) tab[n] = stages[n];
    tide_plan::Slot* slot = nullptr;
    if ((st = commit_table(pl, TABLE_RD, (size_t)pl->M * 8, s, &slot)) != TIDE_OK) return st;
    for (int32_t d = 0; d < rounds; ++d) {
      AgArgs a;
      a.items = pl->d_rd_items[d];
      a.n_items = pl->rd_n_items[d];
      a.units = pl->d_rd_units[d];
      a.n_units = pl->rd_n_units[d];
      a.shard_tab = (const unsigned char* const*)slot->dev;
      a.param_tab = (unsigned char* const*)slot->dev;
      a.elem_bytes = elem_bytes;
      const int lerr = launch_ag(a, pl->ag_grid, stream);
      ++pl->last_launches;
      if (d + 1 < rounds && lerr != cudaSuccess) return cuda_fail((cudaError_t)lerr, "exchange launch");
      if (d + 1 == rounds) return finish(slot, lerr, s, "exchange launch");
    }
    return TIDE_OK;
  }
  // stage buffers at one stride: two strided copies per round (rows up to 16 MiB)
  const int64_t T = constant_stride((const void* const*)stages, pl->M, (int64_t)pl->M * (int64_t)piece);
  for (int32_t d = 0; d < rounds; ++d) {
    const int32_t have = 1 << d;                     // pieces every node holds before round d
    const int32_t c = tide_rd_send_count(pl->M, d);  // pieces sent this round
    if (T > 0 && (size_t)c * piece <= kExchangeStridedMaxRow) {
      TIDE_CUDA(rd_round_strided((unsigned char*)stages[0], T, pl->M, have, c, piece, s), "exchange strided copy");
      continue;
    }
    for (int32_t n = 0; n < pl->M; ++n) {
      const unsigned char* from = (const unsigned char*)stages[(n + have) % pl->M];
      unsigned char* to = (unsigned char*)stages[n] + (size_t)have * piece;
      TIDE_CUDA(cudaMemcpyAsync(to, from, (size_t)c * piece, cudaMemcpyDeviceToDevice, s), "exchange copy");
    }
  }
  return TIDE_OK;
}

tide_status tide_ag_rd_exchange_rails(tide_plan* pl, void* const* stages, int32_t elem_bytes, void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  pl->last_launches = 0;
  if (elem_bytes != 2 && elem_bytes != 4) return fail(TIDE_ERR_INVALID_ARG, "elem_bytes must be 2 or 4");
  if (pl->S == 0 || pl->M == 1) return TIDE_OK;
  if (!stages) return fail(TIDE_ERR_INVALID_ARG, "stages array is NULL");
  const int32_t nb = pl->L * pl->M;
  const size_t piece = (size_t)pl->S * elem_bytes;
  for (int32_t i = 0; i < nb; ++i) {
    if (!stages[i]) return fail(TIDE_ERR_INVALID_ARG, "stages[" + std::to_string(i) + "] is NULL");
    if ((uintptr_t)stages[i] % elem_bytes) return fail(TIDE_ERR_ALIGNMENT, "stage pointer not element-aligned");
    for (int32_t j = 0; j < i; ++j)
      if (stages[j] == stages[i]) return fail(TIDE_ERR_INVALID_ARG, "two stage buffers are the same");
  }
  if (pl->check_overlap) {
    std::vector<ByteRange> in, out;
    add_ranges((const void* const*)stages, nb, (size_t)pl->M * piece, "stages", &out);
    tide_status st = check_overlap(in, out);
    if (st != TIDE_OK) return st;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int32_t rounds = tide_rd_rounds(pl->M);
  if (pl->rd_exchange == 1) {
    // SM kernel: one launch per round covers the rounds' copies of every rail.
    tide_status st = ensure_device(pl);
    if (st != TIDE_OK) return st;
    if (rounds > tide_plan::kMaxRounds) return fail(TIDE_ERR_UNIMPLEMENTED, "more than 5 exchange rounds");
    void** tab = (void**)pl->table_scratch.data();
    for (int32_t i = 0; i < nb; ++i) tab[i] = stages[i];
    tide_plan::Slot* slot = nullptr;
    if ((st = commit_table(pl, TABLE_RDR, (size_t)nb * 8, s, &slot)) != TIDE_OK) return st;
    for (int32_t d = 0; d < rounds; ++d) {
      AgArgs a;
      a.items = pl->d_rdr_items[d];
      a.n_items = pl->rdr_n_items[d];
      a.units = pl->d_rdr_units[d];
      a.n_units = pl->rdr_n_units[d];
      a.shard_tab = (const unsigned char* const*)slot->dev;
      a.param_tab = (unsigned char* const*)slot->dev;
      a.elem_bytes = elem_bytes;
      const int lerr = launch_ag(a, pl->ag_grid, stream);
      ++pl->last_launches;
      if (d + 1 < rounds && lerr != cudaSuccess) return cuda_fail((cudaError_t)lerr, "exchange launch");
      if (d + 1 == rounds) return finish(slot, lerr, s, "exchange launch");
    }
    return TIDE_OK;
  }
  // all L*M stage buffers at one stride: two strided copies per rail and round
  // (rows up to 16 MiB)
  const int64_t T = constant_stride((const void* const*)stages, nb, (int64_t)pl->M * (int64_t)piece);
  for (int32_t d = 0; d < rounds; ++d) {
    const int32_t have = 1 << d;
    const int32_t c = tide_rd_send_count(pl->M, d);
    if (T > 0 && (size_t)c * piece <= kExchangeStridedMaxRow) {
      for (int32_t l = 0; l < pl->L; ++l)
        TIDE_CUDA(rd_round_strided((unsigned char*)stages[0] + (size_t)l * pl->M * T, T, pl->M, have, c, piece, s),
                  "exchange strided copy");
      continue;
    }
    for (int32_t l = 0; l < pl->L; ++l)
      for (int32_t n = 0; n < pl->M; ++n) {
        const unsigned char* from = (const unsigned char*)stages[l * pl->M + (n + have) % pl->M];
        unsigned char* to = (unsigned char*)stages[l * pl->M + n] + (size_t)have * piece;
        TIDE_CUDA(cudaMemcpyAsync(to, from, (size_t)c * piece, cudaMemcpyDeviceToDevice, s), "exchange copy");
      }
  }
  return TIDE_OK;
}

tide_status tide_ag_stage_init(tide_plan* pl, const void* const* shards, void* const* stages, int32_t elem_bytes,
                               void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  pl->last_launches = 0;
  if (elem_bytes != 2 && elem_bytes != 4) return fail(TIDE_ERR_INVALID_ARG, "elem_bytes must be 2 or 4");
  if (pl->S == 0) return TIDE_OK;
  if (!shards || !stages) return fail(TIDE_ERR_INVALID_ARG, "shards or stages array is NULL");
  for (int32_t r = 0; r < pl->N; ++r) {
    if (!shards[r]) return fail(TIDE_ERR_INVALID_ARG, "shards[" + std::to_string(r) + "] is NULL");
    if ((uintptr_t)shards[r] % elem_bytes) return fail(TIDE_ERR_ALIGNMENT, "shard pointer not element-aligned");
    if (!stages[r]) return fail(TIDE_ERR_INVALID_ARG, "stages[" + std::to_string(r) + "] is NULL");
    if ((uintptr_t)stages[r] % elem_bytes) return fail(TIDE_ERR_ALIGNMENT, "stage pointer not element-aligned");
  }
  if (pl->check_overlap) {
    std::vector<ByteRange> in, out;
    add_ranges(shards, pl->N, (size_t)pl->S * elem_bytes, "shards", &in);
    add_ranges((const void* const*)stages, pl->N, (size_t)pl->S * elem_bytes, "stages", &out);
    tide_status st = check_overlap(in, out);
    if (st != TIDE_OK) return st;
  }
  tide_status st = ensure_device(pl);
  if (st != TIDE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const void** stab = (const void**)pl->table_scratch.data();
  void** dtab = (void**)(pl->table_scratch.data() + (size_t)pl->N * 8);
  for (int32_t r = 0; r < pl->N; ++r) {
    stab[r] = shards[r];
    dtab[r] = stages[r];
  }
  tide_plan::Slot* slot = nullptr;
  if ((st = commit_table(pl, TABLE_INIT, (size_t)pl->N * 16, s, &slot)) != TIDE_OK) return st;
  AgArgs a;
  a.items = pl->d_init_items;
  a.n_items = pl->init_n_items;
  a.units = pl->d_init_units;
  a.n_units = pl->init_units;
  a.shard_tab = (const unsigned char* const*)slot->dev;
  a.param_tab = (unsigned char* const*)(slot->dev + (size_t)pl->N * 8);
  a.elem_bytes = elem_bytes;
  pl->last_launches = 1;
  return finish(slot, launch_ag(a, pl->ag_grid, stream), s, "stage init launch");
}

tide_status tide_ag_stage_place(tide_plan* pl, const void* stage, int32_t node, int32_t rail, void* const* params,
                                int32_t elem_bytes, void* stream) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  pl->last_launches = 0;
  if (elem_bytes != 2 && elem_bytes != 4) return fail(TIDE_ERR_INVALID_ARG, "elem_bytes must be 2 or 4");
  if (node < 0 || node >= pl->M || rail < 0 || rail >= pl->L) return fail(TIDE_ERR_INVALID_ARG, "node or rail out of range");
  if (pl->ag_items.empty()) return TIDE_OK;
  if (!stage || !params) return fail(TIDE_ERR_INVALID_ARG, "stage or params is NULL");
  if ((uintptr_t)stage % elem_bytes) return fail(TIDE_ERR_ALIGNMENT, "stage pointer not element-aligned");
  for (int32_t p = 0; p < pl->P; ++p) {
    if (pl->e[p] == 0) continue;
    if (!params[p]) return fail(TIDE_ERR_INVALID_ARG, "params[" + std::to_string(p) + "] is NULL");
    if ((uintptr_t)params[p] % elem_bytes) return fail(TIDE_ERR_ALIGNMENT, "param pointer not element-aligned");
  }
  if (pl->check_overlap) {
    std::vector<ByteRange> in, out;
    in.push_back({(uintptr_t)stage, (uintptr_t)stage + (uintptr_t)pl->M * pl->S * elem_bytes, "stage", 0});
    add_param_ranges(pl, params, elem_bytes, false, &out);
    tide_status st = check_overlap(in, out);
    if (st != TIDE_OK) return st;
  }
  tide_status st = ensure_device(pl);
  if (st != TIDE_OK) return st;
  if (pl->rail_n_items[rail] == 0) return TIDE_OK;
  tide_plan::Slot* slot = nullptr;
  // Shard table indexed by rank: rank ((node + k) mod M) * L + rail reads slot k.
  const unsigned char** stab = (const unsigned char**)pl->table_scratch.data();
  void** ptab = (void**)(pl->table_scratch.data() + (size_t)pl->N * 8);
  for (int32_t r = 0; r < pl->N; ++r) stab[r] = nullptr;
  for (int32_t k = 0; k < pl->M; ++k) {
    const int32_t r = ((node + k) % pl->M) * pl->L + rail;
    stab[r] = (const unsigned char*)stage + (size_t)k * pl->S * elem_bytes;
  }
  for (int32_t p = 0; p < pl->P; ++p) ptab[p] = params[p];
  cudaStream_t s = (cudaStream_t)stream;
  if ((st = commit_table(pl, TABLE_STAGE, ag_table_bytes(pl), s, &slot)) != TIDE_OK) return st;
  AgArgs a;
  a.items = pl->d_rail_items[rail];
  a.n_items = pl->rail_n_items[rail];
  a.units = pl->d_rail_units[rail];
  a.n_units = pl->rail_n_units[rail];
  a.shard_tab = (const unsigned char* const*)slot->dev;
  a.param_tab = (unsigned char* const*)(slot->dev + (size_t)pl->N * 8);
  a.elem_bytes = elem_bytes;
  pl->last_launches = 1;
  return finish(slot, launch_ag(a, pl->ag_grid, stream), s, "ag_place (stage) launch");
}

}  // extern "C"

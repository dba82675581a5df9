// Internal definitions shared by the host plan builder and the CUDA kernels of
// libtide.  Nothing here is part of the public ABI (include/tide.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/tide.h"

namespace tide {

// Largest supported group: ranks and GPUs per NVSwitch domain.
constexpr int kMaxL = 8;                 // at most eight GPUs per domain
constexpr int kMaxM = 32;                // nodes (more than L: sources go in batches of L)
constexpr int kMaxN = kMaxL * kMaxM;     // ranks
constexpr int kMaxNdim = 8;

// Work-item kinds (RS_VALID / RS_PAD for the reduce-scatter list, AG for the
// all-gather list).
enum ItemKind : int16_t { RS_VALID = 0, RS_PAD = 1, AG_COPY = 2 };

// One contiguous range of one (parameter, destination rank) piece.  32 bytes,
// read once per CTA iteration.
struct RsItem {
  int64_t src_off;   // element offset inside every contributor's gradient of p
  int64_t dst_off;   // element offset inside destination rank r's packed shard
  int32_t n;         // elements in the range
  int32_t p;         // parameter
  int32_t r;         // destination rank
  int16_t slice;     // level-2 slice of the whole range (ranges never straddle one)
  int16_t kind;      // RS_VALID or RS_PAD
};
static_assert(sizeof(RsItem) == 32, "RsItem layout");

struct AgItem {
  int64_t src_off;   // element offset inside source rank r's packed shard
  int64_t dst_off;   // element offset inside parameter p's gathered block
  int32_t n;
  int32_t p;
  int32_t r;
  int32_t pad_;
};
static_assert(sizeof(AgItem) == 32, "AgItem layout");

// Work-list chunking.  A valid RS chunk covers at most rs_chunk_elems(N)
// elements and starts on a multiple of it in contributor-index space, so
// interior chunks are whole, 16-byte aligned runs of every contributor; padding
// chunks only write, so they are larger.  AG chunks are kAgChunkBytes / 2
// elements whatever the element size: 64 KiB of bf16 payload, 128 KiB when
// the all-gather moves 4-byte elements.
constexpr int kRsThreads = 256;
// An RS item reads 2*N bytes per element.  Items of about 128-256 KB of reads
// were fastest in a sweep of 1024-32768 elements on the four full-size
// workloads: larger ones leave a long tail when the last items finish, smaller
// ones pay the per-item set-up more often.  So the chunk is the power of two
// nearest below 128 Ki / N elements, kept within [2048, 8192].
inline int64_t rs_chunk_elems(int32_t N) {
  int64_t c = 8192;
  while (c > 2048 && c * N > (int64_t)1 << 17) c >>= 1;
  return c;
}
constexpr int64_t kRsPadChunk = 32768;
constexpr int kAgThreads = 256;
constexpr int64_t kAgChunkBytes = 65536;

// All-gather load balance.  Every item has a cost (a start-up charge for its
// descriptor and pointer loads, plus bytes moved per element) and the plan
// keeps the prefix sum of the costs.  When the plan is set up on a device it
// cuts the total cost into U = k*W equal units (W = warps of the grid),
// splitting items where a boundary falls inside one.  Warp w takes units
// w, w+W, w+2W, ...: every warp gets k units of equal cost, and at any moment
// neighbouring warps copy neighbouring parts of the item list, which keeps
// DRAM accesses in nearly address order.  (The reduce-scatter's items are
// already of near-equal cost -- rs_chunk_elems(N) elements -- and its CTAs
// take them from a shared counter.)
#if defined(__CUDACC__)
#define TIDE_HD __host__ __device__
#else
#define TIDE_HD
#endif
constexpr int64_t kAgItemCost = 2048;

TIDE_HD inline int64_t ag_item_cost(const AgItem& it) { return kAgItemCost + 4 * (int64_t)it.n; }

// First element of an item that a worker whose range starts `rel` cost units
// into the item copies, rounded up to 8 destination elements.
TIDE_HD inline int32_t ag_split(const AgItem& it, int64_t rel) {
  if (rel <= kAgItemCost) return 0;
  int64_t e = (rel - kAgItemCost + 3) / 4;
  e = (it.dst_off + e + 7) / 8 * 8 - it.dst_off;
  return (int32_t)(e < it.n ? e : it.n);
}

// Level-2 order table: order[(n_dest * L + s) * M + k] is the k-th source node
// whose partial is added for slice s of destination node n_dest.  The M
// entries run batch by batch (batches of L relative indices; every batch but
// the last is full), so a batch ends after every L entries and at the last.
constexpr int kOrderTableSize = kMaxM * kMaxL * kMaxM;

// Kernel argument blocks (passed by value as __grid_constant__).
// Start of a unit: item index and first element of that item.  Unit u spans
// [units[u], units[u+1]); units[n_units] = {n_items, 0}.
struct UnitStart {
  int32_t item;
  int32_t off;
};

// Bulk-copy pipeline of the reduce-scatter (rs_bulk.cu): tile geometry and
// shared-memory carve-up, fixed per plan when it is set up on a device.
constexpr int kMaxBulkStages = 16;
constexpr int kBulkCtasPerSm = 4;  // bulk-copy reduce-scatter pipelines per SM
constexpr int TIDE_DEVICE_TIMEOUT = 1;  // status-word bit: a kernel gave up waiting
struct BulkLayout {
  int32_t V;            // 8-element vectors per tile (128: 1024 outputs, 2 KiB windows)
  int32_t stage_bytes;  // 16 * L * V: one node's L windows of one tile
  int32_t stages;
  int32_t off_desc, off_bar, off_ctl, smem_bytes;
  int* status;              // plan's device status word
  uint64_t wait_limit_ns;   // bound on every wait
  int64_t test_drop_tile;   // stage fill whose data the producer withholds (tests); -1: none
};

struct RsArgs {
  const RsItem* items;
  int64_t n_items;
  unsigned long long* counter;      // next item to take: zero at launch, and the kernel leaves it
                                    // zero (see take_item)
  const uint16_t* const* grad_tab;  // [P][N]: contributor src's gradient of p
  float* const* shard_tab;          // [N]
  const uint8_t* uniform_phase;     // [P]: 1 if all N gradients of p share addr mod 16
  int32_t N, M, L, P;
  int64_t S;                        // packed shard length
  int32_t epilogue;                 // EPI_AVERAGE | EPI_ACCUMULATE (rs_device.cuh)
  float* inbox;                     // rs_staged only: [M][L][M][L * slice_len] partials
  int64_t slice_len;                // ceil(S / L)
  BulkLayout bulk;                  // rs_bulk only
  uint8_t order[kOrderTableSize];
};

// Bulk-copy all-gather (ag_bulk.cu): the aligned middles of the bf16 pieces
// in chunks of at most kAgBulkChunkElems elements.
constexpr int64_t kAgBulkChunkElems = 16384;
struct AgBulkArgs {
  const AgItem* items;              // chunks: 16-byte aligned at both ends
  int64_t n_items;
  const unsigned char* const* shard_tab;  // [N]
  unsigned char* const* param_tab;        // [P]
  int* status;                      // TIDE_DEVICE_TIMEOUT on a wait that ran out
  uint64_t wait_limit_ns;
  int64_t test_drop_chunk;          // chunk (counted per CTA) whose load is never issued (tests); -1: none
};

struct AgArgs {
  const AgItem* items;
  int64_t n_items;
  const UnitStart* units;           // [n_units + 1]
  int64_t n_units;
  const unsigned char* const* shard_tab;  // [N]
  unsigned char* const* param_tab;        // [P]
  int32_t elem_bytes;
};

// Launchers (rs_kernel.cu / ag_kernel.cu).  Return the cudaError_t as int.
int launch_rs(const RsArgs& args, int grid, void* stream);
int launch_ag(const AgArgs& args, int grid, void* stream);
int launch_ag_bulk(const AgBulkArgs& args, int grid, void* stream);
int ag_bulk_setup();       // raises the bulk all-gather's dynamic shared-memory limit
int ag_bulk_smem_bytes();
int launch_rs_bulk(const RsArgs& args, int grid, void* stream);
// land_vec: vector width of the landing, 4 or 2 floats (slice length a
// multiple of it, inbox and shards aligned to it), or 0 for 4-byte accesses;
// sum_wide / land_wide: the summing / landing grid cannot fill the GPU (more
// bytes in flight per thread).
int launch_rs_staged(const RsArgs& args, int sum_grid, bool sum_wide, int land_grid_x, int land_vec, bool land_wide,
                     void* stream);
int rs_land_blocks_per_sm(int M, int L, int vec);  // resident landing CTAs per SM (0 on error)
BulkLayout rs_bulk_layout(int N, int M, int L, int smem_budget);
int rs_bulk_setup(int L, int smem_bytes);  // raises the kernel's dynamic shared-memory limit
int rs_bulk_blocks_per_sm(int L, int smem_bytes);  // resident bulk CTAs per SM with that much shared memory
// Resident CTAs per SM of each kernel (occupancy), for grid sizing.
int rs_blocks_per_sm(int L);
// Store-check counters of the kernels' translation units (check.cuh); 0 in
// normal builds.
unsigned int rs_kernel_bounds(bool reset);
unsigned int rs_staged_bounds(bool reset);
unsigned int rs_bulk_bounds(bool reset);
unsigned int ag_kernel_bounds(bool reset);
int ag_bounds_selftest();  // one deliberate out-of-range check, no memory access
int ag_blocks_per_sm();

}  // namespace tide

// The opaque plan.
struct tide_plan {
  uint64_t uid = 0;  // unique per plan in this process, never reused (tide_rs_reduce_noalloc's cache key)
  int32_t N = 0, M = 0, L = 0, P = 0;
  std::vector<int64_t> rows, Kp, Rp, e, o;
  int64_t S = 0;
  std::vector<tide::RsItem> rs_items;
  std::vector<tide::AgItem> ag_items;
  std::vector<tide::AgItem> ag_items_unpadded;   // ag_items restricted to real rows
  // Bulk-copy all-gather split of ag_items (bf16, 16-byte aligned bases):
  // the aligned middles in chunks of at most kAgBulkChunkElems, and the rest.
  std::vector<tide::AgItem> ag_bulk_items, ag_rest_items;
  std::vector<tide::AgItem> pack_items;         // Slot-Reuse: r = grad index r*P+p, p = slot rank
  std::vector<const void*> slot_grads;          // tide_rs_reduce_slots' pointer array (host)
  std::vector<int64_t> ag_prefix;  // all-gather cost prefix sums (load balance)
  uint8_t order[tide::kOrderTableSize] = {};

  // Device state, created by the first compute call.
  int device = -1;
  int num_sms = 0;
  int rs_grid = 0, ag_grid = 0, bulk_grid = 0;
  int* d_status = nullptr;                 // device status word (TIDE_DEVICE_TIMEOUT)
  tide::BulkLayout bulk{};
  // Options (tide_plan_set_option).
  int32_t rs_kernel = 0;                   // 0: direct loads (rs_fused), 1: bulk-copy pipeline
  uint64_t wait_limit_ns = 2000000000ull;  // 2 s
  int64_t test_drop_tile = -1;
  int32_t rs_epilogue = 0;                 // averaging / accumulate bits
  int32_t sum_order = TIDE_SUM_LANDING;    // level-2 reading (order table)
  bool check_overlap = false;              // TIDE_OPT_CHECK_OVERLAP
  bool ag_unpadded = false;
  tide::RsItem* d_rs_items = nullptr;
  tide::AgItem* d_ag_items = nullptr;
  tide::UnitStart* d_ag_units = nullptr;
  int64_t ag_units = 0;
  // Unpadded all-gather and Slot-Reuse packing work lists and units.
  tide::AgItem* d_agu_items = nullptr;
  tide::UnitStart* d_agu_units = nullptr;
  int64_t agu_units = 0;
  tide::AgItem* d_pack_items = nullptr;
  tide::UnitStart* d_pack_units = nullptr;
  int64_t pack_units = 0;
  // Per-rail all-gather work (tide_ag_stage_place): rail l's items (ranks
  // r = n*L + l) and their equal-cost units.
  tide::AgItem* d_rail_items[tide::kMaxL] = {};
  tide::UnitStart* d_rail_units[tide::kMaxL] = {};
  int64_t rail_n_items[tide::kMaxL] = {};
  int64_t rail_n_units[tide::kMaxL] = {};
  // Recursive-doubling exchange on the SMs (TIDE_OPT_RD_EXCHANGE = 1): round
  // d's copies as all-gather items whose shard and parameter tables are both
  // the M stage buffers (r = source node, p = destination node).
  static constexpr int kMaxRounds = 5;  // ceil(log2 32)
  tide::AgItem* d_rd_items[kMaxRounds] = {};
  tide::UnitStart* d_rd_units[kMaxRounds] = {};
  int64_t rd_n_items[kMaxRounds] = {};
  int64_t rd_n_units[kMaxRounds] = {};
  // The same rounds for every rail at once (tide_ag_rd_exchange_rails): the
  // tables hold the L*M stage buffers, rail l's node n at l*M + n.
  tide::AgItem* d_rdr_items[kMaxRounds] = {};
  tide::UnitStart* d_rdr_units[kMaxRounds] = {};
  int64_t rdr_n_items[kMaxRounds] = {};
  int64_t rdr_n_units[kMaxRounds] = {};
  // tide_ag_stage_init: rank r's shard (r = n*L + l) to slot 0 of stage
  // buffer l*M + n.
  tide::AgItem* d_init_items = nullptr;
  tide::UnitStart* d_init_units = nullptr;
  int64_t init_n_items = 0;
  int64_t init_units = 0;
  int32_t rd_exchange = 0;                 // 0: copy engines, 1: SM kernel
  int32_t ag_transport = TIDE_AG_SM;       // TIDE_OPT_AG_TRANSPORT (tide_ag_transport)
  mutable int32_t last_launches = 0;       // kernels launched by the latest compute call
  // Bulk-copy all-gather lists (bf16, base pointers 16-byte aligned): chunks
  // of the pieces' aligned middles, and the rest (heads, tails, pieces whose
  // source and destination differ in phase) for ag_place_kernel.
  tide::AgItem* d_agb_items = nullptr;
  int64_t agb_n_items = 0;
  tide::AgItem* d_agr_items = nullptr;
  tide::UnitStart* d_agr_units = nullptr;
  int64_t agr_n_items = 0;
  int64_t agr_units = 0;
  bool ag_bulk_ok = false;                 // the device has the shared memory for it
  static constexpr int kRing = 8;
  struct Slot {
    unsigned char* host = nullptr;
    unsigned char* dev = nullptr;
    void* done = nullptr;   // cudaEvent_t
    bool in_flight = false;
    uint64_t gen = 0;        // bumped whenever the slot takes new content
    size_t bytes = 0;        // bytes of the last upload (host copy == device copy)
    void* stream = nullptr;  // stream of the slot's last use
    bool fixed = false;      // a captured call's table: never rewritten
  } ring[kRing];
  // Tables of calls made while their stream was being captured into a CUDA
  // graph: each keeps its slot until the plan is destroyed, so every replay
  // of the graph reads (and re-uploads) exactly the table of the capture.
  static constexpr int kCaptureSlots = 8;
  Slot captured[kCaptureSlots];
  int n_captured = 0;
  int next_slot = 0;
  size_t slot_bytes = 0;
  // Pointer tables are built in table_scratch; a call whose table equals the
  // previous one of its kind reuses that slot's device copy (no upload).
  static constexpr int kTableKinds = 7;  // RS, AG, Slot-Reuse pack, stage placement, exchange,
                                         // exchange of all rails, stage init
  std::vector<unsigned char> table_scratch;
  int cached_slot[kTableKinds] = {-1, -1, -1, -1, -1, -1, -1};
  uint64_t cached_gen[kTableKinds] = {};
  uint64_t next_gen = 0;
};

namespace tide {
// Equal-cost all-gather unit boundaries for W workers (plan.cpp); at most
// max_k units per worker, each worth about `target` cost units.
std::vector<UnitStart> ag_unit_starts(const tide_plan* pl, int64_t workers, int64_t target, int64_t max_k);
std::vector<UnitStart> ag_unit_starts_of(const std::vector<AgItem>& items, int64_t workers, int64_t target,
                                         int64_t max_k);
// Thread-local error reporting (plan.cpp).
tide_status fail(tide_status st, const std::string& msg);
void clear_error();
// Argument checks shared by every reduce-scatter entry point: null and
// misaligned pointers, and the overlap check when it is on (runtime.cu).
tide_status check_rs_call(const tide_plan* pl, const void* const* grads, float* const* shards, const float* inbox);
// Fills plan->order for the plan's sum_order (plan.cpp).
void build_order_table(tide_plan* pl);
// A byte range [lo, hi) a call reads or writes, named for error messages.
struct ByteRange {
  uintptr_t lo, hi;
  const char* what;
  int64_t index;
};
// INVALID_ARG if two outputs overlap or an output overlaps an input (inputs
// may overlap each other); empty ranges are ignored (plan.cpp).
tide_status check_overlap(const std::vector<ByteRange>& inputs, std::vector<ByteRange> outputs);
}  // namespace tide

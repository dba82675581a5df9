/*
 * tide.h -- C ABI of libtide: the per-element hot path of TIDE's layout-aware
 * FSDP2 collectives, emulated on one GPU with every rank's buffers resident in
 * that GPU's memory.
 *
 * Sources (three web pages about the TIDE preprint, arXiv 2610.38228):
 *   [Endgame]  "The Endgame of FSDP Communication: Layout-Aware Collectives on
 *              Copy Engines, RDMA, and NVSwitch"
 *   [Richland] "TIDE gives FSDP2 layout-aware zero-copy collectives: up to
 *              27.1% faster steps on 64 GPUs, zero-SM all-gather, bf16->fp32
 *              reduce-scatter"
 *   [Abstract] the preprint's abstract page, its figure captions and tables
 *
 * Notation ([Abstract] Table 2): M nodes, L GPUs per NVSwitch domain,
 * N = M*L ranks, rank r = n*L + l.  For parameter p of shape (R_p, d1, ...):
 *   Kp = d1*d2*...   (1 for a 1-D tensor; a 0-D tensor counts as [1])
 *   Rp = ceil(R_p / N), the padded per-rank row count; rank r owns global rows
 *        [r*Rp, (r+1)*Rp), and rows at or beyond R_p are zero padding
 *   e_p = Rp*Kp elements per rank ("sp" of Table 2, in elements)
 *   op  = e_0 + ... + e_{p-1}, the prefix offset inside a packed shard
 *   S   = sum of e_p, the packed shard length in elements.
 * The dim-0 chunk-and-pad rule and the gap-free prefix sum are this library's
 * reading of "sliced, zero-padded" ([Endgame] "What problem is it actually
 * solving?") and of Table 2's "padded per-rank rows" and "prefix offset".
 *
 * Conventions for every call below:
 *   - All sizes and offsets are in elements unless a name says bytes.
 *   - Pointer arrays (grads, shards, params) are host arrays of DEVICE
 *     pointers, read on the host during the call only.  The caller owns every
 *     tensor; the library never frees or keeps a caller pointer.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Compute calls enqueue work on it and return; a fault inside a
 *     kernel surfaces on a later synchronisation (as TIDE_ERR_CUDA from the
 *     next call, or from the caller's own CUDA error check).
 *   - Errors are status codes; nothing aborts, throws across the ABI or
 *     exits.  tide_last_error() gives a thread-local message for the last
 *     failing call.
 *   - A plan may be used from one host thread at a time.  Its device state
 *     (work lists, pointer-table ring) is created on the device current at
 *     the first compute call and that device only; the first compute call
 *     therefore allocates and synchronises, and must come before any CUDA
 *     graph capture.  Later calls are stream-ordered and never allocate.
 *   - Each call passes its pointer arrays to the kernels through a device
 *     table.  A call whose table equals the previous one of the same kind
 *     reuses it (no upload), so unchanged buffers cost no host-to-device
 *     copy per call.
 *   - CUDA graphs: a call made while `stream` is being captured takes one of
 *     8 table slots reserved per plan and keeps it until tide_plan_destroy;
 *     every replay re-uploads that fixed table, so it uses the pointers
 *     given at capture (the data behind them may change between replays).
 *     A ninth captured call returns TIDE_ERR_INVALID_ARG.  The plan must
 *     outlive its graphs.  tide_rs_reduce_noalloc returns
 *     TIDE_ERR_INVALID_ARG on a stream under capture.
 *   - Outputs must not overlap inputs or each other (undefined results
 *     otherwise; TIDE_OPT_CHECK_OVERLAP turns on a host-side check).
 */
#ifndef TIDE_H
#define TIDE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tide_status {
  TIDE_OK = 0,
  TIDE_ERR_INVALID_ARG = 1,     /* bad descriptor, null pointer, bad index   */
  TIDE_ERR_ALIGNMENT = 2,       /* pointer not aligned to its element size   */
  TIDE_ERR_OVERFLOW = 3,        /* a size or offset does not fit in int64    */
  TIDE_ERR_OUT_OF_MEMORY = 4,   /* host or device allocation failed          */
  TIDE_ERR_CUDA = 5,            /* a CUDA runtime call failed                */
  TIDE_ERR_UNIMPLEMENTED = 6,   /* valid request outside what is built       */
  TIDE_ERR_DEVICE_MISMATCH = 7, /* plan used on another device than its own  */
  TIDE_ERR_TIMEOUT = 8          /* a kernel gave up a bounded wait (see
                                   tide_plan_check)                          */
} tide_status;

/* A parameter group over N = M*L ranks ([Abstract] Table 2).
 *   P     number of parameters (>= 0)
 *   ndim  [P] number of dimensions of each parameter (0..8)
 *   dims  the P shapes concatenated, dim 0 first; every dim >= 0
 *   M, L  nodes and GPUs per node: 1 <= L <= 8 (at most eight GPUs per
 *         NVSwitch domain, [Endgame] "Where I think it falls short"),
 *         1 <= M <= 32.  With M > L the level-2 sum runs in batches of L
 *         sources ([Endgame] "Reduce-scatter: two levels of addition...":
 *         more machines than a read-and-add can take go in batches)
 *   N     must equal M*L.
 * The descriptor is copied; the caller may free it after tide_plan_create. */
typedef struct tide_group_desc {
  int32_t P;
  const int32_t* ndim;
  const int64_t* dims;
  int32_t N;
  int32_t M;
  int32_t L;
} tide_group_desc;

typedef struct tide_plan tide_plan;  /* opaque; owned by the library */

/* Build the geometry (Kp, Rp, e_p, op, S) and the per-CTA work lists of a
 * group.  Host-only: touches no GPU.  On success *out_plan owns host memory
 * until tide_plan_destroy.  Errors: INVALID_ARG (null pointer, N != M*L,
 * L or M out of range, negative dim, ndim > 8), OVERFLOW (N*S or a shape
 * product beyond int64), OUT_OF_MEMORY. */
tide_status tide_plan_create(const tide_group_desc* desc, tide_plan** out_plan);

/* Release a plan and its host and device state.  NULL-safe.  Waits for the
 * plan's in-flight uses (its pointer-table slots) to finish first. */
void tide_plan_destroy(tide_plan* plan);

/* S, the packed shard length in elements; -1 for a NULL plan. */
int64_t tide_plan_shard_elems(const tide_plan* plan);

/* Geometry of parameter p: R_p (unpadded dim-0 rows), Rp, Kp and op.
 * Any output pointer may be NULL.  INVALID_ARG for a bad plan or p. */
tide_status tide_plan_param_geometry(const tide_plan* plan, int32_t p, int64_t* rows,
                                     int64_t* Rp, int64_t* Kp, int64_t* op);

/* Work-list introspection for tests.  which = 0: reduce-scatter items,
 * which = 1: all-gather items, which = 2 / 3: the all-gather items as the
 * TIDE_AG_BULK transport splits them (2: the 16-byte aligned middles it moves
 * by bulk copies, 3: the rest, moved by the SM kernel; bf16 offsets, base
 * pointers assumed 16-byte aligned).  Each item is 6 int64 values
 * {kind, p, r, src_off, dst_off, n}:
 *   RS: kind 0 = reduce valid rows, 1 = zero padding; src_off is the element
 *       offset inside every contributor's gradient of p, dst_off the offset
 *       inside rank r's packed shard, n the element count; one level-2 slice.
 *   AG (which 1..3): kind 2; src_off inside rank r's packed shard, dst_off
 *       inside parameter p's gathered block.
 * tide_plan_num_items returns the count (-1 for a bad plan/which);
 * tide_plan_get_items copies min(cap, count) items to out. */
int64_t tide_plan_num_items(const tide_plan* plan, int32_t which);
tide_status tide_plan_get_items(const tide_plan* plan, int32_t which, int64_t* out,
                                int64_t cap);

/* Level-2 summation order used by tide_rs_reduce for slice s (0 <= s < L)
 * of destination node n_dest (0 <= n_dest < M): writes the M source node
 * numbers, in the order their fp32 partials are added, to out[0..M) (batch
 * after batch when M > L: a batch ends after every L entries).  By default
 * the order is the Latin-square landing order of [Endgame] "Reduce-scatter:
 * two levels of addition, the last one done by NVSwitch" and [Abstract]
 * Figure 6(b): destination GPU g = 0..L-1 holds the partial of the source
 * with relative index c = (s - g) mod L, if c < M; TIDE_OPT_SUM_ORDER selects
 * the other reading.  Errors: INVALID_ARG. */
tide_status tide_plan_level2_order(const tide_plan* plan, int32_t n_dest, int32_t s, int32_t* out);

/* Plan options, set before or between calls (never while a call of the
 * plan is in flight on another thread).
 *   TIDE_OPT_RS_KERNEL     0 (default): every thread loads its
 *                          contributions directly (16-byte loads); 1: a
 *                          producer warp streams the contributors into shared
 *                          memory with bulk copies (TMA).  Both add in the
 *                          same order and give bit-identical results; the
 *                          bulk path stages one source node's windows (up
 *                          to 2 KiB per contributor) per step of its
 *                          shared-memory ring, whatever the number of
 *                          ranks; it takes at most 8 nodes (UNIMPLEMENTED
 *                          beyond).
 *   TIDE_OPT_WAIT_LIMIT_NS bound, in nanoseconds, on every wait inside the
 *                          bulk-copy kernels (default 2e9).  A kernel that runs
 *                          out records TIDE_ERR_TIMEOUT for tide_plan_check,
 *                          drains its copies and returns; the outputs of that
 *                          call are then undefined.
 *   TIDE_OPT_RS_AVERAGE, TIDE_OPT_RS_ACCUMULATE, TIDE_OPT_AG_UNPADDED
 *                          result variants (below); apply to tide_rs_reduce
 *                          (both kernels), tide_rs_staged,
 *                          tide_rs_reduce_noalloc and tide_ag_place.  The
 *                          pages give neither averaging nor an unpadded
 *                          destination; accumulating follows "accumulate the
 *                          result straight into the fp32 gradient shard"
 *                          ([Endgame] "Reduce-scatter...").
 *   TIDE_OPT_SUM_ORDER     the level-2 addition order (tide_sum_order,
 *                          below); default TIDE_SUM_LANDING.
 *   TIDE_OPT_TEST_DROP_TILE  test hook: the bulk reduce-scatter's producer
 *                          withholds the given stage fill (one source
 *                          node's windows of one tile), and the bulk
 *                          all-gather skips the given chunk's load (both
 *                          counted per CTA from 0), so a bounded wait runs
 *                          out; -1 (default) disables.
 * Errors: INVALID_ARG for an unknown option or value. */
typedef enum tide_option {
  TIDE_OPT_RS_KERNEL = 1,
  TIDE_OPT_WAIT_LIMIT_NS = 2,
  TIDE_OPT_TEST_DROP_TILE = 3,
  TIDE_OPT_RS_AVERAGE = 4,     /* 1: every reduce-scatter result is divided
                                  by N (fp32, correctly rounded) */
  TIDE_OPT_RS_ACCUMULATE = 5,  /* 1: the result is added to the shard's
                                  previous value (one fp32 add, after the sum
                                  and the division) instead of overwriting */
  TIDE_OPT_AG_UNPADDED = 6,    /* 1: tide_ag_place writes only the R_p real
                                  rows; params[p] then needs R_p*Kp elements */
  TIDE_OPT_SUM_ORDER = 7,      /* level-2 addition order, a tide_sum_order */
  TIDE_OPT_CHECK_OVERLAP = 8,  /* 1: every call first checks on the host that
                                  no output byte range overlaps an input or
                                  another output (INVALID_ARG, naming the
                                  pair); costs O(n log n) host time in the
                                  number of pointers; default 0 */
  TIDE_OPT_RD_EXCHANGE = 9,    /* tide_ag_rd_exchange's copies: 0 (default)
                                  one copy-engine copy per node per round, as
                                  the pages' transport; 1 one SM kernel launch
                                  per round over all M copies (same bytes,
                                  same result) */
  TIDE_OPT_AG_TRANSPORT = 10   /* how tide_ag_place moves the pieces, a
                                  tide_ag_transport (default TIDE_AG_SM) */
} tide_option;

/* Transports for TIDE_OPT_AG_TRANSPORT; all give the same result.  The pages'
 * all-gather uses no SM threads ([Richland] "What shipped").
 *   TIDE_AG_SM            (default) one kernel over the work list, every
 *                         thread copying 16-byte words;
 *   TIDE_AG_COPY_ENGINES  copy-engine copies, no kernel: one per (parameter,
 *                         rank) piece, or, when the N shards lie at one
 *                         constant stride (rows of one buffer) and the
 *                         unpadded option is off, one strided 2-D copy per
 *                         parameter whose pieces are at most 4 MiB (larger
 *                         pieces still go one by one);
 *   TIDE_AG_BULK          bf16 only: one thread per SM moves each piece's
 *                         16-byte aligned middle global -> shared -> global
 *                         with bulk copies (TMA), the SM kernel the rest
 *                         (two launches); a training step with it takes as
 *                         long as with TIDE_AG_SM.
 *                         Needs every shard and parameter pointer 16-byte
 *                         aligned and the padded layout; otherwise, and for
 *                         4-byte elements, the call uses TIDE_AG_SM.  Its
 *                         waits are bounded by TIDE_OPT_WAIT_LIMIT_NS
 *                         (TIDE_ERR_TIMEOUT from tide_plan_check). */
typedef enum tide_ag_transport {
  TIDE_AG_SM = 0,
  TIDE_AG_COPY_ENGINES = 1,
  TIDE_AG_BULK = 2
} tide_ag_transport;

/* Orders for TIDE_OPT_SUM_ORDER.  The pages do not say in which order the
 * NVSwitch read-and-add combines the partials ([Endgame] "Reduce-scatter:
 * two levels of addition..."), so two readings are offered; both keep the
 * batches of L relative indices, and both are exact and deterministic.
 *   TIDE_SUM_LANDING   (default) by the destination GPU g = 0..L-1 the
 *                      partial lands on, as described under tide_rs_reduce;
 *   TIDE_SUM_RELATIVE  by ascending relative index c = (n_d - n) mod M
 *                      (the same for every slice).
 * Applies to every reduce-scatter entry point; tide_plan_level2_order
 * reports the order in force. */
typedef enum tide_sum_order { TIDE_SUM_LANDING = 0, TIDE_SUM_RELATIVE = 1 } tide_sum_order;
tide_status tide_plan_set_option(tide_plan* plan, int32_t option, int64_t value);

/* Synchronise the device the plan runs on and report whether any of the
 * plan's kernels gave up a bounded wait since the last check
 * (TIDE_ERR_TIMEOUT; the flag is then cleared).  TIDE_OK for a plan that has
 * not run yet.  Errors: INVALID_ARG, CUDA. */
tide_status tide_plan_check(tide_plan* plan);

/* Kernels the plan's most recent compute call launched (0 for a call that
 * only enqueued copies or had nothing to do; tide_rs_reduce_noalloc counts
 * its table kernel too); -1 for a NULL plan.  Host-side bookkeeping, no
 * synchronisation. */
int32_t tide_plan_last_launches(const tide_plan* plan);

/* Checked builds only (libtide_checked.so, compiled with TIDE_CHECKED): every
 * global store of the kernels is first compared with the range of the work
 * item it belongs to, and a store outside it is skipped and counted.  Returns
 * the count since the last reset, after synchronising the current device
 * (reset != 0 clears it); -1 in normal builds, -2 if the synchronisation
 * failed. */
int64_t tide_debug_bounds_violations(int32_t reset);

/* Positive control of the store checks: launches one thread that asks the
 * check about an address outside a made-up range, touching no memory; a
 * checked build's count goes up by one, a normal build's stays -1.
 * Errors: CUDA. */
tide_status tide_debug_bounds_selftest(void);

/* TIDE-RS: per-parameter bf16 gradients read in place, reduced in fp32
 * straight into every rank's packed fp32 shard at its final offset
 * ([Richland] "What shipped"; [Abstract] abstract and Figure 6;
 * [Endgame] "Reduce-scatter: two levels of addition, the last one done by
 * NVSwitch").
 *   grads   host array [N*P] of device pointers; entry r*P + p is rank r's
 *           bf16 gradient of parameter p, R_p*Kp contiguous row-major
 *           elements, 2-byte aligned.  May be NULL where R_p*Kp == 0.
 *   shards  host array [N] of device pointers; shards[r] receives S fp32
 *           values, 4-byte aligned.  Every element is overwritten.
 * For destination rank r = n_d*L + l_d and element e < e_p of parameter p,
 * the result at shards[r][op + e] is, for a real row g = r*Rp + e/Kp < R_p:
 *   level 1: part_n = fp32 sum over l = 0..L-1 of grads[n*L+l][p][r*e_p + e]
 *            for every source node n (round-to-nearest-even, from +0.0);
 *   level 2: the M partials added, from +0.0, in the order of the destination
 *            GPU g = 0..L-1 they land on under the Latin-square placement
 *            (the default TIDE_SUM_LANDING; see TIDE_OPT_SUM_ORDER):
 *            slice s = (op+e) / ceil(S/L); GPU g holds the partial of the
 *            source whose relative index c = (n_d - n) mod M satisfies
 *            (s - c) mod L == g.  When M > L, relative indices go in batches
 *            [b*L, b*L + L): each batch is summed that way from +0.0 and the
 *            batch sums are added in ascending b.
 * and +0.0 for a padding row.  The result is bit-identical to that order.
 * Errors: INVALID_ARG (null plan/arrays/pointer; overlapping buffers when
 * TIDE_OPT_CHECK_OVERLAP is on), ALIGNMENT, CUDA, OUT_OF_MEMORY (first call's
 * device set-up), DEVICE_MISMATCH, UNIMPLEMENTED (the bulk-copy kernel with
 * more than 8 nodes). */
tide_status tide_rs_reduce(tide_plan* plan, const void* const* grads, float* const* shards,
                           void* stream);

/* TIDE-AG direct landing: every rank's packed shard piece is written once,
 * at its final parameter-major address, with no rank-major temporary
 * ([Endgame] "All-gather: parameters land at their final address";
 * [Richland] "What shipped"; [Abstract] Figure 1).
 *   shards      host array [N] of device pointers, S elements each
 *   params      host array [P] of device pointers; params[p] receives the
 *               padded gathered block of N*Rp rows x Kp (the parameter proper
 *               is its first R_p rows).  May be NULL where e_p == 0.
 *   elem_bytes  2 (bf16 parameters) or 4 (fp32, e.g. to gather RS output)
 * For every p, r and e < e_p: params[p][r*e_p + e] = shards[r][op + e],
 * bit for bit.  Pointers must be elem_bytes-aligned.
 * Errors: INVALID_ARG, ALIGNMENT, CUDA, OUT_OF_MEMORY, DEVICE_MISMATCH. */
tide_status tide_ag_place(tide_plan* plan, const void* const* shards, void* const* params,
                          int32_t elem_bytes, void* stream);

/* tide_rs_reduce for callers that cannot allocate device memory.  The pages
 * have no counterpart to this call; it exists for users of this library.
 * tide_rs_reduce allocates device memory for its work list and pointer tables
 * on first use; some callers cannot: a process whose free device memory all
 * belongs to a caching allocator, code that must not take the implicit device
 * synchronisation that cudaMalloc/cudaFree can bring, or a fixed memory
 * budget reserved up front.  This call allocates nothing.  It keeps the same
 * data in one fixed 8 MiB __device__ array that every GPU loading libtide
 * holds until the process exits, and runs the same kernel, so its results
 * are bit-identical to tide_rs_reduce's.
 *   plan, grads, shards, stream: as for tide_rs_reduce.  The plan's own
 *   device state is not used or created.
 * The first call on a device looks up the array's address on that device;
 * make that first call before any CUDA graph capture.  A call on a stream
 * that is being captured returns TIDE_ERR_INVALID_ARG before touching the
 * array: a captured launch would keep reading tables that later calls
 * rewrite.  Host threads calling on one device are serialised (one lock per
 * device, held across the uploads).  The array is shared by
 * all calls on a device and keeps the last call's contents; the library
 * remembers, per device, which plan's work list it holds and which pointer
 * arrays its tables were built from, and a call copies into it (from
 * pageable host memory, so the call may wait for earlier work on `stream`)
 * only what differs: the work list when the plan changes, a pointer table
 * when its pointers change.  Calling the same plan on the same buffers
 * uploads nothing.  The kernel's work counter also lives in the array; it is
 * zeroed with cudaMemsetAsync when a plan's work list is copied in, and every
 * launch leaves it at zero.  Calls whose work overlaps on the GPU (different
 * streams, no ordering) race on the array.  tide_plan_last_launches counts
 * the table kernel only when the gradient pointers changed.
 * Errors: as tide_rs_reduce; INVALID_ARG also when the group's work list and
 * tables exceed the 8 MiB array (use tide_rs_reduce for such groups). */
tide_status tide_rs_reduce_noalloc(const tide_plan* plan, const void* const* grads, float* const* shards,
                                   void* stream);

/* ---- Slot-Reuse ------------------------------------------------------------
 * [Endgame] "Reduce-scatter: two levels of addition...", last paragraph;
 * [Abstract] Figure 7: gradients are copied into the all-gather slot that has
 * just been vacated, so their own memory can be freed at once; the
 * reduce-scatter then reads them from the slot.  A rank's slot is its
 * gathered parameter group: N*S bf16 elements, parameter p's padded block at
 * N*op (the tide_ag_place layout).
 *
 * tide_slot_pack: slots[r][N*op + e] = grads[r*P + p][e] for e < R_p*Kp
 * (bf16).  grads as tide_rs_reduce; slots: host array [N] of device pointers
 * to N*S elements, 2-byte aligned; the padding rows of a slot are left as
 * they are.  tide_rs_reduce_slots: tide_rs_reduce with rank r's gradient of
 * p read at slots[r] + N*op (same options, same bits).  Errors: as
 * tide_rs_reduce. */
tide_status tide_slot_pack(tide_plan* plan, const void* const* grads, void* const* slots, void* stream);
tide_status tide_rs_reduce_slots(tide_plan* plan, const void* const* slots, float* const* shards, void* stream);

/* ---- Reduce-scatter in the pages' two stages -----------------------------
 * [Endgame] "Reduce-scatter: two levels of addition, the last one done by
 * NVSwitch"; [Abstract] Figure 6.  Same result as tide_rs_reduce, bit for
 * bit, computed the way the pages split it:
 *   stage 1 (summing CTAs): for every destination rank r = n_d*L + l_d and
 *   source node n_s, the fp32 sum of n_s's L local copies (l ascending) is
 *   written to the inbox slot where the Latin square lands it: destination
 *   GPU g = (s - c) mod L, c = (n_d - n_s) mod M, for slice s;
 *   stage 2 (landing CTAs): each destination element adds its slice's
 *   partials in the plan's level-2 order (by default from landing GPUs
 *   g = 0..L-1 in turn), batch by batch when M > L.
 * The inbox costs 8*M extra bytes of traffic per shard element. */

/* Floats the inbox needs: M * L * M * L * ceil(S / L) (0 when S == 0); -1
 * for a NULL plan.  Layout [n_d][g][c][L * B], rank l_d's block at l_d * B. */
int64_t tide_plan_inbox_elems(const tide_plan* plan);

/* grads, shards, stream: as tide_rs_reduce.  inbox: device pointer to
 * tide_plan_inbox_elems() floats, 4-byte aligned, caller-owned scratch whose
 * contents are overwritten.  sum_ctas_per_rank / landing_ctas_per_rank: CTAs
 * of each stage per emulated rank (16 and 4 reproduce the pages' training
 * budget); 0 picks a grid that fills the GPU.  Errors: as tide_rs_reduce;
 * INVALID_ARG for a NULL inbox or a negative CTA count. */
tide_status tide_rs_staged(tide_plan* plan, const void* const* grads, float* const* shards, float* inbox,
                           int32_t sum_ctas_per_rank, int32_t landing_ctas_per_rank, void* stream);

/* ---- All-gather across nodes by recursive doubling ----------------------
 * [Endgame] "All-gather: parameters land at their final address" and
 * [Abstract] Figure 5: on rail l (GPU l of every node) each node starts with
 * its own packed shard; in round d = 0, 1, ... a node sends the first
 * min(2^d, M - 2^d) pieces it has collected to node (n - 2^d) mod M and
 * appends as many from node (n + 2^d) mod M.  After ceil(log2 M) rounds node
 * n's stage slot k holds node (n + k) mod M's shard (rank
 * ((n + k) mod M) * L + l). */

/* Rounds the exchange needs: ceil(log2 M) (0 for M = 1); -1 if M < 1. */
int32_t tide_rd_rounds(int32_t M);

/* Pieces each node sends in round d: min(2^d, M - 2^d); -1 if d is not a
 * round of the exchange. */
int32_t tide_rd_send_count(int32_t M, int32_t d);

/* Emulate one rail's exchange between the M nodes' stage buffers on this GPU.
 *   stages      host array [M] of device pointers; stages[n] holds M packed
 *               shards of S elements (slot k at k*S); slot 0 must already
 *               hold node n's own shard.  Slots 1..M-1 are overwritten.
 *   elem_bytes  2 or 4
 * Every round is one device-to-device copy per node (copy engines, as the
 * pages' transport), enqueued on `stream` in round order; when the M stage
 * buffers lie at one constant stride (rows of one buffer) and a round's
 * copies are at most 16 MiB each, the round is two strided copies instead.
 * With TIDE_OPT_RD_EXCHANGE = 1 every round is one SM kernel launch.
 * Errors: INVALID_ARG (null or aliasing buffers), CUDA, OUT_OF_MEMORY and
 * DEVICE_MISMATCH (SM exchange: first call's set-up). */
tide_status tide_ag_rd_exchange(tide_plan* plan, void* const* stages, int32_t elem_bytes, void* stream);

/* Destination phase of the exchange ([Abstract] Figure 5(b)): write rail
 * `rail`'s M pieces from node `node`'s stage buffer (slot k = rank
 * ((node + k) mod M) * L + rail, S elements each) into the parameters'
 * parameter-major blocks, every piece once at its final address:
 * params[p][r*e_p + e] = stage[k*S + op + e].  Same kernel and the same
 * argument rules as tide_ag_place; `stage` is a device pointer to M*S
 * elements.  Errors: INVALID_ARG, ALIGNMENT, CUDA, OUT_OF_MEMORY,
 * DEVICE_MISMATCH. */
tide_status tide_ag_stage_place(tide_plan* plan, const void* stage, int32_t node, int32_t rail,
                                void* const* params, int32_t elem_bytes, void* stream);

/* ---- Every rail at once --------------------------------------------------
 * On the pages every GPU forwards its own rail's data across nodes
 * ([Richland] "What shipped"; [Abstract] Figure 5 draws one rail), so the L
 * rails exchange independently and at the same time.  These calls emulate
 * all of them together, in one launch per step instead of one per rail; the
 * bytes moved and their order are those of the rail-by-rail calls.  Buffer l*M + n of a `stages` array is node n's stage
 * buffer on rail l (M*S elements, slot k at k*S); all L*M are distinct,
 * caller-owned device buffers. */

/* Slot 0 of every stage buffer gets its own shard:
 * stages[l*M + n][0 .. S) = shards[n*L + l][0 .. S).
 *   shards      host array [N] of device pointers (S elements each), read
 *   stages      host array [L*M] of device pointers, slot 0 written
 *   elem_bytes  2 or 4
 * One all-gather kernel launch on `stream`.  Errors: INVALID_ARG (null
 * pointers; with TIDE_OPT_CHECK_OVERLAP, a slot 0 overlapping a shard or
 * another slot 0), ALIGNMENT (pointer not element-aligned), CUDA,
 * OUT_OF_MEMORY, DEVICE_MISMATCH. */
tide_status tide_ag_stage_init(tide_plan* plan, const void* const* shards, void* const* stages, int32_t elem_bytes,
                               void* stream);

/* tide_ag_rd_exchange on every rail: afterwards slot k of stages[l*M + n]
 * holds rank ((n + k) mod M)*L + l's shard, for every l and n.  With
 * TIDE_OPT_RD_EXCHANGE = 1 each round is one SM kernel launch covering all
 * rails; with copy engines (default) each round is L*M copies, or two
 * strided copies per rail when the L*M buffers lie at one constant stride and
 * the round's copies are at most 16 MiB each.
 *   stages      host array [L*M] of device pointers, slot 0 already filled
 *               (tide_ag_stage_init); slots 1..M-1 are overwritten
 * Errors: INVALID_ARG (null or repeated buffers; with
 * TIDE_OPT_CHECK_OVERLAP, overlapping buffers), ALIGNMENT, UNIMPLEMENTED
 * (SM exchange with more than 5 rounds, M > 32), CUDA, OUT_OF_MEMORY,
 * DEVICE_MISMATCH.
 *
 * Placement from every rail at once needs no entry point of its own: node
 * `node`'s pieces land with tide_ag_place given
 * shards[r] = stages[(r % L)*M + node] + ((r / L - node) mod M) * S elements,
 * which writes params[p][r*e_p + e] from slot (r/L - node) mod M of rail
 * r % L, as tide_ag_stage_place does rail by rail. */
tide_status tide_ag_rd_exchange_rails(tide_plan* plan, void* const* stages, int32_t elem_bytes, void* stream);

/* Static text for a status code. */
const char* tide_status_string(tide_status status);

/* Thread-local message describing the last failing call on this thread
 * ("" if none). */
const char* tide_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TIDE_H */

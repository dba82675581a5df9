// Host side of libtide: group validation, per-parameter shard geometry, the
// Latin-square level-2 order table and the per-CTA work lists.  Touches no GPU.
//
// Geometry follows the notation table of the TIDE preprint's abstract page
// (Table 2: M, L, N = M*L, r = n*L + l, Rp, Kp, sp, op, S) with dim-0
// chunk-and-pad sharding: Rp = ceil(R_p / N), rank r owns rows
// [r*Rp, (r+1)*Rp), rows at or beyond R_p are zero padding, and op is the
// gap-free prefix sum of the per-rank pieces e_p = Rp*Kp.

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <iterator>
#include <new>

#include "tide_internal.h"

namespace tide {

namespace {
thread_local std::string g_last_error;

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

}  // namespace

// Level-2 order for slice s of destination node n_dest ("Reduce-scatter: two
// levels of addition, the last one done by NVSwitch" in "The Endgame of FSDP
// Communication"; the preprint's Figure 6(b)).  Slice s from the source with
// relative index c = (n_dest - n_src) mod M lands on destination GPU
// (s - c) mod L, so within batch b GPU g holds c = b*L + (s - g) mod L, if that
// c is below M.  The partials are added in landing-GPU order g = 0..L-1, batch
// after batch; with TIDE_SUM_RELATIVE, by ascending c within each batch.
void build_order_table(tide_plan* pl) {
  const int M = pl->M, L = pl->L;
  for (int n_dest = 0; n_dest < M; ++n_dest) {
    for (int s = 0; s < L; ++s) {
      int k = 0;
      // With M > L the sources go in batches of L relative indices (one
      // read-and-add sums at most one partial per destination GPU).
      for (int b = 0; b * L < M; ++b) {
        for (int j = 0; j < L; ++j) {
          const int c = pl->sum_order == TIDE_SUM_RELATIVE ? b * L + j : b * L + ((s - j) % L + L) % L;
          if (c < M) pl->order[(n_dest * L + s) * M + k++] = (uint8_t)(((n_dest - c) % M + M) % M);
        }
      }
    }
  }
}

tide_status check_overlap(const std::vector<ByteRange>& inputs, std::vector<ByteRange> outputs) {
  auto describe = [](const ByteRange& r) { return std::string(r.what) + "[" + std::to_string(r.index) + "]"; };
  outputs.erase(std::remove_if(outputs.begin(), outputs.end(), [](const ByteRange& r) { return r.hi <= r.lo; }),
                outputs.end());
  std::sort(outputs.begin(), outputs.end(), [](const ByteRange& a, const ByteRange& b) { return a.lo < b.lo; });
  for (size_t i = 1; i < outputs.size(); ++i)
    if (outputs[i].lo < outputs[i - 1].hi)
      return fail(TIDE_ERR_INVALID_ARG, "outputs " + describe(outputs[i - 1]) + " and " + describe(outputs[i]) +
                                            " overlap");
  for (const ByteRange& in : inputs) {
    if (in.hi <= in.lo) continue;
    // Outputs are sorted and disjoint: only the last one starting before
    // in.hi can reach into [in.lo, in.hi).
    auto it = std::lower_bound(outputs.begin(), outputs.end(), in.hi,
                               [](const ByteRange& o, uintptr_t v) { return o.lo < v; });
    if (it != outputs.begin() && std::prev(it)->hi > in.lo)
      return fail(TIDE_ERR_INVALID_ARG, "output " + describe(*std::prev(it)) + " overlaps input " + describe(in));
  }
  return TIDE_OK;
}

namespace {

void build_rs_items(tide_plan* pl) {
  const int64_t S = pl->S;
  const int64_t chunk = rs_chunk_elems(pl->N);
  const int64_t slice_len = S > 0 ? (S + pl->L - 1) / pl->L : 1;
  for (int32_t p = 0; p < pl->P; ++p) {
    const int64_t e_p = pl->e[p], o_p = pl->o[p];
    if (e_p == 0) continue;
    for (int32_t r = 0; r < pl->N; ++r) {
      const int64_t real_rows = std::min(pl->Rp[p], std::max<int64_t>(0, pl->rows[p] - r * pl->Rp[p]));
      const int64_t v = real_rows * pl->Kp[p];
      const int64_t src0 = r * e_p;  // rank r's rows start at global row r*Rp
      for (int64_t e = 0; e < v;) {
        const int64_t s = (o_p + e) / slice_len;
        const int64_t slice_end = (s + 1) * slice_len - o_p;
        const int64_t chunk_end = ((src0 + e) / chunk + 1) * chunk - src0;
        const int64_t end = std::min(v, std::min(slice_end, chunk_end));
        pl->rs_items.push_back(RsItem{src0 + e, o_p + e, (int32_t)(end - e), p, r, (int16_t)s, RS_VALID});
        e = end;
      }
      for (int64_t e = v; e < e_p;) {
        const int64_t s = (o_p + e) / slice_len;
        const int64_t slice_end = (s + 1) * slice_len - o_p;
        const int64_t chunk_end = ((o_p + e) / kRsPadChunk + 1) * kRsPadChunk - o_p;
        const int64_t end = std::min(e_p, std::min(slice_end, chunk_end));
        pl->rs_items.push_back(RsItem{0, o_p + e, (int32_t)(end - e), p, r, (int16_t)s, RS_PAD});
        e = end;
      }
    }
  }
}

// Split every all-gather item for the bulk-copy transport, for bf16 pieces
// and 16-byte aligned base pointers: an item whose source and destination
// byte offsets differ mod 16 stays whole on the SM kernel; otherwise its head
// (up to the destination's next 16-byte boundary) and tail (below 16 bytes)
// go to the SM kernel and the aligned middle to bulk copies, in chunks of at
// most kAgBulkChunkElems elements.
void build_ag_bulk_items(tide_plan* pl) {
  for (const AgItem& it : pl->ag_items) {
    const int64_t sb = 2 * it.src_off, db = 2 * it.dst_off;
    if ((sb - db) % 16 != 0) {
      pl->ag_rest_items.push_back(it);
      continue;
    }
    const int64_t head = std::min<int64_t>(it.n, ((16 - db % 16) % 16) / 2);
    const int64_t mid = (it.n - head) / 8 * 8;
    if (head > 0) pl->ag_rest_items.push_back(AgItem{it.src_off, it.dst_off, (int32_t)head, it.p, it.r, 0});
    for (int64_t c = 0; c < mid; c += kAgBulkChunkElems)
      pl->ag_bulk_items.push_back(AgItem{it.src_off + head + c, it.dst_off + head + c,
                                         (int32_t)std::min<int64_t>(kAgBulkChunkElems, mid - c), it.p, it.r, 0});
    if (head + mid < it.n)
      pl->ag_rest_items.push_back(AgItem{it.src_off + head + mid, it.dst_off + head + mid,
                                         (int32_t)(it.n - head - mid), it.p, it.r, 0});
  }
}

void build_ag_items(tide_plan* pl) {
  const int64_t chunk = kAgChunkBytes / 2;  // elements; 64 KiB of bf16
  for (int32_t p = 0; p < pl->P; ++p) {
    const int64_t e_p = pl->e[p], o_p = pl->o[p];
    for (int32_t r = 0; r < pl->N; ++r) {
      const int64_t dst0 = r * e_p;
      for (int64_t e = 0; e < e_p;) {
        const int64_t end = std::min(e_p, ((dst0 + e) / chunk + 1) * chunk - dst0);
        pl->ag_items.push_back(AgItem{o_p + e, dst0 + e, (int32_t)(end - e), p, r, 0});
        e = end;
      }
    }
  }
}
// The all-gather items of real rows only (an unpadded parameter is the
// first R_p rows of the padded block, so offsets are unchanged), and the
// Slot-Reuse packing items: rank r's gradient of p (R_p*Kp elements) copied
// to offset N*op of rank r's all-gather slot.
void build_variant_items(tide_plan* pl) {
  for (const AgItem& it : pl->ag_items) {
    const int64_t real = pl->rows[it.p] * pl->Kp[it.p];  // elements of the unpadded parameter
    const int64_t end = std::min<int64_t>(it.dst_off + it.n, real);
    if (end > it.dst_off) {
      AgItem c = it;
      c.n = (int32_t)(end - it.dst_off);
      pl->ag_items_unpadded.push_back(c);
    }
  }
  const int64_t chunk = kAgChunkBytes / 2;
  for (int32_t r = 0; r < pl->N; ++r) {
    for (int32_t p = 0; p < pl->P; ++p) {
      const int64_t n = pl->rows[p] * pl->Kp[p];
      for (int64_t e = 0; e < n;) {
        const int64_t end = std::min(n, (e / chunk + 1) * chunk);
        pl->pack_items.push_back(AgItem{e, (int64_t)pl->N * pl->o[p] + e, (int32_t)(end - e), r, r * pl->P + p, 0});
        e = end;
      }
    }
  }
  pl->slot_grads.assign((size_t)pl->N * pl->P, nullptr);
}

void build_prefixes(tide_plan* pl) {
  pl->ag_prefix.resize(pl->ag_items.size() + 1);
  pl->ag_prefix[0] = 0;
  for (size_t i = 0; i < pl->ag_items.size(); ++i)
    pl->ag_prefix[i + 1] = pl->ag_prefix[i] + ag_item_cost(pl->ag_items[i]);
}
}  // namespace

namespace {
template <class Item, class Split>
std::vector<UnitStart> unit_starts(const std::vector<Item>& items, const std::vector<int64_t>& prefix,
                                   int64_t workers, int64_t target, int64_t max_k, Split split) {
  const int64_t total = prefix.back();
  const int64_t n_items = (int64_t)items.size();
  int64_t k = workers > 0 ? (total + workers * target - 1) / (workers * target) : 1;
  k = std::max<int64_t>(1, std::min(k, max_k));
  const int64_t U = std::max<int64_t>(1, k * workers);
  std::vector<UnitStart> out(U + 1);
  int64_t i = 0;
  for (int64_t u = 0; u <= U; ++u) {
    const int64_t t = (int64_t)((__int128)total * u / U);
    while (i < n_items && prefix[i + 1] <= t) ++i;  // prefix[i] <= t < prefix[i + 1]
    int64_t item = i, off = 0;
    if (i < n_items) {
      off = split(items[i], t - prefix[i]);
      if (off >= items[i].n) {
        item = i + 1;
        off = 0;
      }
    }
    out[u] = UnitStart{(int32_t)item, (int32_t)off};
  }
  return out;
}
}  // namespace

std::vector<UnitStart> ag_unit_starts_of(const std::vector<AgItem>& items, int64_t workers, int64_t target,
                                         int64_t max_k) {
  std::vector<int64_t> prefix(items.size() + 1, 0);
  for (size_t i = 0; i < items.size(); ++i) prefix[i + 1] = prefix[i] + ag_item_cost(items[i]);
  return unit_starts(items, prefix, workers, target, max_k, [](const AgItem& it, int64_t rel) { return ag_split(it, rel); });
}

std::vector<UnitStart> ag_unit_starts(const tide_plan* pl, int64_t workers, int64_t target, int64_t max_k) {
  return unit_starts(pl->ag_items, pl->ag_prefix, workers, target, max_k,
                     [](const AgItem& it, int64_t rel) { return ag_split(it, rel); });
}

tide_status fail(tide_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

void clear_error() { g_last_error.clear(); }

}  // namespace tide

using namespace tide;

extern "C" {

const char* tide_status_string(tide_status status) {
  switch (status) {
    case TIDE_OK: return "ok";
    case TIDE_ERR_INVALID_ARG: return "invalid argument";
    case TIDE_ERR_ALIGNMENT: return "misaligned pointer";
    case TIDE_ERR_OVERFLOW: return "size overflow";
    case TIDE_ERR_OUT_OF_MEMORY: return "out of memory";
    case TIDE_ERR_CUDA: return "CUDA error";
    case TIDE_ERR_UNIMPLEMENTED: return "not implemented";
    case TIDE_ERR_DEVICE_MISMATCH: return "plan used on another device";
    case TIDE_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
  }
  return "unknown status";
}

const char* tide_last_error(void) { return g_last_error.c_str(); }

tide_status tide_plan_create(const tide_group_desc* d, tide_plan** out_plan) {
  clear_error();
  if (!out_plan) return fail(TIDE_ERR_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  if (!d) return fail(TIDE_ERR_INVALID_ARG, "descriptor is NULL");
  if (d->P < 0) return fail(TIDE_ERR_INVALID_ARG, "P < 0");
  if (d->P > 0 && (!d->ndim || !d->dims)) return fail(TIDE_ERR_INVALID_ARG, "ndim or dims is NULL");
  if (d->L < 1 || d->L > kMaxL) return fail(TIDE_ERR_INVALID_ARG, "L must be in [1, 8]");
  if (d->M < 1) return fail(TIDE_ERR_INVALID_ARG, "M must be >= 1");
  if (d->M > kMaxM) return fail(TIDE_ERR_INVALID_ARG, "M must be at most 32");
  if ((int64_t)d->M * d->L != d->N) return fail(TIDE_ERR_INVALID_ARG, "N must equal M*L");

  tide_plan* pl = new (std::nothrow) tide_plan();
  if (!pl) return fail(TIDE_ERR_OUT_OF_MEMORY, "plan allocation failed");
  static std::atomic<uint64_t> next_uid{1};
  pl->uid = next_uid.fetch_add(1);
  try {
    pl->N = d->N;
    pl->M = d->M;
    pl->L = d->L;
    pl->P = d->P;
    pl->rows.resize(d->P);
    pl->Kp.resize(d->P);
    pl->Rp.resize(d->P);
    pl->e.resize(d->P);
    pl->o.resize(d->P);
    int64_t at = 0, offset = 0;
    for (int32_t p = 0; p < d->P; ++p) {
      const int32_t nd = d->ndim[p];
      if (nd < 0 || nd > kMaxNdim) {
        delete pl;
        return fail(TIDE_ERR_INVALID_ARG, "ndim must be in [0, 8] (parameter " + std::to_string(p) + ")");
      }
      int64_t rows = 1, k = 1;  // a 0-D parameter counts as shape [1]
      for (int32_t i = 0; i < nd; ++i) {
        const int64_t dim = d->dims[at + i];
        if (dim < 0) {
          delete pl;
          return fail(TIDE_ERR_INVALID_ARG, "negative dimension (parameter " + std::to_string(p) + ")");
        }
        if (i == 0) rows = dim;
        else if (!mul_ok(k, dim, &k)) {
          delete pl;
          return fail(TIDE_ERR_OVERFLOW, "row length overflows int64");
        }
      }
      at += nd;
      const int64_t rp = (rows + d->N - 1) / d->N;
      int64_t e_p, block;
      if (!mul_ok(rp, k, &e_p) || !mul_ok(e_p, d->N, &block) || !add_ok(offset, e_p, &pl->S)) {
        delete pl;
        return fail(TIDE_ERR_OVERFLOW, "shard size overflows int64");
      }
      pl->rows[p] = rows;
      pl->Kp[p] = k;
      pl->Rp[p] = rp;
      pl->e[p] = e_p;
      pl->o[p] = offset;
      offset = pl->S;
    }
    pl->S = offset;
    int64_t total;
    if (!mul_ok(pl->S, pl->N, &total) || !mul_ok(total, 4, &total)) {
      delete pl;
      return fail(TIDE_ERR_OVERFLOW, "N*S overflows int64");
    }
    build_order_table(pl);
    build_rs_items(pl);
    build_ag_items(pl);
    build_ag_bulk_items(pl);
    build_variant_items(pl);
    build_prefixes(pl);
  } catch (const std::bad_alloc&) {
    delete pl;
    return fail(TIDE_ERR_OUT_OF_MEMORY, "host allocation failed while building the plan");
  }
  *out_plan = pl;
  return TIDE_OK;
}

int32_t tide_rd_rounds(int32_t M) {
  if (M < 1) return -1;
  int32_t d = 0;
  while ((int64_t(1) << d) < M) ++d;  // rounds run while 2^d < M
  return d;
}

int32_t tide_rd_send_count(int32_t M, int32_t d) {
  if (M < 1 || d < 0 || d >= tide_rd_rounds(M)) return -1;
  const int64_t half = int64_t(1) << d;
  return (int32_t)std::min<int64_t>(half, M - half);
}

int64_t tide_plan_shard_elems(const tide_plan* pl) { return pl ? pl->S : -1; }

tide_status tide_plan_param_geometry(const tide_plan* pl, int32_t p, int64_t* rows, int64_t* Rp,
                                     int64_t* Kp, int64_t* op) {
  clear_error();
  if (!pl) return fail(TIDE_ERR_INVALID_ARG, "plan is NULL");
  if (p < 0 || p >= pl->P) return fail(TIDE_ERR_INVALID_ARG, "parameter index out of range");
  if (rows) *rows = pl->rows[p];
  if (Rp) *Rp = pl->Rp[p];
  if (Kp) *Kp = pl->Kp[p];
  if (op) *op = pl->o[p];
  return TIDE_OK;
}

tide_status tide_plan_level2_order(const tide_plan* pl, int32_t n_dest, int32_t s, int32_t* out) {
  clear_error();
  if (!pl || !out) return fail(TIDE_ERR_INVALID_ARG, "plan or out is NULL");
  if (n_dest < 0 || n_dest >= pl->M || s < 0 || s >= pl->L)
    return fail(TIDE_ERR_INVALID_ARG, "n_dest or slice out of range");
  for (int32_t k = 0; k < pl->M; ++k) out[k] = pl->order[(n_dest * pl->L + s) * pl->M + k];
  return TIDE_OK;
}

int64_t tide_plan_num_items(const tide_plan* pl, int32_t which) {
  if (!pl) return -1;
  if (which == 0) return (int64_t)pl->rs_items.size();
  if (which == 1) return (int64_t)pl->ag_items.size();
  if (which == 2) return (int64_t)pl->ag_bulk_items.size();
  if (which == 3) return (int64_t)pl->ag_rest_items.size();
  return -1;
}

tide_status tide_plan_get_items(const tide_plan* pl, int32_t which, int64_t* out, int64_t cap) {
  clear_error();
  if (!pl || (!out && cap > 0) || cap < 0) return fail(TIDE_ERR_INVALID_ARG, "bad plan, buffer or cap");
  if (which == 0) {
    const int64_t n = std::min<int64_t>(cap, (int64_t)pl->rs_items.size());
    for (int64_t i = 0; i < n; ++i) {
      const RsItem& it = pl->rs_items[i];
      int64_t* o = out + 6 * i;
      o[0] = it.kind; o[1] = it.p; o[2] = it.r; o[3] = it.src_off; o[4] = it.dst_off; o[5] = it.n;
    }
    return TIDE_OK;
  }
  if (which >= 1 && which <= 3) {
    const std::vector<AgItem>& v = which == 1 ? pl->ag_items : which == 2 ? pl->ag_bulk_items : pl->ag_rest_items;
    const int64_t n = std::min<int64_t>(cap, (int64_t)v.size());
    for (int64_t i = 0; i < n; ++i) {
      const AgItem& it = v[i];
      int64_t* o = out + 6 * i;
      o[0] = AG_COPY; o[1] = it.p; o[2] = it.r; o[3] = it.src_off; o[4] = it.dst_off; o[5] = it.n;
    }
    return TIDE_OK;
  }
  return fail(TIDE_ERR_INVALID_ARG, "which must be 0 (RS), 1 (AG), 2 or 3 (bulk AG split)");
}

}  // extern "C"

"""Plain CPU oracle: TIDE's packed-shard layout, two-level fp32 reduce-scatter
and direct-landing all-gather, written from the pages' definitions.

TEST INFRASTRUCTURE ONLY -- imported by the tests, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``; never by the CUDA library, with
which it shares no code.  Slow and obvious on purpose: numpy float32 arrays are
used only for elementwise IEEE round-to-nearest-even adds across independent
output elements; the order of the additions for each output element is exactly
the one written out below, with no blocking, fusion or reordering.

Sources (three web pages about the TIDE preprint, arXiv 2610.38228):

[Endgame]  "The Endgame of FSDP Communication: Layout-Aware Collectives on Copy
           Engines, RDMA, and NVSwitch" (explainer)
[Richland] "TIDE gives FSDP2 layout-aware zero-copy collectives: up to 27.1%
           faster steps on 64 GPUs, zero-SM all-gather, bf16->fp32
           reduce-scatter" (news post)
[Abstract] the preprint's abstract page with its figure captions and tables

Notation follows [Abstract] Table 2 (Notation): M nodes, L GPUs per NVSwitch
domain, N = M*L ranks, r = n*L + l; for parameter p, Rp padded per-rank rows,
Kp row length, sp / op per-rank shard size and prefix offset (kept here in
elements, not bytes), S per-rank packed shard size.

Readings taken where the pages leave a step open (each is marked "Reading" at
its use below):
  R1  Rp = ceil(R_p / N); rank r owns global rows [r*Rp, (r+1)*Rp); rows at or
      beyond R_p are zero padding.
  R2  Kp = product of the dims after dim 0 (1 for a 1-D tensor; a 0-D tensor
      is treated as shape [1]).
  R3  op is the plain prefix sum of the per-rank piece sizes, no alignment gap.
  R4  the reduction is a plain sum (no averaging), fp32 round-to-nearest-even,
      every accumulator starting from +0.0.
  R5  level 2 adds the node partials in landing-GPU order g = 0..L-1; with
      more nodes than GPUs per node, batch by batch (batches of L relative
      indices, batch sums added in ascending batch order).
  R14 the alternative order ``RELATIVE``: within each batch the partials are
      added in ascending relative index c = (n_dest - n_src) mod M instead.
  R6  slice s of a destination node is block s of each of its ranks' packed
      shards, cut into L contiguous blocks of ceil(S / L) elements.
  R8  level 1 adds the L local contributions in ascending local index l.
  R9  the all-gather writes the padded [N*Rp, Kp] parameter-major block.
"""

from dataclasses import dataclass

import numpy as np

__all__ = [
    "Geometry", "geometry", "rank_major_offset", "param_major_offset", "valid_elems",
    "owner_of_row", "relative_index", "landing_gpu", "handled_slice", "slice_len",
    "slice_of", "level2_order", "level2_batches", "LANDING", "RELATIVE", "bf16_to_f32", "rs_reduce",
    "ag_place", "rs_element", "ag_element",
]


# --------------------------------------------------------------------------
# Layout: [Abstract] Table 2 (Notation); [Endgame] "What problem is it
# actually solving?" (the hand-checkable example of rank-major vs
# parameter-major offsets); [Abstract] Figure 1.
# --------------------------------------------------------------------------

@dataclass
class Geometry:
    N: int
    P: int
    rows: list   # R_p, the unpadded dim-0 size of parameter p
    Kp: list     # row length of p (Reading R2)
    Rp: list     # padded per-rank rows of p (Reading R1)
    e: list      # per-rank piece of p in elements, Rp * Kp
    o: list      # prefix offset op of p inside a packed shard, in elements (R3)
    S: int       # per-rank packed shard size in elements


def geometry(shapes, N):
    """Per-parameter dim-0 shard geometry of a parameter group over N ranks."""
    if N < 1:
        raise ValueError("N must be >= 1")
    rows, Kp, Rp, e, o = [], [], [], [], []
    offset = 0
    for shape in shapes:
        shape = tuple(int(d) for d in shape) or (1,)          # Reading R2: 0-D as [1]
        if any(d < 0 for d in shape):
            raise ValueError("negative dimension")
        k = 1
        for d in shape[1:]:
            k *= d                                            # Reading R2
        r_pad = -(-shape[0] // N)                             # Reading R1: ceil(R_p / N)
        rows.append(shape[0])
        Kp.append(k)
        Rp.append(r_pad)
        e.append(r_pad * k)
        o.append(offset)                                      # Reading R3
        offset += r_pad * k
    return Geometry(N=N, P=len(rows), rows=rows, Kp=Kp, Rp=Rp, e=e, o=o, S=offset)


def rank_major_offset(geo, p, r):
    """Element offset of rank r's piece of p in the flat rank-major buffer.

    All of rank 0's pieces come first, then rank 1's, and so on
    ([Endgame] "What problem is it actually solving?").
    """
    return r * geo.S + geo.o[p]


def param_major_offset(geo, p, r):
    """Element offset of rank r's piece of p when every parameter is one block.

    Parameter p's block starts after the N full pieces of every earlier
    parameter (N * op), and rank r's piece sits r pieces into it
    ([Endgame] "What problem is it actually solving?"; [Abstract] Figure 1).
    """
    return geo.N * geo.o[p] + r * geo.e[p]


def owner_of_row(geo, p, g):
    """Rank that holds global row g of parameter p (Reading R1)."""
    return g // geo.Rp[p]


def valid_elems(geo, p, r):
    """Elements of rank r's piece of p that come from real rows (the rest pad)."""
    real_rows = min(geo.Rp[p], max(0, geo.rows[p] - r * geo.Rp[p]))
    return real_rows * geo.Kp[p]


# --------------------------------------------------------------------------
# Latin-square placement: [Endgame] "Reduce-scatter: two levels of addition,
# the last one done by NVSwitch"; [Abstract] Figure 6(b).
# --------------------------------------------------------------------------

def relative_index(n_dest, n_src, M):
    """c = destination's node number minus the source's, modulo M."""
    return (n_dest - n_src) % M


def handled_slice(j, c, L):
    """On a source node with relative index c, GPU j sums slice (j + c) mod L."""
    return (j + c) % L


def landing_gpu(s, c, L):
    """Slice s from the source with relative index c lands on GPU (s - c) mod L.

    GPU j of the source sends over line j to GPU j of the destination, and it
    handles slice s = (j + c) mod L, so j = (s - c) mod L.
    """
    return (s - c) % L


def slice_len(S, L):
    """Elements per slice when a packed shard is cut into L blocks (Reading R6)."""
    return -(-S // L) if S > 0 else 0


def slice_of(x, S, L):
    """Slice index of packed-shard position x (Reading R6)."""
    return x // slice_len(S, L)


LANDING = "landing"    # Reading R5: landing-GPU order within a batch
RELATIVE = "relative"  # Reading R14: ascending relative index within a batch


def level2_batches(s, n_dest, M, L, order=LANDING):
    """Source nodes of slice s in the order their partials are added, batch
    by batch (Reading R5; Reading R14 with ``order=RELATIVE``).

    Relative indices are taken in batches of L -- batch b holds c in
    [b*L, (b+1)*L) -- because one read-and-add sums at most one partial per
    destination GPU; with M <= L there is a single batch.  Within a batch the
    destination's GPUs are visited g = 0, 1, ..., L-1, GPU g holding the
    partial of the batch's source whose slice s lands on it (none when c >= M);
    or, in the RELATIVE reading, the batch's sources are taken by ascending c.
    """
    if order not in (LANDING, RELATIVE):
        raise ValueError(order)
    batches = []
    for b in range(-(-M // L)):
        batch = []
        if order == LANDING:
            for g in range(L):
                for n_src in range(M):
                    c = relative_index(n_dest, n_src, M)
                    if b * L <= c < (b + 1) * L and landing_gpu(s, c, L) == g:
                        batch.append(n_src)
        else:
            for c in range(b * L, min(M, (b + 1) * L)):
                batch += [n_src for n_src in range(M) if relative_index(n_dest, n_src, M) == c]
        batches.append(batch)
    return batches


def level2_order(s, n_dest, M, L, order=LANDING):
    """All source nodes of slice s in addition order (batches concatenated)."""
    return [n for batch in level2_batches(s, n_dest, M, L, order) for n in batch]


# --------------------------------------------------------------------------
# Reduce-scatter: bf16 per-parameter gradients in, fp32 packed shards out.
# [Endgame] "Reduce-scatter: two levels of addition, the last one done by
# NVSwitch"; [Richland] "What shipped" (bf16 gradients consumed in place and
# reduced into fp32 shards; fp32 node partials); [Endgame] "What problem is it
# actually solving?" (sliced, zero-padded, upcast).
# --------------------------------------------------------------------------

def bf16_to_f32(bits):
    """Exact bf16 -> fp32 widening: the 16 bits become the high half of fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _node_partial(grad_slice_of, n_src, L, count):
    """Level 1: fp32 sum of node n_src's L local bf16 copies, l = 0..L-1 (R8)."""
    acc1 = np.zeros(count, dtype=np.float32)                 # Reading R4: start at +0.0
    for l in range(L):
        acc1 = acc1 + bf16_to_f32(grad_slice_of(n_src * L + l))
    return acc1


def rs_reduce(geo, grads, M, L, order=LANDING, ranks=None):
    """Reduce-scatter of grads[rank][p] (uint16 bf16 bits, R_p*Kp row-major).

    Returns N float32 arrays of S elements: rank r's packed fp32 gradient shard.
    ``order`` picks the level-2 reading (R5 or R14).  ``ranks`` (default: all)
    restricts the result to those destination ranks, in the order given; each
    rank's shard is computed exactly as in the full call.
    """
    N = geo.N
    if N != M * L:
        raise ValueError("N must equal M * L")
    shards = []
    for r in (range(N) if ranks is None else ranks):
        n_dest = r // L
        out = np.empty(geo.S, dtype=np.float32)
        for p in range(geo.P):
            e_p, o_p = geo.e[p], geo.o[p]
            v = valid_elems(geo, p, r)
            # Rows at or beyond R_p are zero padding (Reading R1).
            out[o_p + v:o_p + e_p] = np.float32(0.0)
            a = 0
            while a < v:
                s = slice_of(o_p + a, geo.S, L)
                b = min(v, (s + 1) * slice_len(geo.S, L) - o_p)
                src0 = r * e_p + a   # rank r's rows start at global row r*Rp

                def grad_slice_of(src_rank, p=p, src0=src0, count=b - a):
                    return grads[src_rank][p][src0:src0 + count]

                acc2 = np.zeros(b - a, dtype=np.float32)      # Reading R4
                for batch in level2_batches(s, n_dest, M, L, order):  # level 2, Reading R5
                    bsum = np.zeros(b - a, dtype=np.float32)
                    for n_src in batch:
                        bsum = bsum + _node_partial(grad_slice_of, n_src, L, b - a)
                    acc2 = acc2 + bsum
                out[o_p + a:o_p + b] = acc2
                a = b
        shards.append(out)
    return shards


def rs_element(geo, M, L, r, x, grad_at, order=LANDING):
    """One element of rank r's packed fp32 shard at position x, from scratch.

    ``grad_at(src_rank, p, idx)`` returns the bf16 bits of contributor
    src_rank's gradient of p at flat indices idx.  Same arithmetic and order as
    ``rs_reduce``; used for sampled checks at sizes the full oracle cannot hold.
    """
    p = next(q for q in range(geo.P) if geo.o[q] <= x < geo.o[q] + geo.e[q])
    e = x - geo.o[p]
    if e >= valid_elems(geo, p, r):
        return np.float32(0.0)
    s = slice_of(x, geo.S, L)
    idx = np.array([r * geo.e[p] + e], dtype=np.int64)
    acc2 = np.float32(0.0)
    for batch in level2_batches(s, r // L, M, L, order):
        bsum = np.float32(0.0)
        for n_src in batch:
            acc1 = np.float32(0.0)
            for l in range(L):
                acc1 = np.float32(acc1 + bf16_to_f32(grad_at(n_src * L + l, p, idx))[0])
            bsum = np.float32(bsum + acc1)
        acc2 = np.float32(acc2 + bsum)
    return acc2


# --------------------------------------------------------------------------
# All-gather with direct landing: each rank's packed shard piece is written
# once, at its final parameter-major address.  [Endgame] "All-gather:
# parameters land at their final address"; [Richland] "What shipped";
# [Abstract] Figure 1 and Figure 5(b).
# --------------------------------------------------------------------------

def ag_place(geo, shards, ranks=None, out=None):
    """All-gather of N packed shards (1-D arrays of S elements, any dtype).

    Returns P arrays: parameter p as its padded N*Rp x Kp block, flattened
    (Reading R9; the parameter proper is its first R_p rows).  ``out``
    (default: fresh arrays) receives the blocks instead; ``ranks`` (default:
    all) places only those ranks' pieces, leaving the rest of ``out`` as it is.
    """
    params = out if out is not None else [np.empty(geo.N * geo.e[p], dtype=shards[0].dtype)
                                          for p in range(geo.P)]
    for p in range(geo.P):
        e_p, o_p = geo.e[p], geo.o[p]
        block = params[p]
        for r in (range(geo.N) if ranks is None else ranks):
            block[r * e_p:(r + 1) * e_p] = shards[r][o_p:o_p + e_p]
    return params


def ag_element(geo, p, y, shard_at):
    """Element y of parameter p's gathered block, from ``shard_at(r, idx)``."""
    r, e = divmod(y, geo.e[p])
    return shard_at(r, np.array([geo.o[p] + e], dtype=np.int64))[0]


# --------------------------------------------------------------------------
# All-gather across nodes by recursive doubling ([Endgame] "All-gather:
# parameters land at their final address"; [Abstract] Figure 5).  On rail l
# (GPU l of every node) each node starts with its own piece; in round d
# (from 0) a node sends the first min(2^d, M - 2^d) pieces it has collected
# to the node 2^d lower and receives as many from the node 2^d higher
# (modulo M), appending them in arrival order.
# --------------------------------------------------------------------------

def rd_send_count(M, d):
    """Pieces each node sends in round d."""
    return min(2 ** d, M - 2 ** d)


def rd_rounds(M):
    """Rounds until every node holds every piece: rounds run while 2^d < M."""
    d = 0
    while 2 ** d < M:
        d += 1
    return d


def rd_simulate(M):
    """Collected pieces (source node numbers, in arrival order) of every node
    after each round: a list of rounds, each a list of M lists."""
    have = [[n] for n in range(M)]
    history = []
    for d in range(rd_rounds(M)):
        c = rd_send_count(M, d)
        sent = [list(have[n][:c]) for n in range(M)]          # what each node sends this round
        for n in range(M):
            have[n] = have[n] + sent[(n + 2 ** d) % M]        # received from the node 2^d higher
        history.append([list(h) for h in have])
    return history


def rd_stage_place(geo, stage, node, rail, L, params):
    """Place rail `rail`'s pieces from node `node`'s stage buffer into params.

    stage[k] is the packed shard held in stage slot k (arrival order), which
    is node (node + k) mod M's shard on this rail, i.e. rank
    ((node + k) mod M) * L + rail.  Every parameter receives its M pieces of
    this rail at their parameter-major offsets ([Abstract] Figure 5(b))."""
    M = len(stage)
    for p in range(geo.P):
        e_p, o_p = geo.e[p], geo.o[p]
        for k in range(M):
            r = ((node + k) % M) * L + rail
            params[p][r * e_p:(r + 1) * e_p] = stage[k][o_p:o_p + e_p]
    return params


# --------------------------------------------------------------------------
# Reduce-scatter in the pages' two stages, with the inbox made explicit
# ([Endgame] "Reduce-scatter: two levels of addition, the last one done by
# NVSwitch"; [Abstract] Figure 6).  Stage 1: on source node n_src, for
# destination node n_dest, the GPU that owns slice s sums the node's L local
# copies into one fp32 partial and sends it on its own line, so it lands on
# destination GPU g = (s - c) mod L, c = relative_index(n_dest, n_src, M).
# Stage 2: every destination rank adds the partials of its own block of each
# slice from the landing GPUs 0..L-1 in turn.  Inbox layout:
# inbox[n_dest][g][c] is an array of L*B floats (B = slice_len), rank
# n_dest*L + l_d's block at l_d*B.
# --------------------------------------------------------------------------

def rs_inbox(geo, grads, M, L):
    """Stage 1: every node partial, at the inbox position it lands on."""
    N, S = geo.N, geo.S
    B = slice_len(S, L)
    inbox = np.zeros((M, L, M, L * B), dtype=np.float32)
    for r in range(N):
        n_dest, l_dest = divmod(r, L)
        for p in range(geo.P):
            e_p, o_p = geo.e[p], geo.o[p]
            v = valid_elems(geo, p, r)
            a = 0
            while a < v:
                s = slice_of(o_p + a, S, L)
                b = min(v, (s + 1) * B - o_p)
                first = r * e_p + a             # rank r's rows start at global row r*Rp
                for n_src in range(M):
                    part = _node_partial(lambda k, p=p, s0=first, cnt=b - a: grads[k][p][s0:s0 + cnt],
                                         n_src, L, b - a)
                    c = relative_index(n_dest, n_src, M)
                    g = landing_gpu(s, c, L)
                    x0 = o_p + a - s * B
                    inbox[n_dest, g, c, l_dest * B + x0:l_dest * B + x0 + (b - a)] = part
                a = b
            # padding rows carry +0.0 partials (inbox starts at +0.0)
    return inbox


def rs_land(geo, inbox, M, L, order=LANDING):
    """Stage 2: each destination rank's shard from the landed partials
    (landing GPUs in turn; with ``order=RELATIVE``, relative indices in turn)."""
    N, S = geo.N, geo.S
    B = slice_len(S, L)
    shards = []
    for r in range(N):
        n_dest, l_dest = divmod(r, L)
        out = np.empty(S, dtype=np.float32)
        for s in range(L):
            lo, hi = s * B, min(S, (s + 1) * B)
            if lo >= hi:
                continue
            acc = np.zeros(hi - lo, dtype=np.float32)
            for b in range(-(-M // L)):                 # one read-and-add per batch of L sources
                bsum = np.zeros(hi - lo, dtype=np.float32)
                if order == LANDING:
                    for g in range(L):
                        c = b * L + (s - g) % L             # the batch's source whose slice s lands on GPU g
                        if c < M:
                            bsum = bsum + inbox[n_dest, g, c, l_dest * B:l_dest * B + (hi - lo)]
                else:
                    for c in range(b * L, min(M, (b + 1) * L)):
                        g = landing_gpu(s, c, L)            # where relative index c's slice s landed
                        bsum = bsum + inbox[n_dest, g, c, l_dest * B:l_dest * B + (hi - lo)]
                acc = acc + bsum
            out[lo:hi] = acc
        shards.append(out)
    return shards


# --------------------------------------------------------------------------
# Variants.
#   rs_finish: the reduce-scatter result optionally averaged over the N ranks
#   (divided by N in fp32, correctly rounded) and optionally accumulated into
#   the shard's previous value (old + result, one fp32 add after the sum).
#   ag_place_unpadded: the all-gather writing only each parameter's R_p real
#   rows.  slot_pack: Slot-Reuse -- each rank's bf16 gradients copied into the
#   all-gather slot it has just vacated, parameter p at offset N * op
#   ([Endgame] "Reduce-scatter: two levels of addition...", last paragraph;
#   [Abstract] Figure 7).
# --------------------------------------------------------------------------

def rs_finish(geo, sums, average=False, old=None):
    out = []
    for r in range(geo.N):
        x = sums[r]
        if average:
            x = (x / np.float32(geo.N)).astype(np.float32)
        if old is not None:
            x = (old[r] + x).astype(np.float32)
        out.append(x)
    return out


def ag_place_unpadded(geo, shards):
    params = ag_place(geo, shards)
    return [params[p][:geo.rows[p] * geo.Kp[p]] for p in range(geo.P)]


def slot_pack(geo, grads):
    """Each rank's gradients packed into its N*S-element slot at N*op."""
    slots = []
    for r in range(geo.N):
        slot = np.zeros(geo.N * geo.S, dtype=grads[r][0].dtype if geo.P else np.uint16)
        for p in range(geo.P):
            n = geo.rows[p] * geo.Kp[p]
            slot[geo.N * geo.o[p]:geo.N * geo.o[p] + n] = grads[r][p][:n]
        slots.append(slot)
    return slots

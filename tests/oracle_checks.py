"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``check_*`` raises AssertionError when the oracle disagrees with:
* the pages' worked examples (``tests/golden/*.json``, each citing its page),
* brute-force enumeration over full parameters on tiny groups,
* exact integer arithmetic (integer-valued bf16 sums are exact in fp32),
* the rigorous error bound of recursive fp32 summation against an fp64 sum,
* structural invariants (bijections, zero padding, round trips).

They are plain functions so that ``test_oracle_mutations`` can plant a
mistake in the oracle and confirm that at least one check notices it.
"""

import json
import os

import numpy as np

import oracle.tide_oracle as O
from synth import gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- layout pins

def check_hand_layout_example():
    g = _golden("layout_example.json")
    N = g["N"]
    for unit in (1, 64):   # one unit = one row of `unit` elements
        shapes = [(k * N, unit) for k in g["piece_units"]]
        geo = O.geometry(shapes, N)
        assert [x // unit for x in geo.e] == g["piece_units"]
        assert geo.S // unit == g["units_per_rank"]
        p, r = g["param"], g["rank"]
        assert O.rank_major_offset(geo, p, r) == g["rank_major_offset_units"] * unit
        assert O.param_major_offset(geo, p, r) == g["param_major_offset_units"] * unit


def _tiny_groups():
    """Small parameter groups with padding, 1-D/3-D/0-D shapes and rows < N."""
    groups = [
        ([(8, 64), (4, 64), (12, 64)], 1, 4),
        ([(5, 3), (1,), (7, 2, 2), (), (3, 1)], 2, 2),
        ([(13, 5), (2, 7), (17,), (6, 6)], 2, 3),
        ([(1, 9), (16, 8), (31, 3)], 4, 4),
        ([(11, 1), (3, 4)], 1, 1),
        ([(9, 5), (40, 3), (2, 2)], 3, 4),
        ([(16, 8)], 4, 4),
        ([(23, 3), (5, 5), (0, 4)], 2, 3),
        ([(19, 5), (3, 7), (40,)], 4, 2),      # more nodes than GPUs per node
        ([(31, 2), (6, 3)], 5, 2),
    ]
    return groups


def check_bruteforce_index_maps():
    """Row ownership and both offsets, enumerated element by element."""
    for shapes, M, L in _tiny_groups():
        N = M * L
        geo = O.geometry(shapes, N)
        seen_rank_major = np.zeros(N * geo.S, dtype=np.int64)
        seen_param_major = np.zeros(N * geo.S, dtype=np.int64)
        for p, shape in enumerate(shapes):
            shape = tuple(shape) or (1,)
            R = shape[0]
            K = int(np.prod(shape[1:])) if len(shape) > 1 else 1
            rp = -(-R // N)
            assert geo.Rp[p] == rp and geo.Kp[p] == K and geo.rows[p] == R
            for r in range(N):
                # rank r's piece of p holds rows [r*rp, (r+1)*rp), real or padding
                real = sum(1 for g in range(r * rp, (r + 1) * rp) if g < R)
                assert O.valid_elems(geo, p, r) == real * K
                for i in range(rp * K):
                    seen_rank_major[O.rank_major_offset(geo, p, r) + i] += 1
                    seen_param_major[O.param_major_offset(geo, p, r) + i] += 1
            for g in range(R):
                assert O.owner_of_row(geo, p, g) == g // rp
        # both layouts tile [0, N*S) exactly once
        assert (seen_rank_major == 1).all() and (seen_param_major == 1).all()
        # parameters are contiguous and in order in the parameter-major layout
        for p in range(geo.P):
            assert O.param_major_offset(geo, p, 0) == N * sum(geo.e[:p])


def check_no_padding_when_divisible():
    for shapes, N in [([(8192, 8192), (1024, 8192), (8192,)], 8),
                      ([(4096, 2048), (768, 2048), (2048,)], 16),
                      ([(5120, 5120), (13824, 5120), (5120,)], 64)]:
        geo = O.geometry(shapes, N)
        G = sum(int(np.prod(s)) for s in shapes)
        assert N * geo.S == G
    geo = O.geometry([(49, 3)], 48)   # 49 rows over 48 ranks: 2 rows each, 47 padding
    assert geo.Rp == [2] and 48 * geo.S - 49 * 3 == 47 * 3


def check_pack_buffer_size_identity():
    """Stock FSDP2's fp32 pack is twice the padded bf16 group (same element count)."""
    for shapes, M, L in _tiny_groups():
        N = M * L
        geo = O.geometry(shapes, N)
        padded_bf16_bytes = 2 * sum(N * geo.Rp[p] * geo.Kp[p] for p in range(geo.P))
        assert 4 * N * geo.S == 2 * padded_bf16_bytes


# ---------------------------------------------------------- Latin-square pins

def check_latin_square_figure6():
    g = _golden("latin_square_fig6.json")
    L = g["L"]
    for name, c in g["relative_index"].items():
        assert O.landing_gpu(0, c, L) == g["slice0_landing_gpu"][name]
    table = g["derived_by_hand"]["landing_gpu_by_slice_then_c"]
    for s in range(L):
        for c in range(g["M"]):
            assert O.landing_gpu(s, c, L) == table[s][c]
    # D, A, B, C numbered 0..3 as destination 0 and sources with indices 1..3
    M = g["M"]
    n_dest = 0
    for name, c in g["relative_index"].items():
        n_src = (n_dest - c) % M
        assert O.relative_index(n_dest, n_src, M) == c


def check_latin_property():
    """Every row and column of the seating table holds each source exactly once,
    and the source-side rule (GPU j sums slice (j+c) mod L and sends on line j)
    agrees with the landing rule."""
    for L in range(1, 9):
        for M in range(1, L + 1):
            for n_dest in range(M):
                for s in range(L):
                    gpus = [O.landing_gpu(s, O.relative_index(n_dest, n, M), L) for n in range(M)]
                    assert len(set(gpus)) == M
                for g in range(L):
                    srcs = [n for n in range(M) for s in range(L)
                            if O.landing_gpu(s, O.relative_index(n_dest, n, M), L) == g]
                    # source c lands on GPU g for exactly one slice, (g + c) mod L
                    assert sorted(srcs) == list(range(M))
            for c in range(M):
                for j in range(L):
                    s = O.handled_slice(j, c, L)
                    assert O.landing_gpu(s, c, L) == j


def check_level2_order_cases():
    cases = _golden("level2_order_cases.json")["cases"]
    for case in cases:
        for s, expect in enumerate(case["order_by_slice"]):
            assert O.level2_order(s, case["n_dest"], case["M"], case["L"]) == expect


def check_level2_batches_cases():
    for case in _golden("level2_order_cases.json")["batched_cases"]:
        for s, expect in enumerate(case["batches_by_slice"]):
            assert O.level2_batches(s, case["n_dest"], case["M"], case["L"]) == expect
    # with M <= L there is one batch, the landing-GPU order
    for case in _golden("level2_order_cases.json")["cases"]:
        for s, expect in enumerate(case["order_by_slice"]):
            assert O.level2_batches(s, case["n_dest"], case["M"], case["L"]) == [expect]


def check_level2_batches_property():
    """Every source appears once per slice; a batch never puts two sources on
    one landing GPU; batch b holds exactly relative indices [bL, bL+L) < M."""
    for L in range(1, 9):
        for M in range(1, 3 * L + 2):
            for n_dest in range(M):
                for s in range(L):
                    bs = O.level2_batches(s, n_dest, M, L)
                    flat = [n for b in bs for n in b]
                    assert sorted(flat) == list(range(M))
                    for b, batch in enumerate(bs):
                        cs = sorted(O.relative_index(n_dest, n, M) for n in batch)
                        assert cs == list(range(b * L, min(M, (b + 1) * L)))
                        gpus = [O.landing_gpu(s, O.relative_index(n_dest, n, M), L) for n in batch]
                        assert len(set(gpus)) == len(gpus) and gpus == sorted(gpus)


def check_relative_order_cases():
    """The alternative level-2 reading: ascending relative index per batch."""
    for case in _golden("level2_order_cases.json")["relative_order"]["cases"]:
        for s, expect in enumerate(case["batches_by_slice"]):
            assert O.level2_batches(s, case["n_dest"], case["M"], case["L"], O.RELATIVE) == expect
    for L in range(1, 9):
        for M in range(1, 3 * L + 2):
            for n_dest in range(M):
                for s in range(L):
                    bs = O.level2_batches(s, n_dest, M, L, O.RELATIVE)
                    assert [len(b) for b in bs] == [len(b) for b in O.level2_batches(s, n_dest, M, L)]
                    cs = [O.relative_index(n_dest, n, M) for b in bs for n in b]
                    assert cs == list(range(M))


def check_relative_order_cancellation():
    _check_cancellations(_golden("level2_order_cases.json")["relative_order"]["cancellations"], O.RELATIVE)


def check_level2_order_cancellation():
    """Order-sensitive sums whose fp32 results were worked out by hand."""
    _check_cancellations(_golden("level2_order_cases.json")["cancellations"], O.LANDING)


def _check_cancellations(groups, order):
    for g in groups:
        M, L = g["M"], g["L"]
        N = M * L
        R, K = g["shape"]
        geo = O.geometry([(R, K)], N)
        grads = [[np.zeros(R * K, dtype=np.uint16)] for _ in range(N)]
        for n, v in enumerate(g["V"]):
            bits = gen.f32_to_bf16_bits(np.full(K, v, dtype=np.float32))
            for row in g["planted_rows"]:
                grads[n * L][0][row * K:(row + 1) * K] = bits
        out = O.rs_reduce(geo, grads, M, L, order)
        for r in range(N):
            expect = np.array(g["expected_shard"].get(str(r), [g["other_ranks"]] * geo.S),
                              dtype=np.float32)
            assert np.array_equal(out[r], expect), (r, out[r], expect)
        # the single-element form and the two-stage form agree
        landed = O.rs_land(geo, O.rs_inbox(geo, grads, M, L), M, L, order)
        for r in range(N):
            assert np.array_equal(landed[r], out[r]), r
            for x in range(geo.S):
                val = O.rs_element(geo, M, L, r, x, lambda k, p, idx: grads[k][p][idx], order)
                assert val == out[r][x]


# ----------------------------------------------------------- reduction pins

def _int_grads(shapes, N, seed):
    grads = []
    for r in range(N):
        row = []
        for p, s in enumerate(shapes):
            n = int(np.prod(s)) if len(s) else 1
            row.append(gen.bf16_values(gen.tensor_key(seed, r, p),
                                       np.arange(n, dtype=np.uint64), gen.INTEGER))
        grads.append(row)
    return grads


def _bf16_as_float(bits):
    """Independent widening for the checks: scale the bf16 fields directly."""
    bits = np.asarray(bits, dtype=np.int64)
    sign = np.where(bits >> 15, -1.0, 1.0)
    exp = (bits >> 7) & 0xFF
    man = bits & 0x7F
    normal = sign * (1.0 + man / 128.0) * np.exp2(exp.astype(np.float64) - 127.0)
    sub = sign * (man / 128.0) * 2.0 ** -126
    return np.where(exp == 0, sub, normal)


def check_exact_integer_sums_bruteforce():
    """Integer-valued bf16 gradients: every output must be the exact integer sum,
    whatever the summation order; every padding slot must be +0.0."""
    for t, (shapes, M, L) in enumerate(_tiny_groups()):
        N = M * L
        geo = O.geometry(shapes, N)
        grads = _int_grads(shapes, N, seed=77 + t)
        out = O.rs_reduce(geo, grads, M, L)
        covered = [np.zeros(geo.S, dtype=bool) for _ in range(N)]
        for p, shape in enumerate(shapes):
            shape = tuple(shape) or (1,)
            R = shape[0]
            K = int(np.prod(shape[1:])) if len(shape) > 1 else 1
            rp = -(-R // N)
            total = sum(_bf16_as_float(grads[k][p]) for k in range(N)) if R * K else None
            for g in range(R):
                owner = g // rp
                for k in range(K):
                    pos = geo.o[p] + (g - owner * rp) * K + k
                    assert out[owner][pos] == total[g * K + k], (p, g, k)
                    covered[owner][pos] = True
        for r in range(N):
            pad = out[r][~covered[r]]
            assert (pad.view(np.uint32) == 0).all(), "padding must be +0.0"


def check_fp64_error_bound():
    """Random normal inputs: |oracle - fp64 sum| <= gamma_{(L-1)+(M-1)} * sum|x|."""
    u = 2.0 ** -24
    for shapes, M, L in [([(64, 33), (17, 5)], 2, 4), ([(128, 16)], 4, 4), ([(96, 7)], 1, 8),
                         ([(50, 9)], 3, 3)]:
        N = M * L
        geo = O.geometry(shapes, N)
        grads = [[gen.bf16_values(gen.tensor_key(5, r, p), np.arange(int(np.prod(s)), dtype=np.uint64),
                                  gen.OUTLIER) for p, s in enumerate(shapes)] for r in range(N)]
        out = O.rs_reduce(geo, grads, M, L)
        k = (L - 1) + (M - 1)
        gamma = k * u / (1 - k * u)
        for p, s in enumerate(shapes):
            R, K = s[0], int(np.prod(s[1:]))
            rp = geo.Rp[p]
            x = np.stack([_bf16_as_float(grads[r][p]) for r in range(N)])
            exact = x.sum(axis=0)
            mag = np.abs(x).sum(axis=0)
            for g in range(R):
                owner = g // rp
                a = geo.o[p] + (g - owner * rp) * K
                got = out[owner][a:a + K].astype(np.float64)
                assert (np.abs(got - exact[g * K:(g + 1) * K]) <= gamma * mag[g * K:(g + 1) * K]).all()
            # and the bound is not vacuous: the result is not just zero
            assert np.abs(np.concatenate([o for o in out])).max() > 0


def check_signed_zero_and_subnormals():
    """-0.0 inputs sum to +0.0 (accumulators start at +0.0); bf16 subnormals are kept."""
    N, M, L = 4, 2, 2
    geo = O.geometry([(4, 2)], N)
    neg0 = np.full(8, 0x8000, dtype=np.uint16)
    grads = [[neg0.copy()] for _ in range(N)]
    tiny = np.uint16(0x0001)            # smallest positive bf16 subnormal, 2^-133
    grads[0][0][0] = tiny
    grads[3][0][0] = tiny
    out = O.rs_reduce(geo, grads, M, L)
    assert out[0][0] == np.float32(2.0 ** -132)
    for r in range(N):
        rest = out[r].view(np.uint32)[1:] if r == 0 else out[r].view(np.uint32)
        assert (rest == 0).all()


# ---------------------------------------------------------------- AG pins

def check_ag_bruteforce():
    """Every element of every gathered parameter comes from the right rank/offset."""
    for shapes, M, L in _tiny_groups():
        N = M * L
        geo = O.geometry(shapes, N)
        shards = [np.arange(r * geo.S, (r + 1) * geo.S, dtype=np.int64) for r in range(N)]
        params = O.ag_place(geo, shards)
        hits = np.zeros(N * geo.S, dtype=np.int64)
        for p, shape in enumerate(shapes):
            shape = tuple(shape) or (1,)
            K = int(np.prod(shape[1:])) if len(shape) > 1 else 1
            rp = -(-shape[0] // N)
            assert params[p].size == N * rp * K
            for g in range(N * rp):
                owner = g // rp
                for k in range(K):
                    src = owner * geo.S + geo.o[p] + (g - owner * rp) * K + k
                    assert params[p][g * K + k] == src
                    hits[src] += 1
                    y = g * K + k
                    assert O.ag_element(geo, p, y, lambda r, idx: shards[r][idx]) == src
        assert (hits == 1).all()


def check_ag_of_rs_round_trip():
    """AG(RS(x)) in fp32 equals the full sum of x on real rows and 0 on padding."""
    for t, (shapes, M, L) in enumerate(_tiny_groups()):
        N = M * L
        geo = O.geometry(shapes, N)
        grads = _int_grads(shapes, N, seed=300 + t)
        full = O.ag_place(geo, O.rs_reduce(geo, grads, M, L))
        for p, shape in enumerate(shapes):
            shape = tuple(shape) or (1,)
            n = int(np.prod(shape))
            total = sum(_bf16_as_float(grads[k][p]) for k in range(N)) if n else np.zeros(0)
            assert np.array_equal(full[p][:n].astype(np.float64), total)
            assert (full[p][n:].view(np.uint32) == 0).all()


def check_staged_reduce_scatter_equals_fused():
    """The two-stage form (partials landed in the inbox, then added per
    landing GPU) gives the same bits as the direct definition, and every
    partial sits where the Latin square puts it."""
    for t, (shapes, M, L) in enumerate(_tiny_groups()):
        N = M * L
        geo = O.geometry(shapes, N)
        grads = [[gen.bf16_values(gen.tensor_key(900 + t, r, p), np.arange(int(np.prod(s)) if len(s) else 1,
                                                                          dtype=np.uint64), gen.OUTLIER)
                  for p, s in enumerate(shapes)] for r in range(N)]
        inbox = O.rs_inbox(geo, grads, M, L)
        for order in (O.LANDING, O.RELATIVE):
            staged = O.rs_land(geo, inbox, M, L, order)
            fused = O.rs_reduce(geo, grads, M, L, order)
            for r in range(N):
                assert np.array_equal(staged[r].view(np.uint32), fused[r].view(np.uint32)), (order, r)
        # within a batch of L relative indices each partial of a slice lands on its own GPU
        for n_dest in range(M):
            for s in range(L):
                for b in range(-(-M // L)):
                    cs = range(b * L, min(M, (b + 1) * L))
                    gpus = [O.landing_gpu(s, c, L) for c in cs]
                    assert len(set(gpus)) == len(cs)


def check_average_and_accumulate():
    """Average = the exact integer sum divided by N, correctly rounded to fp32;
    accumulate = old + result, exact for integers."""
    for t, (shapes, M, L) in enumerate(_tiny_groups()):
        N = M * L
        geo = O.geometry(shapes, N)
        grads = _int_grads(shapes, N, seed=500 + t)
        sums = O.rs_reduce(geo, grads, M, L)
        avg = O.rs_finish(geo, sums, average=True)
        old = [np.arange(geo.S, dtype=np.float32) - 7 for _ in range(N)]
        acc = O.rs_finish(geo, sums, old=old)
        both = O.rs_finish(geo, sums, average=True, old=old)
        for r in range(N):
            exact = sums[r].astype(np.float64)          # integer sums are exact in fp32
            assert np.array_equal(avg[r], (exact / N).astype(np.float32))
            assert np.array_equal(acc[r].astype(np.float64), old[r].astype(np.float64) + exact)
            assert np.array_equal(both[r], (old[r].astype(np.float64) + (exact / N).astype(np.float32)).astype(np.float32))


def check_unpadded_gather_and_slot_pack():
    for t, (shapes, M, L) in enumerate(_tiny_groups()):
        N = M * L
        geo = O.geometry(shapes, N)
        shards = [np.arange(r * geo.S, (r + 1) * geo.S, dtype=np.int64) for r in range(N)]
        full = O.ag_place(geo, shards)
        unp = O.ag_place_unpadded(geo, shards)
        for p, shape in enumerate(shapes):
            n = int(np.prod(shape)) if len(shape) else 1
            assert unp[p].size == n and np.array_equal(unp[p], full[p][:n])
        grads = _int_grads(shapes, N, seed=700 + t)
        slots = O.slot_pack(geo, grads)
        for r in range(N):
            for p, shape in enumerate(shapes):
                n = int(np.prod(shape)) if len(shape) else 1
                assert np.array_equal(slots[r][N * geo.o[p]:N * geo.o[p] + n], grads[r][p])
        # reducing from the slots gives the same shards as reducing in place
        from_slots = O.rs_reduce(geo, [[slots[r][N * geo.o[p]:N * geo.o[p] + geo.rows[p] * geo.Kp[p]]
                                        for p in range(geo.P)] for r in range(N)], M, L)
        direct = O.rs_reduce(geo, grads, M, L)
        assert all(np.array_equal(a.view(np.uint32), b.view(np.uint32)) for a, b in zip(from_slots, direct))


# ------------------------------------------------------ recursive doubling

def check_recursive_doubling_page_facts():
    g = _golden("recursive_doubling.json")
    for m, rounds in g["rounds"].items():
        assert O.rd_rounds(int(m)) == rounds
    assert O.rd_rounds(8) < g["ring_rounds"]["8"] == 8 - 1
    assert [O.rd_send_count(5, d) for d in range(O.rd_rounds(5))] == g["send_counts_M5"]


def check_recursive_doubling_bruteforce():
    """For M = 1..64: every node ends with every piece exactly once, after
    ceil(log2 M) rounds, and node n's k-th piece is node (n + k) mod M's."""
    import math
    for M in range(1, 65):
        hist = O.rd_simulate(M)
        assert len(hist) == (math.ceil(math.log2(M)) if M > 1 else 0)
        final = hist[-1] if hist else [[n] for n in range(M)]
        for n in range(M):
            assert final[n] == [(n + k) % M for k in range(M)], (M, n)
        for d, state in enumerate(hist):  # counts double until the last round
            assert all(len(h) == min(2 ** (d + 1), M) for h in state)


def check_stage_place_equals_direct_landing():
    """Placing every rail's stage buffer of one node gives the direct all-gather."""
    for shapes, M, L in _tiny_groups():
        N = M * L
        geo = O.geometry(shapes, N)
        shards = [np.arange(r * geo.S, (r + 1) * geo.S, dtype=np.int64) for r in range(N)]
        direct = O.ag_place(geo, shards)
        for node in range(M):
            params = [np.full(N * e, -1, dtype=np.int64) for e in geo.e]
            for rail in range(L):
                stage = [shards[((node + k) % M) * L + rail] for k in range(M)]
                O.rd_stage_place(geo, stage, node, rail, L, params)
            assert all(np.array_equal(a, b) for a, b in zip(params, direct))


def check_rs_buffer_accounting():
    """Table 8's stock-FSDP2 buffers are N x the output plus a small constant,
    as the N*S packed layout implies; and the staged reduce-scatter's inbox
    carries one fp32 partial per node where the raw cross-node data would be
    L bf16 copies, a quarter of the bytes at L = 8."""
    g = _golden("rs_buffer_accounting.json")
    for mib, extra in ((32, 0.03), (128, 0.12)):
        for row in (r for r in g["rows"] if r["output_mib"] == mib):
            N = row["gpus"]
            # P = 16 equal bf16 parameters whose per-rank fp32 shard is `mib` MiB
            S = mib * 2 ** 20 // 4
            geo = O.geometry([(N * (S // 16 // 1024), 1024)] * 16, N)
            assert 4 * geo.S == mib * 2 ** 20
            packed_gib = 4 * N * geo.S / 2 ** 30           # the packed fp32 reduce-scatter input
            assert abs(row["stock_buffer_gib"] - packed_gib - extra) < 0.006, (row, packed_gib)
    ratio = g["cross_node_ratio"]
    M, L = 2, ratio["L"]
    geo = O.geometry([(M * L * 4, 16)], M * L)
    grads = [[np.zeros(M * L * 4 * 16, dtype=np.uint16)] for _ in range(M * L)]
    inbox = O.rs_inbox(geo, grads, M, L)
    partial_bytes = 4 * inbox.size                     # fp32 partials the landing side reads
    raw_bytes = 2 * (M * L) * (M * L) * geo.S          # every contributor's bf16 slice, for every destination
    assert abs(partial_bytes / raw_bytes - ratio["ratio"]) < 1e-12


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]

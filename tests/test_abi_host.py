"""Host-side checks of libtide that need no GPU.

* the shared library loads and exports every function include/tide.h declares;
* plan geometry and the level-2 order table equal the oracle's, exactly;
* the work lists tile every output exactly once, with the right sources;
* invalid arguments return status codes (no GPU call is reached).
"""

import ctypes
import os
import re

import pytest
import torch

import fsdp_layout_aware_gb300 as tide
import oracle.tide_oracle as O
from synth import configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(tide_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert "tide_rs_reduce" in names and "tide_ag_place" in names and len(names) >= 10
    lib = ctypes.CDLL(tide.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


GROUPS = [
    ([(8, 64), (4, 64), (12, 64)], 1, 4),
    ([(5, 3), (1,), (7, 2, 2), (), (3, 1)], 2, 2),
    ([(13, 5), (2, 7), (17,), (6, 6)], 2, 3),
    ([(1, 9), (16, 8), (31, 3), (0, 5)], 4, 4),
    ([(49, 3), (97, 4095), (1, 1), (48, 1), (47, 1)], 6, 8),
    ([(100000, 3), (3, 70001)], 3, 5),
    # more nodes than GPUs per node: level-2 sources in batches of L
    ([(13, 5), (2, 7), (17,), (6, 6)], 4, 2),
    ([(9, 3), (33, 2), (1,)], 7, 3),
    ([(41, 5), (3, 9)], 12, 8),
]


def _check_plan_against_oracle(shapes, M, L):
    N = M * L
    geo = O.geometry(shapes, N)
    with tide.TidePlan(shapes, N, M, L) as plan:
        assert plan.S == geo.S
        assert plan.rows == geo.rows and plan.Rp == geo.Rp and plan.Kp == geo.Kp and plan.o == geo.o
        for n_dest in range(M):
            for s in range(L):
                assert plan.level2_order(n_dest, s) == O.level2_order(s, n_dest, M, L)
        _check_rs_items(plan, geo, M, L)
        _check_ag_items(plan, geo)


def _rs_chunk(N):
    """Elements per RS item: the power of two at or below 128 Ki / N, in [2048, 8192]."""
    c = 8192
    while c > 2048 and c * N > 1 << 17:
        c //= 2
    return c


def _check_rs_items(plan, geo, M, L):
    N = geo.N
    chunk = _rs_chunk(N)
    cover = [bytearray(geo.S) for _ in range(N)]
    for it in plan.items(0):
        p, r, n, dst = it["p"], it["r"], it["n"], it["dst_off"]
        assert n > 0 and geo.o[p] <= dst and dst + n <= geo.o[p] + geo.e[p]
        e0 = dst - geo.o[p]
        v = O.valid_elems(geo, p, r)
        assert O.slice_of(dst, geo.S, L) == O.slice_of(dst + n - 1, geo.S, L)   # one slice per item
        if it["kind"] == 0:
            assert e0 + n <= v
            assert it["src_off"] == r * geo.e[p] + e0     # contributors' rows r*Rp...
            # never across a chunk boundary of the contributors' index space
            assert it["src_off"] // chunk == (it["src_off"] + n - 1) // chunk
        else:
            assert it["kind"] == 1 and e0 >= v
        for x in range(dst, dst + n):
            cover[r][x] += 1
    for r in range(N):
        assert all(c == 1 for c in cover[r]), f"rank {r}: RS items must tile the shard exactly once"


def _check_ag_items(plan, geo):
    N = geo.N
    hits = bytearray(N * geo.S)
    for it in plan.items(1):
        p, r, n = it["p"], it["r"], it["n"]
        e0 = it["dst_off"] - r * geo.e[p]
        assert 0 <= e0 and e0 + n <= geo.e[p]
        assert it["src_off"] == geo.o[p] + e0
        base = O.param_major_offset(geo, p, r) + e0
        for y in range(base, base + n):
            hits[y] += 1
    assert all(h == 1 for h in hits), "AG items must tile the gathered group exactly once"


@pytest.mark.parametrize("shapes,M,L", GROUPS)
def test_plan_matches_oracle(shapes, M, L):
    _check_plan_against_oracle(shapes, M, L)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_workload_geometry_matches_oracle(cfg):
    w = configs.get(cfg)
    geo = O.geometry(w.shapes, w.N)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        assert (plan.S, plan.Rp, plan.Kp, plan.o) == (geo.S, geo.Rp, geo.Kp, geo.o)
        for n_dest in range(w.M):
            for s in range(w.L):
                assert plan.level2_order(n_dest, s) == O.level2_order(s, n_dest, w.M, w.L)
        items = plan.items(0)
        # per destination rank, item lengths add up to the shard; valid items
        # hold at most one chunk (8192 elements for N <= 16, 2048 for N >= 48)
        per_rank = [0] * w.N
        for it in items:
            per_rank[it["r"]] += it["n"]
            if it["kind"] == 0:
                assert it["n"] <= _rs_chunk(w.N)
        assert per_rank == [geo.S] * w.N
        assert _rs_chunk(w.N) == {1: 8192, 2: 8192, 3: 8192, 4: 2048, 5: 2048}[cfg]
        if cfg == 1:
            _check_rs_items(plan, geo, w.M, w.L)
            _check_ag_items(plan, geo)


def test_all_level2_orders_small_groups():
    for L in range(1, 9):
        for M in list(range(1, 2 * L + 2)) + [32]:
            with tide.TidePlan([(2 * M * L, 3)], M * L, M, L) as plan:
                for n_dest in range(M):
                    for s in range(L):
                        assert plan.level2_order(n_dest, s) == O.level2_order(s, n_dest, M, L)
                plan.set_option(tide.TIDE_OPT_SUM_ORDER, tide.TIDE_SUM_RELATIVE)
                for n_dest in range(M):
                    for s in range(L):
                        assert plan.level2_order(n_dest, s) == O.level2_order(s, n_dest, M, L, O.RELATIVE)
                plan.set_option(tide.TIDE_OPT_SUM_ORDER, tide.TIDE_SUM_LANDING)
                assert plan.level2_order(0, L - 1) == O.level2_order(L - 1, 0, M, L)


@pytest.mark.parametrize("shapes,N,M,L,status", [
    ([(4, 4)], 4, 2, 3, 1),      # N != M*L
    ([(4, 4)], 18, 2, 9, 1),     # L > 8
    ([(4, 4)], 0, 0, 4, 1),      # M < 1
    ([(4, 4)], 66, 33, 2, 1),    # M > 32
    ([(-1, 4)], 4, 1, 4, 1),     # negative dim
    ([(1,) * 9], 4, 1, 4, 1),    # ndim > 8
    ([(4, 1 << 40, 1 << 40)], 4, 1, 4, 3),   # row length overflow
])
def test_plan_create_rejects(shapes, N, M, L, status):
    with pytest.raises(tide.TideError) as err:
        tide.tide_plan_create(shapes, N, M, L)
    assert err.value.status == status


def test_empty_group_is_a_no_op():
    with tide.TidePlan([], 4, 1, 4) as plan:
        assert plan.S == 0 and plan.items(0) == [] and plan.items(1) == []
        plan.rs_reduce([], [None] * 4, stream=0)        # nothing to do: OK without a GPU
        plan.ag_place([None] * 4, [], 2, stream=0)
    with tide.TidePlan([(0, 7), (0,)], 8, 1, 8) as plan:
        assert plan.S == 0
        plan.rs_reduce([None] * 16, [None] * 8, stream=0)


def test_call_argument_errors_need_no_gpu():
    with tide.TidePlan([(8, 64), (4, 64), (12, 64)], 4, 1, 4) as plan:
        good = [0x10000 * (i + 1) for i in range(12)]
        shards = [0x1000000 * (r + 1) for r in range(4)]
        cases = [
            (lambda: plan.rs_reduce(good, shards[:3] + [None], stream=0), 1),
            (lambda: plan.rs_reduce(good[:5] + [None] + good[6:], shards, stream=0), 1),
            (lambda: plan.rs_reduce(good[:5] + [good[5] + 1] + good[6:], shards, stream=0), 2),
            (lambda: plan.rs_reduce(good, [shards[0] + 2] + shards[1:], stream=0), 2),
            (lambda: plan.ag_place(shards, good[:3], 3, stream=0), 1),
            (lambda: plan.ag_place(shards, [good[0] + 2] + good[1:3], 4, stream=0), 2),
            (lambda: plan.ag_place([shards[0] + 1] + shards[1:], good[:3], 2, stream=0), 2),
            (lambda: plan.ag_place(shards, [None] + good[1:3], 2, stream=0), 1),
        ]
        for fn, status in cases:
            with pytest.raises(tide.TideError) as err:
                fn()
            assert err.value.status == status
    with pytest.raises(tide.TideError) as err:
        tide.tide_rs_reduce(None, [], [], 0)
    assert err.value.status == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error path")
def test_cuda_failure_is_a_status_without_a_gpu():
    with tide.TidePlan([(8, 64)], 4, 1, 4) as plan:
        with pytest.raises(tide.TideError) as err:
            plan.rs_reduce([0x10000 * (i + 1) for i in range(4)], [0x1000000 * (r + 1) for r in range(4)], stream=0)
        assert err.value.status == 5


def test_plan_options_validate_without_a_gpu():
    with tide.TidePlan([(8, 64)], 4, 1, 4) as plan:
        plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1)
        plan.set_option(tide.TIDE_OPT_RS_KERNEL, 0)
        plan.set_option(tide.TIDE_OPT_WAIT_LIMIT_NS, 1000)
        plan.set_option(tide.TIDE_OPT_TEST_DROP_TILE, -1)
        plan.check()   # never ran on a device: nothing to report
        for opt, val in [(tide.TIDE_OPT_RS_KERNEL, 2), (tide.TIDE_OPT_WAIT_LIMIT_NS, 0),
                         (tide.TIDE_OPT_TEST_DROP_TILE, -2), (tide.TIDE_OPT_SUM_ORDER, 2),
                         (tide.TIDE_OPT_RD_EXCHANGE, 2), (tide.TIDE_OPT_CHECK_OVERLAP, 3),
                         (tide.TIDE_OPT_AG_TRANSPORT, 3), (tide.TIDE_OPT_AG_TRANSPORT, -1), (99, 0)]:
            with pytest.raises(tide.TideError) as err:
                plan.set_option(opt, val)
            assert err.value.status == 1


def test_pointer_array_is_passed_through():
    arr = tide.pointer_array([0x1000, None, 0x2000])
    assert len(arr) == 3 and arr.arr[0] == 0x1000 and arr.arr[1] is None and arr.arr[2] == 0x2000
    with tide.TidePlan([(8, 64)], 4, 1, 4) as plan:
        bad = tide.pointer_array([0x10000, 0x10001, 0x10000, 0x10000])   # misaligned gradient
        with pytest.raises(tide.TideError) as err:
            plan.rs_reduce(bad, tide.pointer_array([0x100000] * 4), stream=0)
        assert err.value.status == 2


def test_recursive_doubling_schedule_matches_oracle():
    for M in range(1, 65):
        assert tide.tide_rd_rounds(M) == O.rd_rounds(M)
        for d in range(O.rd_rounds(M)):
            assert tide.tide_rd_send_count(M, d) == O.rd_send_count(M, d)
        assert tide.tide_rd_send_count(M, O.rd_rounds(M)) == -1
    assert tide.tide_rd_rounds(0) == -1


def test_staged_rs_arguments_without_a_gpu():
    with tide.TidePlan([(8, 64), (4, 64), (12, 64)], 4, 2, 2) as plan:
        B = -(-plan.S // 2)
        assert tide.tide_plan_inbox_elems(plan.handle) == 2 * 2 * 2 * 2 * B
        good = [0x10000 * (i + 1) for i in range(12)]
        shards = [0x1000000 * (r + 1) for r in range(4)]
        for inbox, sums, lands, status in [(None, 0, 0, 1), (0x2000002, 0, 0, 2), (0x2000000, -1, 0, 1),
                                           (0x2000000, 0, -4, 1)]:
            with pytest.raises(tide.TideError) as err:
                tide.tide_rs_staged(plan.handle, good, shards, inbox, sums, lands, stream=0)
            assert err.value.status == status
    with tide.TidePlan([], 4, 1, 4) as plan:
        assert tide.tide_plan_inbox_elems(plan.handle) == 0


def _overlap_status(fn):
    with pytest.raises(tide.TideError) as err:
        fn()
    return err.value.status, str(err.value)


# Both overlap tests pass fake pointers; a case the check missed would go on
# to launch kernels on them, so they run only where there is no device.
@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers must never reach a device")
def test_overlap_check_rejects_before_any_device_work():
    """TIDE_OPT_CHECK_OVERLAP: outputs overlapping inputs or each other are
    rejected on the host, before any CUDA call."""
    shapes = [(8, 64), (4, 64), (12, 64)]          # N = 4: S = 2*64 + 64 + 3*64 = 384
    with tide.TidePlan(shapes, 4, 2, 2) as plan:
        plan.set_option(tide.TIDE_OPT_CHECK_OVERLAP, 1)
        S = plan.S
        grads = [0x100000 * (i + 1) for i in range(12)]             # 1 MiB apart, each <= 1.5 KiB
        shards = [0x4000000 + 0x10000 * r for r in range(4)]
        # a shard starting inside rank 1's gradient of parameter 2
        bad = list(shards)
        bad[3] = grads[1 * 3 + 2] + 64
        st, msg = _overlap_status(lambda: plan.rs_reduce(grads, bad, stream=0))
        assert st == 1 and "overlaps input grads[5]" in msg
        # two shards overlapping each other (4*S bytes each)
        bad = list(shards)
        bad[2] = shards[1] + 4 * S - 4
        st, msg = _overlap_status(lambda: plan.rs_reduce(grads, bad, stream=0))
        assert st == 1 and "shards[1]" in msg and "shards[2]" in msg
        # the staged inbox overlapping a shard
        st, msg = _overlap_status(lambda: tide.tide_rs_staged(plan.handle, grads, shards, shards[0] + 16, 0, 0, 0))
        assert st == 1 and "inbox" in msg
        # the no-alloc entry point checks too
        bad = list(shards)
        bad[0] = grads[0]
        st, _ = _overlap_status(lambda: tide.tide_rs_reduce_noalloc(plan.handle, grads, bad, stream=0))
        assert st == 1
        # all-gather: parameter 2's block (4 ranks x 3 rows x 64 x 2 bytes)
        # reaching 8 bytes into shard 0
        ag_in = [0x8000000 + 0x10000 * r for r in range(4)]          # 2*S bytes each
        params = [0x9000000, 0x9100000, ag_in[0] - 4 * 3 * 64 * 2 + 8]
        st, msg = _overlap_status(lambda: plan.ag_place(ag_in, params, 2, stream=0))
        assert st == 1 and "params[2]" in msg and "shards[0]" in msg
        # Slot-Reuse pack: a slot over a gradient
        slots = [0xA000000 + 0x100000 * r for r in range(4)]
        slots[1] = grads[7] - 8
        st, msg = _overlap_status(lambda: tide.tide_slot_pack(plan.handle, grads, slots, 0))
        assert st == 1 and "slots[1]" in msg
        # stage placement: a parameter inside the stage buffer
        stage = 0xB000000
        st, msg = _overlap_status(lambda: tide.tide_ag_stage_place(plan.handle, stage, 0, 0,
                                                                   [stage + 2, 0xC000000, 0xD000000], 2, 0))
        assert st == 1 and "stage" in msg
        plan.set_option(tide.TIDE_OPT_CHECK_OVERLAP, 0)
    # a padded parameter (10 rows over 4 ranks: 12 padded rows, 1536 bytes)
    # whose real rows (1280 bytes) end where shard 0 starts
    with tide.TidePlan([(10, 64), (4, 64), (12, 64)], 4, 2, 2) as plan:
        plan.set_option(tide.TIDE_OPT_CHECK_OVERLAP, 1)
        ag_in = [0x8000000 + 0x10000 * r for r in range(4)]
        params = [ag_in[0] - 10 * 64 * 2, 0x9000000, 0x9100000]
        st, msg = _overlap_status(lambda: plan.ag_place(ag_in, params, 2, stream=0))
        assert st == 1 and "params[0]" in msg


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers must never reach a device")
def test_overlap_check_lets_disjoint_and_shared_inputs_through():
    """Inputs may overlap each other; disjoint outputs pass the check and the
    call goes on (to the missing device: status 5)."""
    with tide.TidePlan([(8, 64), (4, 64), (12, 64)], 4, 2, 2) as plan:
        plan.set_option(tide.TIDE_OPT_CHECK_OVERLAP, 1)
        grads = [0x100000] * 12                                      # every rank reads one buffer
        shards = [0x4000000 + 0x10000 * r for r in range(4)]
        st, _ = _overlap_status(lambda: plan.rs_reduce(grads, shards, stream=0))
        assert st == 5
    # the unpadded destination of the padded parameter above stops in time
    with tide.TidePlan([(10, 64), (4, 64), (12, 64)], 4, 2, 2) as plan:
        plan.set_option(tide.TIDE_OPT_CHECK_OVERLAP, 1)
        plan.set_option(tide.TIDE_OPT_AG_UNPADDED, 1)
        ag_in = [0x8000000 + 0x10000 * r for r in range(4)]
        params = [ag_in[0] - 10 * 64 * 2, 0x9000000, 0x9100000]
        st, _ = _overlap_status(lambda: plan.ag_place(ag_in, params, 2, stream=0))
        assert st == 5


def _check_ag_bulk_split(plan, geo, N):
    """The bulk-copy transport's split of the all-gather work: every chunk is
    16-byte aligned at both ends (with 16-byte aligned bases), a multiple of
    16 bytes, at most 32 KiB and inside its shard and block; chunks and the
    rest tile every all-gather item exactly once."""
    hits = {}
    for which in (2, 3):
        for it in plan.items(which):
            p, r, n, so, do = it["p"], it["r"], it["n"], it["src_off"], it["dst_off"]
            assert n > 0 and 0 <= so and so + n <= geo.S and 0 <= do and do + n <= N * geo.e[p]
            assert do - r * geo.e[p] == so - geo.o[p]          # the direct-landing map
            if which == 2:
                assert (2 * so) % 16 == 0 and (2 * do) % 16 == 0 and (2 * n) % 16 == 0 and 2 * n <= 32768
            for y in range(do, do + n):
                hits[(p, y)] = hits.get((p, y), 0) + 1
    assert all(h == 1 for h in hits.values())
    assert sum(hits.values()) == N * geo.S


@pytest.mark.parametrize("shapes,M,L", GROUPS)
def test_ag_bulk_split_small_groups(shapes, M, L):
    N = M * L
    geo = O.geometry(shapes, N)
    with tide.TidePlan(shapes, N, M, L) as plan:
        _check_ag_bulk_split(plan, geo, N)


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_ag_bulk_split_workloads(cfg):
    """Full-size groups, checked by counting instead of element by element."""
    w = configs.get(cfg)
    geo = O.geometry(w.shapes, w.N)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        bulk, rest = plan.items(2), plan.items(3)
        total = 0
        for it in bulk:
            assert (2 * it["src_off"]) % 16 == 0 and (2 * it["dst_off"]) % 16 == 0
            assert (2 * it["n"]) % 16 == 0 and 0 < 2 * it["n"] <= 32768
            assert it["src_off"] + it["n"] <= geo.S and it["dst_off"] + it["n"] <= w.N * geo.e[it["p"]]
            total += it["n"]
        for it in rest:
            assert it["n"] > 0 and it["src_off"] + it["n"] <= geo.S
            total += it["n"]
        assert total == w.N * geo.S
        if cfg in (2, 3, 4):          # even row lengths throughout: nearly everything goes by bulk copy
            assert sum(it["n"] for it in rest) < 0.01 * total


def test_last_launches_without_a_gpu():
    with tide.TidePlan([(8, 64)], 4, 1, 4) as plan:
        assert plan.last_launches() == 0          # nothing ran yet
    assert tide.TIDE_AG_SM == 0 and tide.TIDE_AG_BULK == 2


def test_all_rails_arguments_without_a_gpu():
    """Argument errors of the every-rail calls come back before any device work."""
    with tide.TidePlan([(8, 64), (4, 64), (12, 64)], 4, 2, 2) as plan:
        stages = [0x1000000 * (i + 1) for i in range(4)]      # rail l's node n at l*M + n
        shards = [0x10000000 * (r + 1) for r in range(4)]
        cases = [
            (lambda: tide.tide_ag_rd_exchange_rails(plan.handle, stages[:3] + [None], 2, 0), 1),
            (lambda: tide.tide_ag_rd_exchange_rails(plan.handle, stages[:3] + [stages[1]], 2, 0), 1),
            (lambda: tide.tide_ag_rd_exchange_rails(plan.handle, stages[:3] + [stages[3] + 1], 2, 0), 2),
            (lambda: tide.tide_ag_rd_exchange_rails(plan.handle, stages, 3, 0), 1),
            (lambda: tide.tide_ag_stage_init(plan.handle, shards, stages[:3] + [None], 2, 0), 1),
            (lambda: tide.tide_ag_stage_init(plan.handle, [None] + shards[1:], stages, 2, 0), 1),
            (lambda: tide.tide_ag_stage_init(plan.handle, shards, [stages[0] + 2] + stages[1:], 4, 0), 2),
            (lambda: tide.tide_ag_stage_init(plan.handle, [shards[0] + 1] + shards[1:], stages, 2, 0), 2),
            (lambda: tide.tide_ag_stage_init(plan.handle, shards, stages, 8, 0), 1),
        ]
        for fn, status in cases:
            with pytest.raises(tide.TideError) as err:
                fn()
            assert err.value.status == status
    with tide.TidePlan([(8, 64)], 4, 1, 4) as plan:   # one node: nothing to exchange
        tide.tide_ag_rd_exchange_rails(plan.handle, [None] * 4, 2, 0)
    with tide.TidePlan([], 4, 2, 2) as plan:          # empty group: nothing to copy
        tide.tide_ag_stage_init(plan.handle, [None] * 4, [None] * 4, 2, 0)
        tide.tide_ag_rd_exchange_rails(plan.handle, [None] * 4, 2, 0)


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers must never reach a device")
def test_all_rails_overlap_check():
    with tide.TidePlan([(8, 64), (4, 64), (12, 64)], 4, 2, 2) as plan:
        plan.set_option(tide.TIDE_OPT_CHECK_OVERLAP, 1)
        S = plan.S
        stages = [0x1000000 * (i + 1) for i in range(4)]
        stages[2] = stages[1] + 2 * S * 2 - 2               # last element of buffer 1
        st, msg = _overlap_status(lambda: tide.tide_ag_rd_exchange_rails(plan.handle, stages, 2, 0))
        assert st == 1 and "stages" in msg
        stages = [0x1000000 * (i + 1) for i in range(4)]
        shards = [0x10000000 * (r + 1) for r in range(4)]
        shards[3] = stages[0] + 2                            # a shard inside slot 0 of buffer 0
        st, msg = _overlap_status(lambda: tide.tide_ag_stage_init(plan.handle, shards, stages, 2, 0))
        assert st == 1 and "shards[3]" in msg and "stages[0]" in msg


def test_stage_shard_pointers_follow_the_slot_rule():
    """stage_shard_pointers(node) must hand rank r the slot k of rail r % L
    whose content the exchange defines: slot k of node `node` holds rank
    ((node + k) mod M) * L + rail."""
    for M, L, S, eb in [(1, 4, 10, 2), (3, 2, 7, 2), (5, 3, 11, 4), (8, 8, 3, 2)]:
        stages = [0x10000000 * (i + 1) for i in range(L * M)]
        for node in range(M):
            ptrs = tide.stage_shard_pointers(stages, node, M, L, S, eb)
            assert len(ptrs) == M * L
            for r, a in enumerate(ptrs):
                i = next(j for j, b in enumerate(stages) if b <= a < b + M * S * eb)
                k, rem = divmod(a - stages[i], S * eb)
                assert rem == 0 and i == (r % L) * M + node
                assert ((node + k) % M) * L + r % L == r

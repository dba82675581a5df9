"""GPU parity with more nodes than GPUs per node (M > L), and of the
alternative level-2 reading (ascending relative index).

The level-2 sum then runs in batches of L source nodes, one read-and-add per
batch, and the batch sums are added in ascending batch order ("Reduce-scatter:
two levels of addition, the last one done by NVSwitch" in "The Endgame of FSDP
Communication": machines beyond what one read-and-add takes go in batches).
Every kernel that reduces must equal the oracle bit for bit; each case is also
checked to be one where a flat (unbatched) order gives different bits, so the
comparison has the power to see a missing batch boundary.
"""

import numpy as np
import pytest
import torch

import fsdp_layout_aware_gb300 as tide
import oracle.tide_oracle as O
from synth import configs, gen

from gpu_common import DEV, f32_bits, f32_guarded, host_grads, oracle_rs, to_dev_u16

pytestmark = pytest.mark.gpu

GUARD = 29


def _cases():
    ragged = [(5, 3), (1,), (7, 2, 2), (), (3, 1), (13, 5), (2, 7), (17,), (100, 33), (0, 4), (1031, 257)]
    # near-zero normal values next to outliers span enough exponents that the
    # fp32 sums round, so the order of the additions shows in the bits
    mixed = [gen.NORMAL if p % 2 else gen.OUTLIER for p in range(len(ragged))]
    ws = [
        configs.Workload("nodes4_gpus2", 8, 4, 2, ragged, mixed, sigma=1e-3, seed=401),
        configs.Workload("nodes5_gpus3", 15, 5, 3, ragged, mixed, sigma=1e-3, seed=402),
        configs.scaled(configs.get(4), row_div=1024, N=32, M=8, L=4, name="wan22dit_rows/1024_nodes8_gpus4"),
        configs.Workload("nodes12_gpus8", 96, 12, 8, [(200, 96), (31, 7), (1,), (96, 128)],
                         [gen.OUTLIER, gen.INTEGER, gen.UNIFORM, gen.NORMAL], sigma=1e-2, seed=403),
        configs.Workload("nodes32_gpus8", 256, 32, 8, [(300, 40), (7, 3), (256, 16)],
                         [gen.OUTLIER] * 3, sigma=1e-3, seed=404),
        configs.Workload("nodes16_gpus1", 16, 16, 1, [(77, 9), (16, 16)], [gen.OUTLIER] * 2, sigma=1e-3, seed=405),
    ]
    return ws


CASES = _cases()


@pytest.fixture(scope="module")
def oracle_cache():
    return {}


def _inputs(w, cache):
    if w.name not in cache:
        grads = host_grads(w)
        geo, expect = oracle_rs(w, grads)
        cache[w.name] = (grads, geo, expect)
    return cache[w.name]


def _flat(w, grads, monkeypatch):
    """The oracle's result with all M sources in one batch: what a kernel that
    missed the batch boundaries would produce."""
    orig = O.level2_batches
    with monkeypatch.context() as m:
        m.setattr(O, "level2_batches",
                  lambda s, n, M, L, order=O.LANDING: [[x for b in orig(s, n, M, L, order) for x in b]])
        return O.rs_reduce(O.geometry(w.shapes, w.N), grads, w.M, w.L)


def _device(w, grads):
    return [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]


def _flat_list(w, dev):
    return [dev[r][p] for r in range(w.N) for p in range(w.P)]


def _assert_equal(w, outs, expect, guards=True):
    for r in range(w.N):
        got = f32_bits(outs[r][0] if guards else outs[r])
        bad = np.nonzero(got != expect[r].view(np.uint32))[0]
        assert bad.size == 0, f"{w.name} rank {r}: {bad.size} mismatches, first at {bad[:5]}"
        if guards:
            g = f32_bits(outs[r][1])
            assert (g[:GUARD] == 0x7FC00000).all() and (g[GUARD + expect[r].size:] == 0x7FC00000).all()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_batched_order_is_distinguishable(w, oracle_cache, monkeypatch):
    """Host-only sanity of the cases: batching changes at least one bit
    (skipped for L = 1, where a batch of one source adds +0.0 + x = x)."""
    if w.L == 1:
        pytest.skip("one source per batch: batched and flat sums agree")
    grads, geo, expect = _inputs(w, oracle_cache)
    flat = _flat(w, grads, monkeypatch)
    assert any(not np.array_equal(flat[r].view(np.uint32), expect[r].view(np.uint32)) for r in range(w.N))


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("kernel", ["fused", "staged", "noalloc", "bulk"])
def test_rs_many_nodes_bit_exact(w, kernel, oracle_cache):
    grads, geo, expect = _inputs(w, oracle_cache)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        for n_dest in range(w.M):
            for s in range(w.L):
                assert plan.level2_order(n_dest, s) == O.level2_order(s, n_dest, w.M, w.L)
        dev = _device(w, grads)
        flat = _flat_list(w, dev)
        outs = [f32_guarded(geo.S, GUARD, GUARD) for _ in range(w.N)]
        shards = [o[0] for o in outs]
        if kernel == "bulk":
            plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1)
            if w.M > 8:
                with pytest.raises(tide.TideError) as err:
                    plan.rs_reduce(flat, shards)
                assert err.value.status == 6
                return
            plan.rs_reduce(flat, shards)
        elif kernel == "staged":
            inbox = torch.full((tide.tide_plan_inbox_elems(plan.handle),), float("nan"), dtype=torch.float32,
                               device=DEV)
            tide.tide_rs_staged(plan.handle, flat, shards, inbox, 16, 4)
        elif kernel == "noalloc":
            tide.tide_rs_reduce_noalloc(plan.handle, flat, shards)
        else:
            plan.rs_reduce(flat, shards)
        plan.check()
        _assert_equal(w, outs, expect)


ORDER_CASES = [
    configs.Workload("ragged_3x4", 12, 3, 4, [(5, 3), (1,), (7, 2, 2), (), (13, 5), (100, 33), (1031, 257)],
                     [gen.NORMAL if p % 2 else gen.OUTLIER for p in range(7)], sigma=1e-3, seed=406),
    configs.scaled(configs.get(4), row_div=1024, name="wan22dit_rows/1024"),
    CASES[1], CASES[3],   # (with L = 2 the two readings coincide: a batch of two adds a + b either way)
]


def _relative(w, cache):
    key = ("relative", w.name)
    if key not in cache:
        grads, geo, landing = _inputs(w, cache)
        cache[key] = O.rs_reduce(geo, grads, w.M, w.L, O.RELATIVE)
    return cache[key]


@pytest.mark.parametrize("w", ORDER_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("kernel", ["fused", "staged", "noalloc", "bulk"])
def test_rs_relative_order_bit_exact(w, kernel, oracle_cache):
    """TIDE_OPT_SUM_ORDER = TIDE_SUM_RELATIVE: every kernel follows the
    ascending-relative-index reading bit for bit, and the cases are ones where
    the two readings give different bits."""
    grads, geo, landing = _inputs(w, oracle_cache)
    expect = _relative(w, oracle_cache)
    assert any(not np.array_equal(expect[r].view(np.uint32), landing[r].view(np.uint32)) for r in range(w.N))
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_SUM_ORDER, tide.TIDE_SUM_RELATIVE)
        flat = _flat_list(w, _device(w, grads))
        outs = [f32_guarded(geo.S, GUARD, GUARD) for _ in range(w.N)]
        shards = [o[0] for o in outs]
        if kernel == "bulk":
            if w.M > 8:
                pytest.skip("the bulk kernel takes at most 8 nodes")
            plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1)
            plan.rs_reduce(flat, shards)
        elif kernel == "staged":
            inbox = torch.full((tide.tide_plan_inbox_elems(plan.handle),), float("nan"), dtype=torch.float32,
                               device=DEV)
            tide.tide_rs_staged(plan.handle, flat, shards, inbox)
        elif kernel == "noalloc":
            tide.tide_rs_reduce_noalloc(plan.handle, flat, shards)
        else:
            plan.rs_reduce(flat, shards)
        plan.check()
        _assert_equal(w, outs, expect)
        # switching back restores the default reading on the same plan
        plan.set_option(tide.TIDE_OPT_SUM_ORDER, tide.TIDE_SUM_LANDING)
        if kernel == "fused":
            plan.rs_reduce(flat, shards)
            plan.check()
            _assert_equal(w, outs, landing)


@pytest.mark.parametrize("w", [CASES[0], CASES[3]], ids=lambda w: w.name)
@pytest.mark.parametrize("kernel", ["fused", "staged"])
def test_rs_many_nodes_average_accumulate(w, kernel, oracle_cache):
    grads, geo, sums = _inputs(w, oracle_cache)
    old_h = [((np.arange(geo.S, dtype=np.float32) % 89) - 44.5) * np.float32(0.5) for _ in range(w.N)]
    expect = O.rs_finish(geo, sums, average=True, old=old_h)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_RS_AVERAGE, 1)
        plan.set_option(tide.TIDE_OPT_RS_ACCUMULATE, 1)
        flat = _flat_list(w, _device(w, grads))
        outs = [torch.from_numpy(o.copy()).to(DEV) for o in old_h]
        if kernel == "staged":
            inbox = torch.empty(tide.tide_plan_inbox_elems(plan.handle), dtype=torch.float32, device=DEV)
            tide.tide_rs_staged(plan.handle, flat, outs, inbox)
        else:
            plan.rs_reduce(flat, outs)
        plan.check()
        _assert_equal(w, outs, expect, guards=False)


@pytest.mark.parametrize("w", [CASES[1], CASES[4]], ids=lambda w: w.name)
def test_ag_many_ranks_bit_exact(w):
    """The all-gather does not depend on M, but N = 256 is the widest rank table."""
    geo = O.geometry(w.shapes, w.N)
    rng = np.random.default_rng(31)
    shards_h = [rng.integers(0, 65535, geo.S, dtype=np.uint16) for _ in range(w.N)]
    expect = O.ag_place(geo, shards_h)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        shards = [to_dev_u16(s)[0] for s in shards_h]
        params = [to_dev_u16(np.zeros(w.N * geo.e[p], dtype=np.uint16), GUARD, GUARD, fill=0x1234)
                  for p in range(w.P)]
        plan.ag_place(shards, [x[0] for x in params], 2)
        torch.cuda.synchronize()
        for p in range(w.P):
            got = params[p][1].cpu().numpy().view(np.uint16)
            assert np.array_equal(got[GUARD:GUARD + w.N * geo.e[p]], expect[p]), p
            assert (got[:GUARD] == 0x1234).all() and (got[GUARD + w.N * geo.e[p]:] == 0x1234).all()


def test_full_size_relative_order_sampled():
    """The wan22dit group at full size (M = L = 8, where the two level-2
    readings give different bits) under TIDE_SUM_RELATIVE: sampled outputs
    against the oracle computed one element at a time in that order, and at
    least one sample where the landing order would differ."""
    from gpu_common import device_grads
    w = configs.get(4)
    geo = O.geometry(w.shapes, w.N)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_SUM_ORDER, tide.TIDE_SUM_RELATIVE)
        grads = device_grads(w)
        shards = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        plan.rs_reduce(tide.pointer_array([grads[r][p] for r in range(w.N) for p in range(w.P)]),
                       tide.pointer_array(shards))
        torch.cuda.synchronize()

        def grad_at(src, p, idx):
            return w.grad_values(src, p, idx.astype(np.uint64))

        rng = np.random.default_rng(44)
        differs = 0
        for r, x in zip(rng.integers(0, w.N, 800).tolist(), rng.integers(0, geo.S, 800).tolist()):
            want = O.rs_element(geo, w.M, w.L, r, x, grad_at, O.RELATIVE)
            got = np.float32(shards[r][x].item())
            assert got.view(np.uint32) == np.float32(want).view(np.uint32), (r, x, got, want)
            differs += np.float32(O.rs_element(geo, w.M, w.L, r, x, grad_at)).view(np.uint32) != got.view(np.uint32)
        assert differs > 0
        del grads, shards
    torch.cuda.empty_cache()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("exchange", [0, 1], ids=["copy_engines", "sm_kernel"])
@pytest.mark.parametrize("stage_layout", ["separate", "rows"])
def test_all_rails_exchange_with_many_nodes(w, exchange, stage_layout):
    """The every-rail exchange with up to 32 nodes (5 rounds, the last one
    sending fewer pieces than it holds when M is not a power of two): every
    stage slot holds the shard the slot rule names, and placement from the
    slots equals the direct all-gather."""
    geo = O.geometry(w.shapes, w.N)
    M, L, S = w.M, w.L, geo.S
    rng = np.random.default_rng(31)
    shards_h = [rng.integers(0, 65535, S, dtype=np.uint16) for _ in range(w.N)]
    expect = O.ag_place(geo, shards_h)
    shards = [torch.from_numpy(x.view(np.int16)).to(DEV) for x in shards_h]
    with tide.TidePlan(w.shapes, w.N, M, L) as plan:
        plan.set_option(tide.TIDE_OPT_RD_EXCHANGE, exchange)
        if stage_layout == "rows":   # one buffer: the copy engines take strided copies
            back = torch.full((L * M, M * S), -9, dtype=torch.int16, device=DEV)
            stages = [back[i] for i in range(L * M)]
        else:
            stages = [torch.full((M * S,), -9, dtype=torch.int16, device=DEV) for _ in range(L * M)]
        tide.tide_ag_stage_init(plan.handle, shards, stages, 2)
        tide.tide_ag_rd_exchange_rails(plan.handle, stages, 2)
        torch.cuda.synchronize()
        for l in range(L):
            for n in range(M):
                got = stages[l * M + n].view(M, S)
                want = torch.stack([shards[((n + k) % M) * L + l] for k in range(M)])
                assert torch.equal(got, want), (l, n)
        node = M // 2
        params = [torch.full((w.N * geo.e[p],), -5, dtype=torch.int16, device=DEV) for p in range(w.P)]
        plan.ag_place(tide.stage_shard_pointers(stages, node, M, L, S, 2), params, 2)
        torch.cuda.synchronize()
        for p in range(w.P):
            assert np.array_equal(params[p].cpu().numpy().view(np.uint16), expect[p]), p

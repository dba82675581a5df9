"""GPU parity: libtide's CUDA kernels against the CPU oracle, element by element.

Bit-exact for the all-gather (a copy) and for the reduce-scatter (the kernel
adds in the oracle's order: l = 0..L-1, then Latin-square landing order).
Small cases compare every output; the full-size workloads compare sampled
outputs against the oracle computed one element at a time from the host
generator, plus properties that hold at any size.
"""

import numpy as np
import pytest
import torch

import fsdp_layout_aware_gb300 as tide
import oracle.tide_oracle as O
from synth import configs, gen

from gpu_common import (DEV, device_ag_shards, device_grads, f32_bits, f32_guarded, host_grads, oracle_rs,
                        run_rs, to_dev_u16, u16_of)

pytestmark = pytest.mark.gpu

GUARD = 37  # sentinel elements before and after every output buffer


def _small_workloads():
    """Cases the oracle finishes in seconds: several items and CTAs, ragged tails,
    padding, every level-2 layout (M = 1, 2, 8, 6) and odd row lengths."""
    ws = [configs.get(1)]
    ws.append(configs.scaled(configs.get(2), row_div=512, name="llama70b_rows/512"))
    q = configs.get(3)
    q.shapes = q.shapes[:5] + q.shapes[5:5 + 3 * 4] + q.shapes[-2:]
    q.dists = q.dists[:len(q.shapes)]
    ws.append(configs.scaled(q, row_div=32, name="qwen3moe_4experts_rows/32"))
    ws.append(configs.scaled(configs.get(4), row_div=1024, name="wan22dit_rows/1024"))
    u = configs.get(5)
    shapes = [(min(r, 49), c) for r, c in u.shapes[:12]]
    for r, c in u.shapes[12::12]:
        c2 = min(c, 515)
        if c % 2 and not c2 % 2:
            c2 -= 1
        shapes.append((min(r, 150), c2))
    ws.append(configs.Workload("uneven_subset", u.N, u.M, u.L, shapes,
                               [gen.UNIFORM if p % 2 == 0 else gen.INTEGER for p in range(len(shapes))],
                               seed=u.seed))
    ws.append(configs.Workload("ragged_mix", 12, 3, 4,
                               [(5, 3), (1,), (7, 2, 2), (), (3, 1), (13, 5), (2, 7), (17,), (100, 33), (0, 4)],
                               [gen.OUTLIER] * 10, seed=99))
    ws.append(configs.Workload("single_rank", 1, 1, 1, [(37, 129), (5,)], [gen.UNIFORM] * 2, seed=7))
    return ws


SMALL = _small_workloads()


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_rs_small_bit_exact(w):
    grads = host_grads(w)
    geo, expect = oracle_rs(w, grads)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        assert plan.S == geo.S
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        outs = [f32_guarded(geo.S, GUARD, GUARD) for _ in range(w.N)]
        run_rs(plan, dev, [o[0] for o in outs])
        torch.cuda.synchronize()
        for r in range(w.N):
            got = f32_bits(outs[r][0])
            want = expect[r].view(np.uint32)
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, f"rank {r}: {bad.size} mismatches, first at {bad[:5]}"
            guards = f32_bits(outs[r][1])
            assert (guards[:GUARD] == 0x7FC00000).all() and (guards[GUARD + geo.S:] == 0x7FC00000).all()
        # the inputs are read only: every gradient still holds what was uploaded
        for r in range(w.N):
            for p in range(w.P):
                assert np.array_equal(u16_of(dev[r][p]), grads[r][p]), (r, p)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("elem_bytes", [2, 4])
def test_ag_small_bit_exact(w, elem_bytes):
    geo = O.geometry(w.shapes, w.N)
    rng = np.random.default_rng(11)
    dt = np.uint16 if elem_bytes == 2 else np.uint32
    shards_h = [rng.integers(0, np.iinfo(dt).max, geo.S, dtype=dt) for _ in range(w.N)]
    expect = O.ag_place(geo, shards_h)
    tdt = torch.int16 if elem_bytes == 2 else torch.int32
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        shards = [torch.from_numpy(s.view(np.int16 if elem_bytes == 2 else np.int32)).to(DEV) for s in shards_h]
        backs = [torch.full((GUARD + w.N * geo.e[p] + GUARD,), -7, dtype=tdt, device=DEV) for p in range(w.P)]
        params = [b[GUARD:GUARD + w.N * geo.e[p]] for p, b in enumerate(backs)]
        plan.ag_place(shards, params, elem_bytes)
        torch.cuda.synchronize()
        for p in range(w.P):
            got = params[p].cpu().numpy().view(dt)
            assert np.array_equal(got, expect[p]), f"param {p}"
            g = backs[p].cpu().numpy()
            assert (g[:GUARD] == -7).all() and (g[GUARD + w.N * geo.e[p]:] == -7).all()
        # the shards are read only
        for r in range(w.N):
            assert np.array_equal(shards[r].cpu().numpy().view(dt), shards_h[r]), r


def test_rs_then_ag_round_trip_fp32():
    w = SMALL[5]   # ragged mix
    grads = host_grads(w)
    geo, shards_o = oracle_rs(w, grads)
    expect = O.ag_place(geo, shards_o)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        shards = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        run_rs(plan, dev, shards)
        params = [torch.empty(w.N * geo.e[p], dtype=torch.float32, device=DEV) for p in range(w.P)]
        plan.ag_place(shards, params, 4)
        torch.cuda.synchronize()
        for p in range(w.P):
            assert np.array_equal(params[p].cpu().numpy().view(np.uint32), expect[p].view(np.uint32))


@pytest.mark.parametrize("grad_shift,shard_shift", [((0, 0, 0, 0), 0), ((3, 3, 3, 3), 1), ((1, 5, 2, 7), 3),
                                                    ((6, 6, 6, 6), 2), ((0, 1, 0, 1), 0)])
def test_rs_misaligned_pointers(grad_shift, shard_shift):
    """Gradients at element offsets 0..7 from 16-byte boundaries (equal or
    unequal across ranks) and shards at 4-byte but not 16-byte alignment."""
    w = configs.Workload("misaligned", 4, 2, 2, [(41, 37), (9,), (20, 64), (3, 1001)], [gen.UNIFORM] * 4, seed=5)
    grads = host_grads(w)
    geo, expect = oracle_rs(w, grads)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        keep = []
        dev = []
        for r in range(w.N):
            row = []
            for p in range(w.P):
                view, back = to_dev_u16(grads[r][p], pad_before=grad_shift[r], pad_after=8)
                keep.append(back)
                row.append(view)
            dev.append(row)
        outs = [f32_guarded(geo.S, shard_shift, 4) for _ in range(w.N)]
        run_rs(plan, dev, [o[0] for o in outs])
        torch.cuda.synchronize()
        for r in range(w.N):
            assert np.array_equal(f32_bits(outs[r][0]), expect[r].view(np.uint32))


@pytest.mark.parametrize("src_shift,dst_shift,elem_bytes", [(0, 1, 2), (3, 0, 2), (5, 2, 2), (1, 3, 4), (2, 2, 4),
                                                            (7, 7, 2)])
def test_ag_misaligned_pointers(src_shift, dst_shift, elem_bytes):
    w = configs.Workload("misaligned_ag", 6, 2, 3, [(41, 37), (9,), (20, 64), (3, 1001), (127, 3)],
                         [gen.UNIFORM] * 5, seed=5)
    geo = O.geometry(w.shapes, w.N)
    dt = np.uint16 if elem_bytes == 2 else np.uint32
    tdt = torch.int16 if elem_bytes == 2 else torch.int32
    npdt = np.int16 if elem_bytes == 2 else np.int32
    rng = np.random.default_rng(3)
    shards_h = [rng.integers(0, np.iinfo(dt).max, geo.S, dtype=dt) for _ in range(w.N)]
    expect = O.ag_place(geo, shards_h)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        sb = [torch.zeros(src_shift + geo.S + 8, dtype=tdt, device=DEV) for _ in range(w.N)]
        for r in range(w.N):
            sb[r][src_shift:src_shift + geo.S].copy_(torch.from_numpy(shards_h[r].view(npdt)))
        pb = [torch.full((dst_shift + w.N * geo.e[p] + 8,), -3, dtype=tdt, device=DEV) for p in range(w.P)]
        plan.ag_place([b[src_shift:src_shift + geo.S] for b in sb],
                      [b[dst_shift:dst_shift + w.N * geo.e[p]] for p, b in enumerate(pb)], elem_bytes)
        torch.cuda.synchronize()
        for p in range(w.P):
            got = pb[p].cpu().numpy()
            assert np.array_equal(got[dst_shift:dst_shift + w.N * geo.e[p]].view(dt), expect[p])
            assert (got[:dst_shift] == -3).all() and (got[dst_shift + w.N * geo.e[p]:] == -3).all()


@pytest.mark.filterwarnings("ignore:overflow encountered in add:RuntimeWarning")  # the overflow to inf is the case
def test_rs_edge_values():
    """-0.0 everywhere (result +0.0), bf16 subnormals, and sums that overflow to inf."""
    w = configs.Workload("edges", 8, 2, 4, [(16, 24)], [gen.UNIFORM], seed=1)
    N = w.N
    n = 16 * 24
    grads = [[np.full(n, 0x8000, dtype=np.uint16)] for _ in range(N)]
    for r in range(N):
        grads[r][0][0:24] = 0x0001 + r            # subnormals
        grads[r][0][24:48] = 0x7F7F               # bf16 max: the sum overflows to +inf
        grads[r][0][48:72] = 0xFF7F if r % 2 else 0x7F7F   # +max/-max alternating
    geo, expect = oracle_rs(w, grads)
    with tide.TidePlan(w.shapes, N, w.M, w.L) as plan:
        dev = [[to_dev_u16(grads[r][0])[0]] for r in range(N)]
        shards = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(N)]
        run_rs(plan, dev, shards)
        torch.cuda.synchronize()
        for r in range(N):
            assert np.array_equal(f32_bits(shards[r]), expect[r].view(np.uint32))


def test_rs_repeat_calls_on_a_side_stream():
    """More calls than ring slots, queued without host syncs, on a side stream:
    every call must use its own pointer table."""
    w = SMALL[5]
    geo = O.geometry(w.shapes, w.N)
    s = torch.cuda.Stream()
    sets = []
    for k in range(11):
        ww = configs.Workload(w.name, w.N, w.M, w.L, w.shapes, w.dists, seed=1000 + k)
        grads = host_grads(ww)
        sets.append((grads, oracle_rs(ww, grads)[1]))
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        devs = [[[to_dev_u16(g[r][p])[0] for p in range(w.P)] for r in range(w.N)] for g, _ in sets]
        outs = [[torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)] for _ in sets]
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            for k in range(len(sets)):
                run_rs(plan, devs[k], outs[k], stream=s)
        s.synchronize()
        for k, (_, expect) in enumerate(sets):
            for r in range(w.N):
                assert np.array_equal(f32_bits(outs[k][r]), expect[r].view(np.uint32)), (k, r)


def test_rs_deterministic():
    w = SMALL[2]
    grads = host_grads(w)
    geo = O.geometry(w.shapes, w.N)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        a = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        b = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        run_rs(plan, dev, a)
        run_rs(plan, dev, b)
        torch.cuda.synchronize()
        assert all(torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in zip(a, b))


def test_device_generator_matches_host():
    from synth import device
    for dist in (gen.UNIFORM, gen.NORMAL, gen.OUTLIER, gen.INTEGER):
        key = gen.tensor_key(1238, 5, 3)
        t = torch.empty(100003, dtype=torch.int16, device=DEV)
        device.fill_bf16(t, key, dist, 1e-3, idx0=12345)
        want = gen.bf16_values(key, np.arange(12345, 12345 + 100003, dtype=np.uint64), dist, 1e-3)
        assert np.array_equal(u16_of(t), want), dist


# ------------------------------------------------------------ full size

def _sample_positions(rng, geo, N, count):
    r = rng.integers(0, N, count)
    x = rng.integers(0, max(1, geo.S), count)
    # always include both ends of every rank's shard and every parameter start
    extra = [(rr, 0) for rr in range(N)] + [(rr, geo.S - 1) for rr in range(N)]
    extra += [(int(rng.integers(0, N)), o) for o in geo.o if o < geo.S]
    return list(zip(r.tolist(), x.tolist())) + extra


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_full_size_rs_ag_sampled(cfg):
    """The bench's workloads at full size, through the same plan and launches:
    sampled outputs against the oracle, and whole-output properties."""
    w = configs.get(cfg)
    geo = O.geometry(w.shapes, w.N)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        grads = device_grads(w)
        shards = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        # the bench's call path: pointer arrays built once
        flat = tide.pointer_array([grads[r][p] for r in range(w.N) for p in range(w.P)])
        plan.rs_reduce(flat, tide.pointer_array(shards))
        ag_in = device_ag_shards(w, geo.S)
        params = [torch.empty(w.N * geo.e[p], dtype=torch.int16, device=DEV) for p in range(w.P)]
        plan.ag_place(tide.pointer_array(ag_in), tide.pointer_array(params), 2)
        torch.cuda.synchronize()

        rng = np.random.default_rng(cfg)
        samples = _sample_positions(rng, geo, w.N, 1500)

        def grad_at(src, p, idx):
            return w.grad_values(src, p, idx.astype(np.uint64))

        for r, x in samples:
            want = O.rs_element(geo, w.M, w.L, r, x, grad_at)
            got = shards[r][x].item()
            assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32), (r, x, got, want)

        # AG sampled against the oracle from the host generator
        for _ in range(1500):
            p = int(rng.integers(0, w.P))
            if geo.e[p] == 0:
                continue
            y = int(rng.integers(0, w.N * geo.e[p]))
            want = O.ag_element(geo, p, y, lambda rr, idx: w.ag_values(rr, idx.astype(np.uint64)))
            assert np.uint16(params[p][y].item() & 0xFFFF) == want

        # whole-output properties: AG pieces equal their shard slices; padding is +0.0;
        # integer-valued parameters reduce to their exact sum; the rest meet the
        # two-level fp32 error bound against an fp64 sum.
        u = 2.0 ** -24
        k = (w.L - 1) + (w.M - 1)
        gamma = k * u / (1 - k * u)
        for p in range(w.P):
            e_p, o_p = geo.e[p], geo.o[p]
            if e_p == 0:
                continue
            for r in range(w.N):
                assert torch.equal(params[p][r * e_p:(r + 1) * e_p], ag_in[r][o_p:o_p + e_p])
            n = w.numel(p)
            exact = torch.zeros(n, dtype=torch.float64, device=DEV)
            mag = torch.zeros(n, dtype=torch.float64, device=DEV)
            for src in range(w.N):
                x = grads[src][p].view(torch.bfloat16).double()
                exact += x
                mag += x.abs()
            got = torch.cat([shards[r][o_p:o_p + e_p] for r in range(w.N)])
            assert (got[n:].view(torch.int32) == 0).all(), f"padding of param {p} not +0.0"
            got = got[:n].double()
            if w.dists[p] == gen.INTEGER:
                assert torch.equal(got, exact), f"param {p}: integer sums must be exact"
            else:
                assert ((got - exact).abs() <= gamma * mag).all(), f"param {p}: error bound"
        del grads, shards, ag_in, params
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg,exchange", [(3, 1), (4, 1), (4, 0), (5, 1)],
                         ids=["qwen3moe_sm", "wan22dit_sm", "wan22dit_copy_engines", "uneven_sm"])
def test_full_size_every_rail_all_gather(cfg, exchange):
    """The every-rail all-gather (stage init, exchange of all rails, placement
    from the slots) on the full groups, as bench.py --path rd-ag runs it:
    every stage slot equals the shard the slot rule names, every placed piece
    equals its shard slice, and sampled outputs match the oracle from the
    host generator."""
    w = configs.get(cfg)
    geo = O.geometry(w.shapes, w.N)
    M, L, S = w.M, w.L, geo.S
    with tide.TidePlan(w.shapes, w.N, M, L) as plan:
        plan.set_option(tide.TIDE_OPT_RD_EXCHANGE, exchange)
        ag_in = device_ag_shards(w, S)
        stages = [torch.empty(M * S, dtype=torch.int16, device=DEV) for _ in range(L * M)]
        params = [torch.empty(w.N * geo.e[p], dtype=torch.int16, device=DEV) for p in range(w.P)]
        st = tide.pointer_array(stages)
        tide.tide_ag_stage_init(plan.handle, tide.pointer_array(ag_in), st, 2)
        tide.tide_ag_rd_exchange_rails(plan.handle, st, 2)
        node = M - 1
        plan.ag_place(tide.pointer_array(tide.stage_shard_pointers(stages, node, M, L, S, 2)),
                      tide.pointer_array(params), 2)
        plan.check()
        for l in range(L):
            for n in range(M):
                for k in range(M):
                    assert torch.equal(stages[l * M + n][k * S:(k + 1) * S], ag_in[((n + k) % M) * L + l]), (l, n, k)
        for p in range(w.P):
            e_p, o_p = geo.e[p], geo.o[p]
            for r in range(w.N):
                assert torch.equal(params[p][r * e_p:(r + 1) * e_p], ag_in[r][o_p:o_p + e_p]), (p, r)
        rng = np.random.default_rng(100 + cfg)
        for _ in range(1500):
            p = int(rng.integers(0, w.P))
            if geo.e[p] == 0:
                continue
            y = int(rng.integers(0, w.N * geo.e[p]))
            want = O.ag_element(geo, p, y, lambda rr, idx: w.ag_values(rr, idx.astype(np.uint64)))
            assert np.uint16(params[p][y].item() & 0xFFFF) == want, (p, y)
        del ag_in, stages, params
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", [2, 3], ids=["llama70b_rows16", "qwen3moe_rows16"])
@pytest.mark.parametrize("budget", [(16, 4), (16, 0), (0, 4)], ids=["pages_16_4", "sum16", "land4"])
def test_rs_staged_small_grids(cfg, budget):
    """Budgets whose grids cannot fill the GPU take the wide summing and
    landing instances (16 summing CTAs per rank on 8 or 16 ranks, 4 landing
    CTAs per rank), on groups with thousands of work items: the shards must
    equal tide_rs_reduce's bit for bit, and sampled elements the oracle."""
    w = configs.scaled(configs.get(cfg), row_div=16)
    geo = O.geometry(w.shapes, w.N)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        assert len(plan.items(0)) > 4 * 152   # more items than the full grid has CTAs
        grads = device_grads(w)
        flat = tide.pointer_array([grads[r][p] for r in range(w.N) for p in range(w.P)])
        want = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        got = [torch.full((geo.S,), float("nan"), dtype=torch.float32, device=DEV) for _ in range(w.N)]
        inbox = torch.empty(tide.tide_plan_inbox_elems(plan.handle), dtype=torch.float32, device=DEV)
        plan.rs_reduce(flat, tide.pointer_array(want))
        tide.tide_rs_staged(plan.handle, flat, tide.pointer_array(got), inbox, *budget)
        plan.check()
        for r in range(w.N):
            assert torch.equal(got[r].view(torch.int32), want[r].view(torch.int32)), r
        rng = np.random.default_rng(50 + cfg)

        def grad_at(src, p, idx):
            return w.grad_values(src, p, idx.astype(np.uint64))

        for r, x in _sample_positions(rng, geo, w.N, 300):
            expect = O.rs_element(geo, w.M, w.L, r, x, grad_at)
            assert np.float32(got[r][x].item()).view(np.uint32) == np.float32(expect).view(np.uint32), (r, x)
        del grads, want, got, inbox
    torch.cuda.empty_cache()


# ------------------------------------------------- kernel choice and waits

@pytest.mark.parametrize("w", [SMALL[0], SMALL[2], SMALL[4], SMALL[5], SMALL[6]], ids=lambda w: w.name)
def test_rs_bulk_kernel_bit_exact(w):
    """The bulk-copy kernel (TIDE_OPT_RS_KERNEL = 1) gives the oracle's bits too."""
    grads = host_grads(w)
    geo, expect = oracle_rs(w, grads)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1)
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        outs = [f32_guarded(geo.S, GUARD, GUARD) for _ in range(w.N)]
        run_rs(plan, dev, [o[0] for o in outs])
        plan.check()
        for r in range(w.N):
            assert np.array_equal(f32_bits(outs[r][0]), expect[r].view(np.uint32)), r


def test_bulk_kernel_wait_runs_out_and_context_survives():
    """Withhold one tile's data so the bulk kernel's bounded wait runs out: the
    plan reports TIDE_ERR_TIMEOUT, and the next call on the same context is
    exact again."""
    w = SMALL[1]
    grads = host_grads(w)
    geo, expect = oracle_rs(w, grads)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        outs = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1)
        plan.set_option(tide.TIDE_OPT_WAIT_LIMIT_NS, 20_000_000)
        plan.set_option(tide.TIDE_OPT_TEST_DROP_TILE, 1)
        run_rs(plan, dev, outs)
        with pytest.raises(tide.TideError) as err:
            plan.check()
        assert err.value.status == 8
        plan.set_option(tide.TIDE_OPT_TEST_DROP_TILE, -1)
        plan.set_option(tide.TIDE_OPT_WAIT_LIMIT_NS, 2_000_000_000)
        run_rs(plan, dev, outs)
        plan.check()
        for r in range(w.N):
            assert np.array_equal(f32_bits(outs[r]), expect[r].view(np.uint32)), r


def test_bulk_all_gather_wait_runs_out_and_context_survives():
    """The bulk all-gather with one chunk's load withheld: its bounded wait
    runs out (TIDE_ERR_TIMEOUT), and the next call on the same context is
    exact."""
    w = SMALL[1]
    geo = O.geometry(w.shapes, w.N)
    rng = np.random.default_rng(41)
    shards_h = [rng.integers(0, 65535, geo.S, dtype=np.uint16) for _ in range(w.N)]
    expect = O.ag_place(geo, shards_h)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, tide.TIDE_AG_BULK)
        shards = [to_dev_u16(x)[0] for x in shards_h]
        params = [torch.full((w.N * geo.e[p],), -1, dtype=torch.int16, device=DEV) for p in range(w.P)]
        assert len(plan.items(2)) > 0
        plan.set_option(tide.TIDE_OPT_WAIT_LIMIT_NS, 20_000_000)
        plan.set_option(tide.TIDE_OPT_TEST_DROP_TILE, 0)
        plan.ag_place(shards, params, 2)
        with pytest.raises(tide.TideError) as err:
            plan.check()
        assert err.value.status == 8
        plan.set_option(tide.TIDE_OPT_TEST_DROP_TILE, -1)
        plan.set_option(tide.TIDE_OPT_WAIT_LIMIT_NS, 2_000_000_000)
        plan.ag_place(shards, params, 2)
        plan.check()
        for p in range(w.P):
            assert np.array_equal(params[p].cpu().numpy().view(np.uint16), expect[p]), p


def test_host_buffers_through_the_c_abi():
    """Pinned host memory passed straight to the C ABI (the kernels read and
    write it over the host link): same bits as the oracle."""
    w = SMALL[5]
    grads = host_grads(w)
    geo, expect = oracle_rs(w, grads)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        h = [[torch.from_numpy(grads[r][p].view(np.int16)).pin_memory() for p in range(w.P)] for r in range(w.N)]
        shards = [torch.full((geo.S,), float("nan"), dtype=torch.float32).pin_memory() for _ in range(w.N)]
        run_rs(plan, h, shards)
        params = [torch.empty(w.N * geo.e[p], dtype=torch.float32).pin_memory() for p in range(w.P)]
        plan.ag_place(shards, params, 4)
        torch.cuda.synchronize()
        for r in range(w.N):
            assert np.array_equal(shards[r].numpy().view(np.uint32), expect[r].view(np.uint32)), r
        gathered = O.ag_place(geo, expect)
        for p in range(w.P):
            assert np.array_equal(params[p].numpy().view(np.uint32), gathered[p].view(np.uint32)), p


@pytest.mark.parametrize("w", [SMALL[0], SMALL[3], SMALL[4], SMALL[5]], ids=lambda w: w.name)
@pytest.mark.parametrize("elem_bytes", [2, 4])
@pytest.mark.parametrize("exchange", [0, 1], ids=["copy_engines", "sm_kernel"])
@pytest.mark.parametrize("stage_layout", ["separate", "rows"])
def test_ag_by_recursive_doubling_matches_direct_landing(w, elem_bytes, exchange, stage_layout):
    """All-gather the pages' way -- per rail, recursive-doubling exchange
    between the nodes' stage buffers, then the strided stage placement --
    must land every piece exactly where the direct all-gather does, with the
    exchange on copy engines or on the SMs."""
    geo = O.geometry(w.shapes, w.N)
    M, L, S = w.M, w.L, geo.S
    dt, tdt = (np.uint16, torch.int16) if elem_bytes == 2 else (np.uint32, torch.int32)
    rng = np.random.default_rng(17)
    shards_h = [rng.integers(0, np.iinfo(dt).max, S, dtype=dt) for _ in range(w.N)]
    expect = O.ag_place(geo, shards_h)
    shards = [torch.from_numpy(x.view(np.int16 if elem_bytes == 2 else np.int32)).to(DEV) for x in shards_h]
    with tide.TidePlan(w.shapes, w.N, M, L) as plan:
        plan.set_option(tide.TIDE_OPT_RD_EXCHANGE, exchange)
        for node in sorted({0, M - 1}):
            params = [torch.full((w.N * geo.e[p],), -5, dtype=tdt, device=DEV) for p in range(w.P)]
            for rail in range(L):
                if stage_layout == "rows":   # one buffer: the copy engines take strided copies
                    back = torch.full((M, M * S + 3), -9, dtype=tdt, device=DEV)
                    stages = [back[n, :M * S] for n in range(M)]
                else:
                    stages = [torch.full((M * S,), -9, dtype=tdt, device=DEV) for _ in range(M)]
                for n in range(M):
                    stages[n][:S].copy_(shards[n * L + rail])
                tide.tide_ag_rd_exchange(plan.handle, stages, elem_bytes)
                torch.cuda.synchronize()
                # after the exchange, slot k of node n holds node (n + k) mod M's shard
                for n in range(M):
                    for k in range(M):
                        assert torch.equal(stages[n][k * S:(k + 1) * S], shards[((n + k) % M) * L + rail])
                tide.tide_ag_stage_place(plan.handle, stages[node], node, rail, params, elem_bytes)
            torch.cuda.synchronize()
            for p in range(w.P):
                assert np.array_equal(params[p].cpu().numpy().view(dt), expect[p]), (node, p)


@pytest.mark.parametrize("w", [SMALL[0], SMALL[3], SMALL[4], SMALL[5]], ids=lambda w: w.name)
@pytest.mark.parametrize("elem_bytes", [2, 4])
@pytest.mark.parametrize("exchange", [0, 1], ids=["copy_engines", "sm_kernel"])
@pytest.mark.parametrize("stage_layout", ["separate", "rows"])
def test_ag_by_recursive_doubling_all_rails(w, elem_bytes, exchange, stage_layout):
    """The same all-gather with every rail at once: stage init, the exchange
    of all rails, then tide_ag_place reading the stage slots.  Every stage
    slot must hold the shard the slot rule names, and every piece must land
    where the direct all-gather puts it."""
    geo = O.geometry(w.shapes, w.N)
    M, L, S = w.M, w.L, geo.S
    dt, tdt = (np.uint16, torch.int16) if elem_bytes == 2 else (np.uint32, torch.int32)
    rng = np.random.default_rng(23)
    shards_h = [rng.integers(0, np.iinfo(dt).max, S, dtype=dt) for _ in range(w.N)]
    expect = O.ag_place(geo, shards_h)
    shards = [torch.from_numpy(x.view(np.int16 if elem_bytes == 2 else np.int32)).to(DEV) for x in shards_h]
    with tide.TidePlan(w.shapes, w.N, M, L) as plan:
        plan.set_option(tide.TIDE_OPT_RD_EXCHANGE, exchange)
        if stage_layout == "rows":   # one buffer: the copy engines take strided copies
            back = torch.full((L * M, M * S + 3), -9, dtype=tdt, device=DEV)
            stages = [back[i, :M * S] for i in range(L * M)]
        else:
            stages = [torch.full((M * S,), -9, dtype=tdt, device=DEV) for _ in range(L * M)]
        tide.tide_ag_stage_init(plan.handle, shards, stages, elem_bytes)
        assert plan.last_launches() == (1 if S else 0)
        tide.tide_ag_rd_exchange_rails(plan.handle, stages, elem_bytes)
        if exchange == 1 and M > 1 and S:
            assert plan.last_launches() == O.rd_rounds(M)
        torch.cuda.synchronize()
        for l in range(L):
            for n in range(M):
                for k in range(M):
                    assert torch.equal(stages[l * M + n][k * S:(k + 1) * S], shards[((n + k) % M) * L + l]), (l, n, k)
        for node in sorted({0, M - 1}):
            params = [torch.full((w.N * geo.e[p],), -5, dtype=tdt, device=DEV) for p in range(w.P)]
            plan.ag_place(tide.stage_shard_pointers(stages, node, M, L, S, elem_bytes), params, elem_bytes)
            torch.cuda.synchronize()
            for p in range(w.P):
                assert np.array_equal(params[p].cpu().numpy().view(dt), expect[p]), (node, p)


@pytest.mark.parametrize("w", [SMALL[0], SMALL[2], SMALL[3], SMALL[4], SMALL[5], SMALL[6]], ids=lambda w: w.name)
@pytest.mark.parametrize("budget", [(0, 0), (16, 4)], ids=["fill", "pages_16_4"])
def test_rs_staged_bit_exact_and_inbox(w, budget):
    """The two-stage reduce-scatter equals the oracle bit for bit, and its
    inbox holds every node partial where the Latin square lands it."""
    grads = host_grads(w)
    geo, expect = oracle_rs(w, grads)
    inbox_o = O.rs_inbox(geo, grads, w.M, w.L)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        n_inbox = tide.tide_plan_inbox_elems(plan.handle)
        assert n_inbox == inbox_o.size
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        inbox = torch.full((n_inbox,), float("nan"), dtype=torch.float32, device=DEV)
        outs = [f32_guarded(geo.S, GUARD, GUARD) for _ in range(w.N)]
        flat = [dev[r][p] for r in range(w.N) for p in range(w.P)]
        tide.tide_rs_staged(plan.handle, flat, [o[0] for o in outs], inbox, *budget)
        torch.cuda.synchronize()
        for r in range(w.N):
            assert np.array_equal(f32_bits(outs[r][0]), expect[r].view(np.uint32)), r
        got = inbox.cpu().numpy().reshape(inbox_o.shape)
        B = O.slice_len(geo.S, w.L)
        for n_dest in range(w.M):
            for g in range(w.L):
                for c in range(w.M):
                    s = (g + c) % w.L                   # the slice that lands on GPU g from index c
                    lo, hi = s * B, min(geo.S, (s + 1) * B)
                    for l_dest in range(w.L):
                        a = got[n_dest, g, c, l_dest * B:l_dest * B + (hi - lo)]
                        b = inbox_o[n_dest, g, c, l_dest * B:l_dest * B + (hi - lo)]
                        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (n_dest, g, c, l_dest)


def _vec_cases():
    """Groups whose slice length B = ceil(S / L) is a multiple of 4 (every
    row length a multiple of 96) or 2 mod 4 (one more parameter of row length
    2L), for M = 1, M <= L and M > L, so the 16- and 8-byte landing kernels
    run; ragged row counts keep padding rows in every shard."""
    shapes = [(5, 96), (100, 192), (17, 96), (1, 288), (40, 96)]
    ws = []
    for width in (4, 2):
        for M, L in [(1, 8), (2, 4), (3, 3), (4, 4), (8, 8), (6, 2), (12, 4)]:
            sh = shapes if width == 4 else shapes + [(3, 2 * L)]
            mixed = [gen.NORMAL if p % 2 else gen.OUTLIER for p in range(len(sh))]
            ws.append(configs.Workload(f"vec{width}_{M}x{L}", M * L, M, L, sh, mixed, sigma=1e-3,
                                       seed=700 + M * 10 + L + width))
    return ws


@pytest.mark.parametrize("w", _vec_cases(), ids=lambda w: w.name)
@pytest.mark.parametrize("aligned", [True, False], ids=["16B", "offset"])
@pytest.mark.parametrize("budget", [(0, 0), (16, 4)], ids=["fill", "pages_16_4"])
@pytest.mark.parametrize("variant", ["sum", "average_accumulate"])
def test_rs_staged_vector_landing(w, aligned, budget, variant):
    """With the inbox and every shard on a 16-byte boundary the landing runs
    on 16-byte (slice length a multiple of 4) or 8-byte (slice length 2 mod 4)
    loads and stores, 8 vectors per thread when its grid cannot fill the GPU
    (the pages' 4 landing CTAs per rank); one element off, it runs the 4-byte
    kernels.  All give the oracle's bits, also averaged and accumulated into
    the previous shard, and leave the guard bands alone."""
    grads = host_grads(w)
    geo, sums = oracle_rs(w, grads)
    assert O.slice_len(geo.S, w.L) % 4 == (0 if w.name.startswith("vec4") else 2)
    variants = variant == "average_accumulate"
    old = [((np.arange(geo.S, dtype=np.float32) % 19) - 9.0) * np.float32(0.25) for _ in range(w.N)]
    expect = O.rs_finish(geo, sums, average=variants, old=old if variants else None)
    lead = 32 if aligned else 33     # elements before each output: 128 or 132 bytes
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_RS_AVERAGE, int(variants))
        plan.set_option(tide.TIDE_OPT_RS_ACCUMULATE, int(variants))
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        n_inbox = tide.tide_plan_inbox_elems(plan.handle)
        inbox_back = torch.full((n_inbox + 8,), float("nan"), dtype=torch.float32, device=DEV)
        inbox = inbox_back[0 if aligned else 1:][:n_inbox]
        outs = [f32_guarded(geo.S, lead, 29) for _ in range(w.N)]
        for r in range(w.N):
            outs[r][0].copy_(torch.from_numpy(old[r]))
        flat = [dev[r][p] for r in range(w.N) for p in range(w.P)]
        tide.tide_rs_staged(plan.handle, flat, [o[0] for o in outs], inbox, *budget)
        plan.check()
        for r in range(w.N):
            assert np.array_equal(f32_bits(outs[r][0]), expect[r].view(np.uint32)), r
            back = outs[r][1]
            assert torch.isnan(back[:lead]).all() and torch.isnan(back[lead + geo.S:]).all(), r


CE_MIXED = configs.Workload("ce_mixed_pieces", 4, 2, 2, [(4400, 2048), (9, 33), (4, 1024)], [gen.UNIFORM] * 3,
                            seed=811)   # one 4.5 MB bf16 piece per rank (copied piece by piece), two small ones


@pytest.mark.parametrize("w", [SMALL[0], SMALL[3], SMALL[5], CE_MIXED], ids=lambda w: w.name)
@pytest.mark.parametrize("elem_bytes", [2, 4])
@pytest.mark.parametrize("layout", ["rows", "padded_rows", "separate", "uneven_spacing", "rows_unpadded"])
def test_ag_copy_engine_layouts(w, elem_bytes, layout):
    """The copy-engine all-gather: shards at one constant stride (rows of one
    buffer, with or without padding between rows) go as one strided copy per
    parameter whose pieces are at most 4 MiB, larger pieces one by one;
    separate buffers, unequal spacing and the unpadded destination go piece by
    piece.  Every layout lands the oracle's bits."""
    geo = O.geometry(w.shapes, w.N)
    N, S = w.N, geo.S
    dt, tdt = (np.uint16, torch.int16) if elem_bytes == 2 else (np.uint32, torch.int32)
    rng = np.random.default_rng(41)
    shards_h = [rng.integers(0, np.iinfo(dt).max, S, dtype=dt) for _ in range(N)]
    unpadded = layout == "rows_unpadded"
    expect = O.ag_place_unpadded(geo, shards_h) if unpadded else O.ag_place(geo, shards_h)
    host = [torch.from_numpy(x.view(np.int16 if elem_bytes == 2 else np.int32)) for x in shards_h]
    if layout in ("rows", "rows_unpadded", "padded_rows"):
        back = torch.zeros((N, S + (5 if layout == "padded_rows" else 0)), dtype=tdt, device=DEV)
        shards = [back[r, :S] for r in range(N)]
    elif layout == "uneven_spacing":
        back = torch.zeros((N + 1, S + 8), dtype=tdt, device=DEV)
        shards = [back[r if r < N - 1 else N, :S] for r in range(N)]
    else:
        shards = [torch.zeros(S, dtype=tdt, device=DEV) for _ in range(N)]
    for r in range(N):
        shards[r].copy_(host[r])
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, tide.TIDE_AG_COPY_ENGINES)
        plan.set_option(tide.TIDE_OPT_AG_UNPADDED, int(unpadded))
        sizes = [(geo.rows[p] * geo.Kp[p]) if unpadded else N * geo.e[p] for p in range(w.P)]
        params = [torch.full((max(1, n) + 16,), -7, dtype=tdt, device=DEV) for n in sizes]
        plan.ag_place(shards, [x[:n] for x, n in zip(params, sizes)], elem_bytes)
        torch.cuda.synchronize()
        for p in range(w.P):
            got = params[p].cpu().numpy().view(dt)
            assert np.array_equal(got[:sizes[p]], expect[p]), (layout, p)
            assert (got[sizes[p]:] == np.array(-7).astype(dt)).all(), (layout, p)   # nothing past the block


# --------------------------------------------------------------- variants

@pytest.mark.parametrize("w", [SMALL[0], SMALL[4], SMALL[5], SMALL[6]], ids=lambda w: w.name)
@pytest.mark.parametrize("kernel", ["fused", "bulk", "staged", "noalloc"])
@pytest.mark.parametrize("average,accumulate", [(1, 0), (0, 1), (1, 1)])
def test_rs_average_and_accumulate(w, kernel, average, accumulate):
    grads = host_grads(w)
    geo, sums = oracle_rs(w, grads)
    old_h = [((np.arange(geo.S, dtype=np.float32) % 97) - 48.5) * np.float32(0.25) for _ in range(w.N)]
    expect = O.rs_finish(geo, sums, average=bool(average), old=old_h if accumulate else None)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_RS_AVERAGE, average)
        plan.set_option(tide.TIDE_OPT_RS_ACCUMULATE, accumulate)
        if kernel == "bulk":
            plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1)
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        flat = [dev[r][p] for r in range(w.N) for p in range(w.P)]
        outs = [torch.from_numpy(o.copy()).to(DEV) for o in old_h]
        if kernel == "staged":
            inbox = torch.empty(tide.tide_plan_inbox_elems(plan.handle), dtype=torch.float32, device=DEV)
            tide.tide_rs_staged(plan.handle, flat, outs, inbox)
        elif kernel == "noalloc":
            tide.tide_rs_reduce_noalloc(plan.handle, flat, outs)
        else:
            plan.rs_reduce(flat, outs)
        plan.check()
        for r in range(w.N):
            assert np.array_equal(f32_bits(outs[r]), expect[r].view(np.uint32)), r


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_ag_unpadded_bit_exact(w):
    geo = O.geometry(w.shapes, w.N)
    rng = np.random.default_rng(23)
    shards_h = [rng.integers(0, 65535, geo.S, dtype=np.uint16) for _ in range(w.N)]
    expect = O.ag_place_unpadded(geo, shards_h)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_AG_UNPADDED, 1)
        shards = [torch.from_numpy(s.view(np.int16)).to(DEV) for s in shards_h]
        backs = [torch.full((GUARD + e.size + GUARD,), -7, dtype=torch.int16, device=DEV) for e in expect]
        plan.ag_place(shards, [b[GUARD:GUARD + e.size] for b, e in zip(backs, expect)], 2)
        torch.cuda.synchronize()
        for p, (b, e) in enumerate(zip(backs, expect)):
            got = b.cpu().numpy()
            assert np.array_equal(got[GUARD:GUARD + e.size].view(np.uint16), e), p
            assert (got[:GUARD] == -7).all() and (got[GUARD + e.size:] == -7).all(), p


@pytest.mark.parametrize("w", [SMALL[0], SMALL[1], SMALL[4], SMALL[5]], ids=lambda w: w.name)
def test_slot_reuse_pack_then_reduce(w):
    """Slot-Reuse: gradients packed into the vacated all-gather slots, then
    reduced from there -- same shards as reducing in place."""
    grads = host_grads(w)
    geo, expect = oracle_rs(w, grads)
    packed = O.slot_pack(geo, grads)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        slots = [torch.full((w.N * geo.S,), 0x5A5A, dtype=torch.int16, device=DEV) for _ in range(w.N)]
        tide.tide_slot_pack(plan.handle, [dev[r][p] for r in range(w.N) for p in range(w.P)], slots)
        outs = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        tide.tide_rs_reduce_slots(plan.handle, slots, outs)
        torch.cuda.synchronize()
        for r in range(w.N):
            got = u16_of(slots[r])
            mask = np.zeros(w.N * geo.S, dtype=bool)
            for p in range(w.P):
                mask[w.N * geo.o[p]:w.N * geo.o[p] + geo.rows[p] * geo.Kp[p]] = True
            assert np.array_equal(got[mask], packed[r][mask]), r
            assert (got[~mask] == 0x5A5A).all(), "padding rows of a slot stay untouched"
            assert np.array_equal(f32_bits(outs[r]), expect[r].view(np.uint32)), r


def test_overlap_check_on_real_buffers():
    """With TIDE_OPT_CHECK_OVERLAP on, disjoint torch buffers run exactly as
    before and a shard placed inside a gradient tensor is refused."""
    w = SMALL[5]
    grads = host_grads(w)
    geo, expect = oracle_rs(w, grads)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_CHECK_OVERLAP, 1)
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        flat = [dev[r][p] for r in range(w.N) for p in range(w.P)]
        outs = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        plan.rs_reduce(flat, outs)
        plan.check()
        for r in range(w.N):
            assert np.array_equal(f32_bits(outs[r]), expect[r].view(np.uint32)), r
        big = max(range(len(flat)), key=lambda i: flat[i].numel())
        inside = flat[big].view(torch.float32)[:geo.S] if flat[big].numel() >= 2 * geo.S else None
        if inside is not None:
            with pytest.raises(tide.TideError) as err:
                plan.rs_reduce(flat, [inside] + outs[1:])
            assert err.value.status == 1


@pytest.mark.parametrize("w", [SMALL[0], SMALL[1], SMALL[2], SMALL[4], SMALL[5], SMALL[6]], ids=lambda w: w.name)
@pytest.mark.parametrize("unpadded", [0, 1], ids=["padded", "unpadded"])
@pytest.mark.parametrize("elem_bytes", [2, 4])
@pytest.mark.parametrize("transport", ["copy_engines", "bulk"])
def test_ag_other_transports(w, unpadded, elem_bytes, transport):
    """TIDE_OPT_AG_TRANSPORT: copy-engine copies per piece, or bulk copies of
    the aligned middles plus the SM kernel for the rest, land every piece
    exactly where the kernel does (combinations the bulk transport does not
    take fall back to the kernel and must be exact too)."""
    geo = O.geometry(w.shapes, w.N)
    rng = np.random.default_rng(29)
    dt, tdt = (np.uint16, torch.int16) if elem_bytes == 2 else (np.uint32, torch.int32)
    shards_h = [rng.integers(0, np.iinfo(dt).max, geo.S, dtype=dt) for _ in range(w.N)]
    expect = O.ag_place_unpadded(geo, shards_h) if unpadded else O.ag_place(geo, shards_h)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_AG_TRANSPORT,
                        tide.TIDE_AG_COPY_ENGINES if transport == "copy_engines" else tide.TIDE_AG_BULK)
        plan.set_option(tide.TIDE_OPT_AG_UNPADDED, unpadded)
        shards = [torch.from_numpy(x.view(np.int16 if elem_bytes == 2 else np.int32)).to(DEV) for x in shards_h]
        sizes = [e.size for e in expect]
        lead = 40  # elements before each block: 80 or 160 bytes, so the blocks stay 16-byte aligned
        backs = [torch.full((lead + n + GUARD,), -3, dtype=tdt, device=DEV) for n in sizes]
        params = [b[lead:lead + n] for b, n in zip(backs, sizes)]
        plan.ag_place(shards, params, elem_bytes)
        plan.check()
        for p in range(w.P):
            assert np.array_equal(params[p].cpu().numpy().view(dt), expect[p]), p
            g = backs[p].cpu().numpy()
            assert (g[:lead] == -3).all() and (g[lead + sizes[p]:] == -3).all()


@pytest.mark.parametrize("w", [SMALL[1], SMALL[2], SMALL[4], SMALL[5]], ids=lambda w: w.name)
@pytest.mark.parametrize("shift", [0, 4, 1], ids=["aligned", "shifted_8B", "shifted_2B"])
def test_ag_bulk_transport_alignment(w, shift):
    """The bulk transport with parameter blocks 16-byte aligned (bulk copies),
    8 bytes off (the kernel takes every piece: a base is not 16-byte aligned)
    and 2 bytes off; repeated calls reuse the table; every byte exact."""
    geo = O.geometry(w.shapes, w.N)
    rng = np.random.default_rng(31)
    shards_h = [rng.integers(0, 65535, geo.S, dtype=np.uint16) for _ in range(w.N)]
    expect = O.ag_place(geo, shards_h)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, tide.TIDE_AG_BULK)
        shards = [to_dev_u16(x)[0] for x in shards_h]
        lead = 40 + shift  # 40 bf16 = 80 bytes keeps the block 16-byte aligned; shift moves it off
        outs = [to_dev_u16(np.zeros(w.N * geo.e[p], dtype=np.uint16), lead, GUARD, fill=0x5A5A)
                for p in range(w.P)]
        for _ in range(3):
            for o in outs:
                o[0].fill_(0x1111)
            plan.ag_place(shards, [o[0] for o in outs], 2)
            plan.check()
            for p in range(w.P):
                got = outs[p][1].cpu().numpy().view(np.uint16)
                n = w.N * geo.e[p]
                assert np.array_equal(got[lead:lead + n], expect[p]), p
                assert (got[:lead] == 0x5A5A).all() and (got[lead + n:] == 0x5A5A).all()


def test_ag_bulk_launch_count():
    """The bulk transport launches its kernel plus one remainder launch when
    the split leaves a remainder (llama70b rows/512); the default SM
    transport one kernel; both exact."""
    w = SMALL[1]
    geo = O.geometry(w.shapes, w.N)
    rng = np.random.default_rng(37)
    shards_h = [rng.integers(0, 65535, geo.S, dtype=np.uint16) for _ in range(w.N)]
    expect = O.ag_place(geo, shards_h)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        shards = [to_dev_u16(x)[0] for x in shards_h]
        for transport, want in [(tide.TIDE_AG_SM, 1), (tide.TIDE_AG_BULK, 2)]:
            plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, transport)
            params = [torch.full((w.N * geo.e[p],), -1, dtype=torch.int16, device=DEV) for p in range(w.P)]
            plan.ag_place(shards, params, 2)
            assert plan.last_launches() == want
            plan.check()
            for p in range(w.P):
                assert np.array_equal(params[p].cpu().numpy().view(np.uint16), expect[p]), (transport, p)


@pytest.mark.parametrize("cfg", [2, 4])
@pytest.mark.parametrize("kernel", ["staged", "bulk", "noalloc"])
def test_full_size_other_reduce_kernels_sampled(cfg, kernel):
    """The staged, bulk-copy and no-allocation reduce-scatters on the full
    llama70b and wan22dit groups: sampled outputs against the oracle."""
    w = configs.get(cfg)
    geo = O.geometry(w.shapes, w.N)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        grads = device_grads(w)
        shards = [torch.full((geo.S,), float("nan"), dtype=torch.float32, device=DEV) for _ in range(w.N)]
        flat = tide.pointer_array([grads[r][p] for r in range(w.N) for p in range(w.P)])
        if kernel == "staged":
            inbox = torch.empty(tide.tide_plan_inbox_elems(plan.handle), dtype=torch.float32, device=DEV)
            tide.tide_rs_staged(plan.handle, flat, tide.pointer_array(shards), inbox)
        elif kernel == "bulk":
            plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1)
            plan.rs_reduce(flat, tide.pointer_array(shards))
        else:
            tide.tide_rs_reduce_noalloc(plan.handle, flat, tide.pointer_array(shards))
        plan.check()

        def grad_at(src, p, idx):
            return w.grad_values(src, p, idx.astype(np.uint64))

        rng = np.random.default_rng(100 + cfg)
        for r, x in _sample_positions(rng, geo, w.N, 400):
            want = O.rs_element(geo, w.M, w.L, r, x, grad_at)
            got = shards[r][x].item()
            assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32), (kernel, r, x, got, want)
        # no output left unwritten (NaN sentinel)
        for r in range(w.N):
            assert not torch.isnan(shards[r]).any(), (kernel, r)
        del grads, shards
    torch.cuda.empty_cache()

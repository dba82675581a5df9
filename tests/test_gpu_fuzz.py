"""Seeded random groups through every kernel, bit for bit against the oracle.

Each case draws M, L (M > L included), parameter shapes (0-D, 1-D, 3-D, empty,
fewer rows than ranks, odd row lengths), value distributions, the level-2
order and the averaging / accumulate variants (every fourth case with pieces
of several work items), then runs the reduce-scatter on the direct, staged,
bulk (M <= 8) and no-allocation paths, and the all-gather on the SM and bulk
transports and through the every-rail exchange.  Sizes stay small so the
oracle is quick.
"""

import numpy as np
import pytest
import torch

import fsdp_layout_aware_gb300 as tide
import oracle.tide_oracle as O
from synth import configs

from gpu_common import DEV, f32_bits, host_grads, to_dev_u16

pytestmark = pytest.mark.gpu

SEEDS = list(range(48))


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    L = int(rng.integers(1, 9))
    if seed % 3 == 0:   # more nodes than GPUs per node
        M = int(rng.integers(L + 1, 13)) if L <= 4 else int(rng.integers(L, L + 2))
    else:
        M = int(rng.integers(1, L + 1))
    N = M * L
    big = seed % 4 == 1   # pieces of several work items each
    shapes = []
    for _ in range(int(rng.integers(1, 4 if big else 10))):
        kind = int(rng.integers(0, 6))
        rows = int(rng.integers(0, (40 if big else 2) * N + 2))
        cols = int(rng.integers(1, 600 if big else 90))
        if kind == 0:
            shapes.append(())
        elif kind == 1:
            shapes.append((rows,))
        elif kind == 2:
            shapes.append((rows, cols, int(rng.integers(1, 4))))
        else:
            shapes.append((rows, cols))
    dists = [int(rng.integers(0, 4)) for _ in shapes]
    order = O.RELATIVE if rng.integers(0, 2) else O.LANDING
    average, accumulate = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    w = configs.Workload(f"fuzz{seed}", N, M, L, shapes, dists, sigma=1e-3, seed=5000 + seed)
    return w, order, average, accumulate


@pytest.mark.parametrize("seed", SEEDS)
def test_fuzz_group(seed):
    w, order, average, accumulate = _case(seed)
    geo = O.geometry(w.shapes, w.N)
    grads = host_grads(w)
    sums = O.rs_reduce(geo, grads, w.M, w.L, order)
    old = [((np.arange(geo.S, dtype=np.float32) % 23) - 11.0) * np.float32(0.125) for _ in range(w.N)]
    expect = O.rs_finish(geo, sums, average=average, old=old if accumulate else None)
    rng = np.random.default_rng(seed)
    shards_h = [rng.integers(0, 65535, geo.S, dtype=np.uint16) for _ in range(w.N)]
    ag_expect = O.ag_place(geo, shards_h)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        if geo.S == 0:
            return
        plan.set_option(tide.TIDE_OPT_SUM_ORDER,
                        tide.TIDE_SUM_RELATIVE if order == O.RELATIVE else tide.TIDE_SUM_LANDING)
        plan.set_option(tide.TIDE_OPT_RS_AVERAGE, int(average))
        plan.set_option(tide.TIDE_OPT_RS_ACCUMULATE, int(accumulate))
        dev = [[to_dev_u16(grads[r][p])[0] for p in range(w.P)] for r in range(w.N)]
        flat = [dev[r][p] for r in range(w.N) for p in range(w.P)]
        kernels = ["fused", "staged", "noalloc"] + (["bulk"] if w.M <= 8 else [])
        for kernel in kernels:
            outs = [torch.from_numpy(o.copy()).to(DEV) for o in old]
            plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1 if kernel == "bulk" else 0)
            if kernel == "staged":
                inbox = torch.empty(tide.tide_plan_inbox_elems(plan.handle), dtype=torch.float32, device=DEV)
                tide.tide_rs_staged(plan.handle, flat, outs, inbox)
            elif kernel == "noalloc":
                tide.tide_rs_reduce_noalloc(plan.handle, flat, outs)
            else:
                plan.rs_reduce(flat, outs)
            plan.check()
            for r in range(w.N):
                assert np.array_equal(f32_bits(outs[r]), expect[r].view(np.uint32)), (seed, kernel, r)
        plan.set_option(tide.TIDE_OPT_RS_KERNEL, 0)
        shards = [to_dev_u16(x)[0] for x in shards_h]
        for transport in (tide.TIDE_AG_SM, tide.TIDE_AG_BULK):
            plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, transport)
            params = [torch.full((max(1, w.N * geo.e[p]),), -1, dtype=torch.int16, device=DEV) for p in range(w.P)]
            plan.ag_place(shards, [x[:w.N * geo.e[p]] for p, x in enumerate(params)], 2)
            plan.check()
            for p in range(w.P):
                got = params[p][:w.N * geo.e[p]].cpu().numpy().view(np.uint16)
                assert np.array_equal(got, ag_expect[p]), (seed, transport, p)
        # every rail at once: stage init, exchange (transport by seed), placement from the slots
        plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, tide.TIDE_AG_SM)
        plan.set_option(tide.TIDE_OPT_RD_EXCHANGE, seed % 2)
        stages = [torch.full((w.M * geo.S,), -3, dtype=torch.int16, device=DEV) for _ in range(w.L * w.M)]
        tide.tide_ag_stage_init(plan.handle, shards, stages, 2)
        tide.tide_ag_rd_exchange_rails(plan.handle, stages, 2)
        node = seed % w.M
        params = [torch.full((max(1, w.N * geo.e[p]),), -1, dtype=torch.int16, device=DEV) for p in range(w.P)]
        plan.ag_place(tide.stage_shard_pointers(stages, node, w.M, w.L, geo.S, 2),
                      [x[:w.N * geo.e[p]] for p, x in enumerate(params)], 2)
        plan.check()
        for p in range(w.P):
            got = params[p][:w.N * geo.e[p]].cpu().numpy().view(np.uint16)
            assert np.array_equal(got, ag_expect[p]), (seed, "every rail", p)

"""CUDA-graph capture of the hot path: the reduce-scatter and the all-gather
captured once, replayed with new data behind the same buffers; every replay
must equal the oracle for the data it saw."""

import numpy as np
import pytest
import torch

import fsdp_layout_aware_gb300 as tide
import oracle.tide_oracle as O
from synth import configs, gen

from gpu_common import DEV, f32_bits, host_grads, oracle_rs, to_dev_u16

pytestmark = pytest.mark.gpu

W = configs.Workload("graph_2x4", 8, 2, 4, [(5, 3), (1,), (100, 33), (1031, 257), (0, 4), (64, 64)],
                     [gen.NORMAL if p % 2 else gen.OUTLIER for p in range(6)], sigma=1e-3, seed=601)


def _variant(w, k):
    return configs.Workload(f"{w.name}_{k}", w.N, w.M, w.L, w.shapes, w.dists, sigma=w.sigma, seed=w.seed + 17 * k)


def _load(dev, grads, w):
    for r in range(w.N):
        for p in range(w.P):
            if grads[r][p].size:
                dev[r][p].copy_(torch.from_numpy(grads[r][p].view(np.int16)))


@pytest.mark.parametrize("staged", [False, True], ids=["fused", "staged"])
@pytest.mark.parametrize("transport", ["sm", "bulk", "copy_engines"])
def test_capture_and_replay(staged, transport):
    w = W
    geo = O.geometry(w.shapes, w.N)
    datasets = [host_grads(_variant(w, k)) for k in range(3)]
    expects = [oracle_rs(w, g)[1] for g in datasets]
    rng = np.random.default_rng(3)
    ag_sets = [[rng.integers(0, 65535, geo.S, dtype=np.uint16) for _ in range(w.N)] for _ in range(3)]
    ag_expects = [O.ag_place(geo, s) for s in ag_sets]
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, {"sm": tide.TIDE_AG_SM, "bulk": tide.TIDE_AG_BULK,
                                                     "copy_engines": tide.TIDE_AG_COPY_ENGINES}[transport])
        dev = [[to_dev_u16(datasets[0][r][p])[0] for p in range(w.P)] for r in range(w.N)]
        flat = tide.pointer_array([dev[r][p] for r in range(w.N) for p in range(w.P)])
        outs = [torch.empty(geo.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        shards = tide.pointer_array(outs)
        ag_in = [torch.empty(geo.S, dtype=torch.int16, device=DEV) for _ in range(w.N)]
        params = [torch.empty(w.N * geo.e[p], dtype=torch.int16, device=DEV) for p in range(w.P)]
        inbox = torch.empty(max(1, tide.tide_plan_inbox_elems(plan.handle)), dtype=torch.float32, device=DEV)
        s = torch.cuda.Stream()

        def step():
            if staged:
                tide.tide_rs_staged(plan.handle, flat, shards, inbox, 0, 0, s)
            else:
                plan.rs_reduce(flat, shards, s)
            plan.ag_place(ag_in, params, 2, s)

        with torch.cuda.stream(s):
            step()                      # first call outside capture: device state
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        torch.cuda.synchronize()
        for k in [1, 2, 0, 2]:
            _load(dev, datasets[k], w)
            for r in range(w.N):
                ag_in[r].copy_(torch.from_numpy(ag_sets[k][r].view(np.int16)))
                outs[r].fill_(float("nan"))
            for p in range(w.P):
                params[p].fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            for r in range(w.N):
                assert np.array_equal(f32_bits(outs[r]), expects[k][r].view(np.uint32)), (k, r)
            for p in range(w.P):
                assert np.array_equal(params[p].cpu().numpy().view(np.uint16), ag_expects[k][p]), (k, p)
        del g


def test_capture_slots_run_out_with_a_status():
    w = W
    geo = O.geometry(w.shapes, w.N)
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        ag_in = [torch.zeros(geo.S, dtype=torch.int16, device=DEV) for _ in range(w.N)]
        params = [torch.empty(w.N * geo.e[p], dtype=torch.int16, device=DEV) for p in range(w.P)]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            plan.ag_place(ag_in, params, 2, s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        statuses = []
        with torch.cuda.graph(g, stream=s):
            for _ in range(9):
                try:
                    plan.ag_place(ag_in, params, 2, s)
                    statuses.append(0)
                except tide.TideError as err:
                    statuses.append(err.status)
        assert statuses == [0] * 8 + [1]
        g.replay()
        torch.cuda.synchronize()
        for p in range(w.P):
            assert (params[p] == 0).all()
        del g


W3 = configs.Workload("graph_3x2", 6, 3, 2, [(7, 5), (13,), (40, 9)], [gen.UNIFORM] * 3, seed=602)


@pytest.mark.parametrize("w", [W, W3], ids=lambda w: w.name)
@pytest.mark.parametrize("exchange", [0, 1], ids=["copy_engines", "sm_kernel"])
def test_capture_every_rail_all_gather(w, exchange):
    """Stage init, the exchange of every rail and the placement from the stage
    slots, captured once and replayed with new shards behind the same buffers:
    every replay lands every piece where the direct all-gather puts it."""
    geo = O.geometry(w.shapes, w.N)
    M, L, S = w.M, w.L, geo.S
    rng = np.random.default_rng(5)
    sets = [[rng.integers(0, 65535, S, dtype=np.uint16) for _ in range(w.N)] for _ in range(3)]
    expects = [O.ag_place(geo, x) for x in sets]
    with tide.TidePlan(w.shapes, w.N, M, L) as plan:
        plan.set_option(tide.TIDE_OPT_RD_EXCHANGE, exchange)
        shards = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(w.N)]
        stages = [torch.empty(M * S, dtype=torch.int16, device=DEV) for _ in range(L * M)]
        params = [torch.empty(w.N * geo.e[p], dtype=torch.int16, device=DEV) for p in range(w.P)]
        sh, st = tide.pointer_array(shards), tide.pointer_array(stages)
        slots = tide.pointer_array(tide.stage_shard_pointers(stages, M - 1, M, L, S, 2))
        pp = tide.pointer_array(params)
        s = torch.cuda.Stream()

        def step():
            tide.tide_ag_stage_init(plan.handle, sh, st, 2, s)
            tide.tide_ag_rd_exchange_rails(plan.handle, st, 2, s)
            plan.ag_place(slots, pp, 2, s)

        with torch.cuda.stream(s):
            step()                      # first calls outside capture: device state
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        torch.cuda.synchronize()
        for k in [1, 0, 2]:
            for r in range(w.N):
                shards[r].copy_(torch.from_numpy(sets[k][r].view(np.int16)))
            for x in stages:
                x.fill_(-9)
            for p in range(w.P):
                params[p].fill_(-1)
            g.replay()
            torch.cuda.synchronize()
            for p in range(w.P):
                assert np.array_equal(params[p].cpu().numpy().view(np.uint16), expects[k][p]), (k, p)
        del g

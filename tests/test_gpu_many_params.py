"""A group of many small parameters: 1500 tensors on 16 ranks (2 nodes of 8),
so every call passes 24,000 gradient pointers and the work lists hold tens of
thousands of items.  Every rank's gradients sit in one device buffer at
element (not 16-byte) offsets, so the parameters' address phases differ and
both the vector and the element-wise load paths run.  The reduce-scatter on
the direct, bulk-copy, staged and no-allocation paths and the all-gather on
the SM and bulk transports must equal the oracle bit for bit."""

import numpy as np
import pytest
import torch

import fsdp_layout_aware_gb300 as tide
import oracle.tide_oracle as O
from synth import configs, gen

from gpu_common import DEV, f32_bits, host_grads

pytestmark = pytest.mark.gpu

P_MANY = 1500


def _group():
    rng = np.random.default_rng(77)
    shapes = []
    for p in range(P_MANY):
        kind = p % 7
        if kind == 0:
            shapes.append(())
        elif kind == 1:
            shapes.append((int(rng.integers(0, 40)),))
        elif kind == 2:
            shapes.append((0, int(rng.integers(1, 9))))
        else:
            shapes.append((int(rng.integers(1, 40)), int(rng.integers(1, 21))))
    dists = [gen.INTEGER if p % 3 == 0 else gen.OUTLIER for p in range(P_MANY)]
    return configs.Workload("many_params", 16, 2, 8, shapes, dists, sigma=1e-3, seed=4242)


@pytest.fixture(scope="module")
def group():
    w = _group()
    geo = O.geometry(w.shapes, w.N)
    grads = host_grads(w)
    # every rank's gradients packed back to back in one buffer, at element offsets
    dev, ptrs = [], []
    for r in range(w.N):
        flat = np.concatenate([g for g in grads[r]] + [np.zeros(1, np.uint16)])
        buf = torch.from_numpy(flat.view(np.int16)).to(DEV)
        dev.append(buf)
        off = 0
        for p in range(w.P):
            ptrs.append(buf.data_ptr() + 2 * off)
            off += grads[r][p].size
    rs_want = O.rs_reduce(geo, grads, w.M, w.L)
    rng = np.random.default_rng(5)
    ag_in = [rng.integers(0, 65535, geo.S, dtype=np.uint16) for _ in range(w.N)]
    ag_want = O.ag_place(geo, ag_in)
    return w, geo, dev, ptrs, rs_want, ag_in, ag_want


def _check_rs(geo, outs, want):
    for r, o in enumerate(outs):
        assert np.array_equal(f32_bits(o), want[r].view(np.uint32)), r


@pytest.mark.parametrize("path", ["fused", "bulk", "staged", "noalloc"])
def test_many_params_reduce_scatter(group, path):
    w, geo, _dev, ptrs, want, _, _ = group
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        outs = [torch.full((geo.S,), float("nan"), dtype=torch.float32, device=DEV) for _ in range(w.N)]
        if path == "noalloc":
            tide.tide_rs_reduce_noalloc(plan.handle, ptrs, outs)
        elif path == "staged":
            inbox = torch.empty(tide.tide_plan_inbox_elems(plan.handle), dtype=torch.float32, device=DEV)
            tide.tide_rs_staged(plan.handle, ptrs, outs, inbox, 0, 0)
        else:
            plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1 if path == "bulk" else 0)
            plan.rs_reduce(ptrs, outs)
        torch.cuda.synchronize()
        plan.check()
        _check_rs(geo, outs, want)


@pytest.mark.parametrize("transport", ["sm", "bulk"])
def test_many_params_all_gather(group, transport):
    w, geo, _dev, _ptrs, _, ag_in, want = group
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, tide.TIDE_AG_SM if transport == "sm" else tide.TIDE_AG_BULK)
        shards = [torch.from_numpy(x.view(np.int16)).to(DEV) for x in ag_in]
        params = [torch.full((max(1, w.N * geo.e[p]),), -1, dtype=torch.int16, device=DEV) for p in range(w.P)]
        plan.ag_place(shards, params, 2)
        torch.cuda.synchronize()
        plan.check()
        for p in range(w.P):
            got = params[p].cpu().numpy().view(np.uint16)[:w.N * geo.e[p]]
            assert np.array_equal(got, want[p]), p

"""Offsets past 2^31 elements (and 2^32 bytes): one parameter whose per-rank
piece alone exceeds 2^31 elements, followed by a small padded one, so every
offset of the second parameter, the tail of the first and the parameter-major
all-gather positions (beyond 2^32) need 64-bit arithmetic.  About 52 GB on
the device; outputs are checked at chosen and sampled positions against the
oracle computed one element at a time from the host generator.
"""

import numpy as np
import pytest
import torch

import fsdp_layout_aware_gb300 as tide
import oracle.tide_oracle as O
from synth import configs, gen

from gpu_common import DEV, device_ag_shards, device_grads

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

W = configs.Workload("offsets_beyond_2^31", 2, 2, 1, [(2 * 32769, 65537), (5, 3)], [gen.NORMAL, gen.INTEGER],
                     sigma=1e-3, seed=777)


def test_rs_ag_offsets_beyond_int32():
    w = W
    geo = O.geometry(w.shapes, w.N)
    assert geo.e[0] > 2 ** 31 and geo.o[1] > 2 ** 31 and w.N * geo.e[0] > 2 ** 32
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        assert plan.S == geo.S
        grads = device_grads(w)
        shards = [torch.full((geo.S,), float("nan"), dtype=torch.float32, device=DEV) for _ in range(w.N)]
        plan.rs_reduce(tide.pointer_array([grads[r][p] for r in range(w.N) for p in range(w.P)]),
                       tide.pointer_array(shards))
        torch.cuda.synchronize()
        del grads
        torch.cuda.empty_cache()

        def grad_at(src, p, idx):
            return w.grad_values(src, p, idx.astype(np.uint64))

        rng = np.random.default_rng(11)
        edge = [0, 1, 8191, 8192, 2 ** 31 - 9, 2 ** 31 - 1, 2 ** 31, 2 ** 31 + 1, geo.e[0] - 1]
        edge += list(range(geo.o[1], geo.S))          # the small parameter, padding row included
        picks = edge + [int(x) for x in rng.integers(0, geo.S, 300)]
        for r in range(w.N):
            for x in picks:
                want = O.rs_element(geo, w.M, w.L, r, x, grad_at)
                got = shards[r][x].item()
                assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32), (r, x, got, want)
        del shards
        torch.cuda.empty_cache()

        ag_in = device_ag_shards(w, geo.S)
        params = [torch.full((w.N * geo.e[p],), -1, dtype=torch.int16, device=DEV) for p in range(w.P)]
        plan.ag_place(tide.pointer_array(ag_in), tide.pointer_array(params), 2)
        torch.cuda.synchronize()
        n0 = w.N * geo.e[0]
        ys = [0, geo.e[0] - 1, geo.e[0], 2 ** 32 - 1, 2 ** 32, n0 - 1] + [int(y) for y in rng.integers(0, n0, 300)]
        for p, y in [(0, y) for y in ys] + [(1, y) for y in range(w.N * geo.e[1])]:
            want = O.ag_element(geo, p, y, lambda rr, idx: w.ag_values(rr, idx.astype(np.uint64)))
            assert np.uint16(params[p][y].item() & 0xFFFF) == want, (p, y)
        del ag_in, params
    torch.cuda.empty_cache()

"""tide_rs_reduce_noalloc: the reduce-scatter for callers that cannot allocate
device memory (a process whose free device memory belongs to a caching
allocator, code that must not take cudaMalloc/cudaFree's implicit device
synchronisation, a fixed pre-reserved budget).  It keeps its work list and
pointer tables in a fixed 8 MiB static device array instead of memory the plan
allocates, and runs the same kernel, so its output must equal tide_rs_reduce's
bit for bit -- checked here through the C ABI on two calls in a row, the second
with different inputs so that anything left over from the first call would
show.  This file sorts last so that a run stopping at the first failure has
already run every other test."""

import warnings

import numpy as np
import pytest
import torch

import fsdp_layout_aware_gb300 as tide
from synth import configs, gen

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

WORKLOADS = [
    configs.Workload("ragged_mix", 12, 3, 4,
                     [(5, 3), (1,), (7, 2, 2), (), (3, 1), (13, 5), (2, 7), (17,), (100, 33), (0, 4)],
                     [gen.OUTLIER] * 10, seed=21),
    configs.scaled(configs.get(2), row_div=512, name="llama70b_rows/512"),
    configs.scaled(configs.get(4), row_div=1024, name="wan22dit_rows/1024"),
]


def _device_grads(w, seed):
    out = []
    for r in range(w.N):
        for p in range(w.P):
            bits = gen.bf16_tensor(gen.tensor_key(seed, r, p), w.numel(p), w.dists[p], w.sigma)
            out.append(torch.from_numpy(bits.view(np.int16)).to(DEV))
    return out


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_noalloc_matches_tide_rs_reduce_on_two_calls(w):
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        for call, seed in enumerate((1000, 2000)):
            grads = _device_grads(w, seed)
            want = [torch.empty(plan.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
            got = [torch.full((plan.S,), float("nan"), dtype=torch.float32, device=DEV) for _ in range(w.N)]
            tide.tide_rs_reduce(plan.handle, grads, want)
            tide.tide_rs_reduce_noalloc(plan.handle, grads, got)
            torch.cuda.synchronize()
            for r in range(w.N):
                assert torch.equal(got[r].view(torch.int32), want[r].view(torch.int32)), (call, r)


def test_noalloc_rejects_groups_beyond_its_scratch():
    # 2.5e9 shard elements -> about 300k work items, more than 8 MiB of tables.
    with tide.TidePlan([(8 << 20, 300)], 8, 1, 8) as plan:
        fake_grads = [0x100000 * (r + 1) for r in range(8)]
        fake_shards = [0x10000000 * (r + 1) for r in range(8)]
        with pytest.raises(tide.TideError) as err:
            tide.tide_rs_reduce_noalloc(plan.handle, fake_grads, fake_shards)
        assert err.value.status == 1 and "8388608" in str(err.value)


def test_noalloc_reuses_what_the_array_holds():
    """The array keeps the last call's work list and tables: a repeat call on
    the same buffers uploads nothing and launches only the reduce-scatter;
    new data behind the same pointers, new shard pointers, and two plans
    taking turns must all still give tide_rs_reduce's bits."""
    wa, wb = WORKLOADS[0], WORKLOADS[1]
    with tide.TidePlan(wa.shapes, wa.N, wa.M, wa.L) as pa, tide.TidePlan(wb.shapes, wb.N, wb.M, wb.L) as pb:
        ga, gb = _device_grads(wa, 3000), _device_grads(wb, 3001)
        outs_a = [torch.empty(pa.S, dtype=torch.float32, device=DEV) for _ in range(wa.N)]
        outs_a2 = [torch.empty(pa.S, dtype=torch.float32, device=DEV) for _ in range(wa.N)]
        outs_b = [torch.empty(pb.S, dtype=torch.float32, device=DEV) for _ in range(wb.N)]

        def check(plan, grads, outs):
            want = [torch.empty_like(o) for o in outs]
            tide.tide_rs_reduce(plan.handle, grads, want)
            torch.cuda.synchronize()
            for r, (o, x) in enumerate(zip(outs, want)):
                assert torch.equal(o.view(torch.int32), x.view(torch.int32)), r

        tide.tide_rs_reduce_noalloc(pa.handle, ga, outs_a)
        assert pa.last_launches() == 2            # tables built, then the reduce-scatter
        check(pa, ga, outs_a)
        tide.tide_rs_reduce_noalloc(pa.handle, ga, outs_a)
        assert pa.last_launches() == 1            # nothing changed: the reduce-scatter only
        check(pa, ga, outs_a)
        fresh = _device_grads(wa, 3002)           # new data behind the same pointers
        for g, f in zip(ga, fresh):
            g.copy_(f)
        tide.tide_rs_reduce_noalloc(pa.handle, ga, outs_a)
        assert pa.last_launches() == 1
        check(pa, ga, outs_a)
        tide.tide_rs_reduce_noalloc(pa.handle, ga, outs_a2)   # new shard pointers only
        assert pa.last_launches() == 1
        check(pa, ga, outs_a2)
        for _ in range(2):                        # two plans taking turns on one array
            tide.tide_rs_reduce_noalloc(pb.handle, gb, outs_b)
            assert pb.last_launches() == 2
            check(pb, gb, outs_b)
            tide.tide_rs_reduce_noalloc(pa.handle, ga, outs_a)
            assert pa.last_launches() == 2
            check(pa, ga, outs_a)


def test_noalloc_refuses_a_stream_under_capture():
    """A captured launch would keep reading the shared array after later
    calls rewrote it, so a call on a capturing stream is refused before it
    touches the array; the next ordinary call is still exact."""
    w = WORKLOADS[0]
    with tide.TidePlan(w.shapes, w.N, w.M, w.L) as plan:
        grads = _device_grads(w, 4000)
        got = [torch.full((plan.S,), float("nan"), dtype=torch.float32, device=DEV) for _ in range(w.N)]
        want = [torch.empty(plan.S, dtype=torch.float32, device=DEV) for _ in range(w.N)]
        tide.tide_rs_reduce_noalloc(plan.handle, grads, got)   # set-up outside any capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        status = None
        with warnings.catch_warnings():
            # the refused call enqueues nothing, so the captured graph is empty
            warnings.filterwarnings("ignore", message="The CUDA Graph is empty")
            with torch.cuda.graph(g, stream=s):
                try:
                    tide.tide_rs_reduce_noalloc(plan.handle, grads, got, s)
                except tide.TideError as err:
                    status = err.status
        assert status == 1
        for o in got:
            o.fill_(float("nan"))
        tide.tide_rs_reduce_noalloc(plan.handle, grads, got)
        tide.tide_rs_reduce(plan.handle, grads, want)
        torch.cuda.synchronize()
        for r in range(w.N):
            assert torch.equal(got[r].view(torch.int32), want[r].view(torch.int32)), r

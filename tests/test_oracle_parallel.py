"""The multi-process CPU baseline (oracle.parallel): each worker runs the
oracle, unchanged, on its own destination ranks and generates only the
inputs those ranks read; the merged shards and gathered blocks must equal
the single-process oracle on the full inputs bit for bit."""

import numpy as np
import pytest

import oracle.parallel as OP
import oracle.tide_oracle as O
from synth import configs, gen

WORKLOADS = [
    configs.get("tiny"),
    # 3 nodes x 4 GPUs; fewer rows than ranks (padding-only ranks), 0-D, 1-D, empty
    configs.Workload("ragged_3x4", 12, 3, 4, [(5, 3), (1,), (), (13, 5), (100, 33), (0, 4), (17,)],
                     [gen.UNIFORM, gen.INTEGER, gen.NORMAL, gen.OUTLIER, gen.UNIFORM, gen.UNIFORM, gen.INTEGER],
                     seed=77),
    # more nodes than GPUs per node (batched level 2)
    configs.Workload("batched_6x2", 12, 6, 2, [(31, 7), (12, 12), (3,)], [gen.OUTLIER] * 3, seed=78),
]


def test_rank_sets_cover_every_rank_once():
    for N in (1, 4, 12, 48, 64):
        for workers in (1, 3, 16, 100):
            sets = OP.rank_sets(N, workers)
            assert sorted(r for s in sets for r in s) == list(range(N))
            assert len(sets) == min(N, workers)


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_split_oracle_equals_the_full_oracle(w):
    geo = O.geometry(w.shapes, w.N)
    grads = [[gen.bf16_tensor(w.grad_key(r, p), w.numel(p), w.dists[p], w.sigma) for p in range(w.P)]
             for r in range(w.N)]
    shards_in = [w.ag_values(r, np.arange(geo.S, dtype=np.uint64)) for r in range(w.N)]
    want_rs = O.rs_reduce(geo, grads, w.M, w.L)
    want_ag = O.ag_place(geo, shards_in)
    res = OP.run(w, workers=5, passes=2, warmup=1, want_outputs=True, timeout=300)
    rs, ag = res["outputs"]
    assert res["workers"] == min(5, w.N) and res["passes"] == [2] * res["workers"]
    assert sorted(r for s in res["ranks"] for r in s) == list(range(w.N))
    for r in range(w.N):
        assert np.array_equal(rs[r].view(np.uint32), want_rs[r].view(np.uint32)), r
    for p in range(w.P):
        assert np.array_equal(ag[p], want_ag[p]), p


def test_worker_inputs_hold_exactly_the_rows_their_ranks_read():
    w = WORKLOADS[1]
    geo, grads, shards = OP.worker_inputs(w, [2, 7])
    for src in range(w.N):
        for p in range(w.P):
            full = gen.bf16_tensor(w.grad_key(src, p), w.numel(p), w.dists[p], w.sigma)
            mask = np.zeros(full.size, dtype=bool)
            for r in (2, 7):
                a = r * geo.e[p]
                mask[a:a + O.valid_elems(geo, p, r)] = True
            assert np.array_equal(grads[src][p][mask], full[mask])
            assert not grads[src][p][~mask].any()
    assert [r for r in range(w.N) if shards[r] is not None] == [2, 7]


def test_time_budget_mode_counts_whole_passes():
    w = WORKLOADS[0]
    res = OP.run(w, workers=2, passes=None, seconds=0.2, timeout=300)
    assert res["workers"] == 2 and all(n >= 1 for n in res["passes"])
    assert all(t >= 0.2 for t in res["seconds"]) and res["wall"] >= max(res["seconds"]) * 0.99

"""The oracle run on all host cores: disjoint sets of destination ranks, one
set per worker process.

TEST INFRASTRUCTURE ONLY -- used by the tests and by the CPU-baseline leg of
``bench.py``; the CUDA library never calls it.

Every destination rank's packed shard ([Abstract] Table 2) depends only on
that rank's rows of every contributor's gradient, and every all-gather piece
only on its own rank's shard ([Endgame] "All-gather: parameters land at their
final address"), so the work splits by destination rank with no exchange.
Each worker calls ``rs_reduce`` and ``ag_place`` of this package, unchanged,
on its own ranks: a rank's results are computed exactly as in the full call,
so the merged output equals the single-process oracle bit for bit.

Workers are started with the ``spawn`` method (never forked from a process
that may hold a CUDA context).  A worker generates, from the seeded
generator, only the values its ranks read -- rows [r*Rp, (r+1)*Rp) of every
contributor's gradient of every parameter, and its ranks' packed shards --
into arrays of the full length whose other entries stay zero and are never
read.  Once every worker reports ready the parent releases them together and
times from that moment to the last worker's report.
"""

import multiprocessing as mp
import time

import numpy as np

from synth.gen import bf16_tensor

from .tide_oracle import ag_place, geometry, rs_reduce, valid_elems


def rank_sets(N, workers):
    """Destination ranks dealt round-robin to ``workers`` sets (padding-only
    ranks sit at the end of a group, so round-robin balances them)."""
    workers = max(1, min(workers, N))
    return [list(range(k, N, workers)) for k in range(workers)]


def worker_inputs(w, ranks):
    """The gradients and packed all-gather shards that ``ranks`` read; every
    other entry is zero (gradients) or None (shards)."""
    geo = geometry(w.shapes, w.N)
    if sorted(ranks) == list(range(w.N)):   # every rank: whole tensors, one call each
        grads = [[bf16_tensor(w.grad_key(src, p), w.numel(p), w.dists[p], w.sigma) for p in range(w.P)]
                 for src in range(w.N)]
        return geo, grads, [w.ag_values(r, np.arange(geo.S, dtype=np.uint64)) for r in range(w.N)]
    grads = [[np.zeros(w.numel(p), dtype=np.uint16) for p in range(w.P)] for _ in range(w.N)]
    for src in range(w.N):
        for p in range(w.P):
            for r in ranks:
                a, v = r * geo.e[p], valid_elems(geo, p, r)
                if v:
                    grads[src][p][a:a + v] = w.grad_values(src, p, np.arange(a, a + v, dtype=np.uint64))
    shards = [None] * w.N
    for r in ranks:
        shards[r] = w.ag_values(r, np.arange(geo.S, dtype=np.uint64))
    return geo, grads, shards


def _worker(w, ranks, passes, seconds, warmup, start, results, want_outputs):
    geo, grads, shards = worker_inputs(w, ranks)
    params = [np.zeros(w.N * geo.e[p], dtype=np.uint16) for p in range(geo.P)]

    def one_pass():
        out = rs_reduce(geo, grads, w.M, w.L, ranks=ranks)
        ag_place(geo, shards, ranks=ranks, out=params)
        return out

    for _ in range(warmup):
        one_pass()
    results.put(("ready",))
    start.wait()
    done, t0 = 0, time.perf_counter()
    while True:
        rs = one_pass()
        done += 1
        elapsed = time.perf_counter() - t0
        if (passes is not None and done >= passes) or (passes is None and elapsed >= seconds):
            break
    out = None
    if want_outputs:
        pieces = {(p, r): params[p][r * geo.e[p]:(r + 1) * geo.e[p]].copy() for p in range(geo.P) for r in ranks}
        out = (dict(zip(ranks, rs)), pieces)
    results.put(("done", ranks, elapsed, done, out))


def _collect(results, procs, kind, count, timeout):
    """``count`` messages of ``kind``; raises if a worker died or time ran out."""
    import queue
    got, deadline = [], time.monotonic() + timeout
    while len(got) < count:
        try:
            msg = results.get(timeout=0.5)
        except queue.Empty:
            dead = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
            if dead:
                raise RuntimeError(f"an oracle worker exited with status {dead[0]}")
            if time.monotonic() > deadline:
                raise TimeoutError(f"oracle workers: {len(got)} of {count} '{kind}' reports in {timeout} s")
            continue
        if msg[0] == kind:
            got.append(msg[1:])
    return got


def run(w, workers, passes=None, seconds=10.0, warmup=0, want_outputs=False, timeout=900.0):
    """Reduce-scatter + all-gather passes of workload ``w`` over ``workers``
    processes: ``passes`` each, or, if ``passes`` is None, as many as fit in
    ``seconds`` (each worker on its own).  Each worker first does ``warmup``
    untimed passes.  Returns a dict: ``wall`` (seconds from the common start
    to the last report), ``workers`` (processes used), ``passes`` and
    ``seconds`` per worker, ``ranks`` per worker, and, if asked for,
    ``outputs`` = (N shards, P gathered blocks) merged from the workers."""
    ctx = mp.get_context("spawn")
    sets = rank_sets(w.N, workers)
    start = ctx.Event()
    results = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(w, s, passes, seconds, warmup, start, results, want_outputs),
                         daemon=True) for s in sets]
    for p in procs:
        p.start()
    try:
        _collect(results, procs, "ready", len(procs), timeout)
        t0 = time.perf_counter()
        start.set()
        reports = _collect(results, procs, "done", len(procs), timeout)
        wall = time.perf_counter() - t0
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    out = {"wall": wall, "workers": len(sets), "ranks": [r[0] for r in reports],
           "seconds": [r[1] for r in reports], "passes": [r[2] for r in reports]}
    if want_outputs:
        geo = geometry(w.shapes, w.N)
        shards = [None] * w.N
        params = [np.zeros(w.N * geo.e[p], dtype=np.uint16) for p in range(geo.P)]
        for _, _, _, (rs, pieces) in reports:
            for r, s in rs.items():
                shards[r] = s
            for (p, r), piece in pieces.items():
                params[p][r * geo.e[p]:(r + 1) * geo.e[p]] = piece
        out["outputs"] = (shards, params)
    return out

"""The five gradient-group workloads the hot path is measured and checked on.

Shapes are those of real model layers (random-initialised, synthetic values):

1. ``tiny``      N=4 (M=1, L=4): 3 parameters whose per-rank pieces are 2, 1
                 and 3 rows of 64 -- the hand-checkable layout example of the
                 "Endgame of FSDP Communication" explainer (section "What
                 problem is it actually solving?"), with one unit = one row.
2. ``llama70b``  N=8 (M=1, L=8): one Llama-3.1-70B decoder layer.
3. ``qwen3moe``  N=16 (M=2, L=8): one Qwen3-30B-A3B MoE layer, 391 tensors.
4. ``wan22dit``  N=64 (M=8, L=8): one Wan2.2 14B DiT block; 10% outliers x100.
5. ``uneven``    N=48 (M=6, L=8): 257 parameters with seeded ragged shapes
                 (rows 1..5000 incl. primes, cols 1..4096 incl. odd), so most
                 parameters carry dim-0 padding.

Values: every emulated rank's gradient tensor is a seeded bf16 stream
(``synth.gen``); all-gather inputs are seeded bf16 shards.
"""

import math
from dataclasses import dataclass, field

import numpy as np

from . import gen

AG_PARAM_STREAM = (1 << 20) - 1  # stream index reserved for all-gather shards


@dataclass
class Workload:
    name: str
    N: int
    M: int
    L: int
    shapes: list            # list of tuples, dim 0 first
    dists: list             # per-parameter value distribution (synth.gen constants)
    sigma: float = 1e-3
    seed: int = 0
    notes: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def P(self):
        return len(self.shapes)

    def numel(self, p):
        return int(np.prod(self.shapes[p], dtype=np.int64)) if len(self.shapes[p]) else 1

    def grad_key(self, rank, p):
        return gen.tensor_key(self.seed, rank, p)

    def ag_key(self, rank):
        return gen.tensor_key(self.seed, rank, AG_PARAM_STREAM)

    def grad_values(self, rank, p, idx):
        """bf16 bits of rank ``rank``'s gradient of parameter p at flat indices idx."""
        return gen.bf16_values(self.grad_key(rank, p), idx, self.dists[p], self.sigma)

    def ag_values(self, rank, idx):
        """bf16 bits of rank ``rank``'s packed all-gather shard at indices idx."""
        return gen.bf16_values(self.ag_key(rank), idx, gen.UNIFORM)

    def total_grad_elems(self):
        return sum(self.numel(p) for p in range(self.P))


def tiny():
    shapes = [(8, 64), (4, 64), (12, 64)]
    return Workload("tiny", 4, 1, 4, shapes, [gen.UNIFORM] * 3, seed=1234 + 1,
                    notes="per-rank pieces of 2, 1, 3 rows x 64; uniform[-1,1]")


def llama70b():
    h, kv, ffn = 8192, 1024, 28672
    shapes = [(h, h), (kv, h), (kv, h), (h, h), (ffn, h), (ffn, h), (h, ffn), (h,), (h,)]
    return Workload("llama70b", 8, 1, 8, shapes, [gen.NORMAL] * len(shapes), sigma=1e-3,
                    seed=1234 + 2,
                    notes="Llama-3.1-70B decoder layer: q,k,v,o, gate, up, down, 2 RMSNorm")


def qwen3moe():
    h, qd, kvd, experts, inter, router = 2048, 4096, 512, 128, 768, 128
    shapes = [(qd, h), (kvd, h), (kvd, h), (h, qd), (router, h)]
    for _ in range(experts):
        shapes += [(inter, h), (inter, h), (h, inter)]
    shapes += [(h,), (h,)]
    return Workload("qwen3moe", 16, 2, 8, shapes, [gen.NORMAL] * len(shapes), sigma=1e-3,
                    seed=1234 + 3,
                    notes="Qwen3-30B-A3B MoE layer: attention, router, 128 experts, 2 norms")


def wan22dit():
    d, f = 5120, 13824
    shapes = [(d, d)] * 8 + [(f, d), (d, f)] + [(d,)] * 3
    return Workload("wan22dit", 64, 8, 8, shapes, [gen.OUTLIER] * len(shapes), sigma=1e-3,
                    seed=1234 + 4,
                    notes="Wan2.2 DiT block: self/cross-attn q,k,v,o, FFN up/down, 3 norms; "
                          "10% of values x100")


UNEVEN_FIXED = [(1, 1), (1, 4096), (47, 1), (48, 1), (49, 3), (97, 4095), (4999, 4093),
                (5000, 4096), (4096, 4095), (2, 2047), (4093, 1), (3, 5)]


def uneven_shapes(seed, count=257, max_rows=5000, max_cols=4096):
    """12 fixed edge shapes, then log-uniform rows x cols; every other one odd-width."""
    shapes = list(UNEVEN_FIXED)
    key = gen.splitmix64_int(seed, 0xC0FFEE)
    k = count - len(shapes)
    u = gen.uniform01(key, np.arange(2 * k, dtype=np.uint64))
    for i in range(k):
        rows = min(max_rows, int(math.floor(math.exp(u[2 * i] * math.log(max_rows)))) + 1)
        cols = min(max_cols, int(math.floor(math.exp(u[2 * i + 1] * math.log(max_cols)))) + 1)
        if i % 2 == 1 and cols % 2 == 0:
            cols -= 1 if cols > 1 else -1
        shapes.append((rows, cols))
    return shapes


def uneven(max_input_bytes=48 << 30):
    N = 48
    seed = 1234 + 5
    while True:
        shapes = uneven_shapes(seed)
        g = sum(r * c for r, c in shapes)
        if 2 * N * g <= max_input_bytes:
            break
        seed += 1
    dists = [gen.UNIFORM if p % 2 == 0 else gen.INTEGER for p in range(len(shapes))]
    return Workload("uneven", N, 6, 8, shapes, dists, seed=seed,
                    notes="257 ragged params; even p uniform[-1,1], odd p integers in [-128,128]")


ALL = {1: tiny, 2: llama70b, 3: qwen3moe, 4: wan22dit, 5: uneven}
BY_NAME = {"tiny": tiny, "llama70b": llama70b, "qwen3moe": qwen3moe, "wan22dit": wan22dit,
           "uneven": uneven}


def get(which):
    if isinstance(which, int) or (isinstance(which, str) and which.isdigit()):
        return ALL[int(which)]()
    return BY_NAME[which]()


def scaled(w, row_div=1, max_rows=None, N=None, M=None, L=None, name=None):
    """A smaller copy of workload ``w`` for fast parity runs (same structure)."""
    shapes = []
    for s in w.shapes:
        r = max(1, s[0] // row_div)
        if max_rows is not None:
            r = min(r, max_rows)
        shapes.append((r,) + tuple(s[1:]))
    return Workload(name or (w.name + "_small"), N or w.N, M or w.M, L or w.L, shapes,
                    list(w.dists), sigma=w.sigma, seed=w.seed, notes="scaled " + w.notes)

"""Shared helpers of the GPU parity tests: build inputs on the host (or on the
device with the seeded generator), run libtide through its C ABI, and fetch
the oracle's answer for the same inputs."""

import numpy as np
import torch

import oracle.tide_oracle as O
from synth import configs, gen

DEV = "cuda:0"


def host_grads(w):
    """All of a workload's gradients as host uint16 arrays, grads[rank][p]."""
    return [[gen.bf16_tensor(w.grad_key(r, p), w.numel(p), w.dists[p], w.sigma) for p in range(w.P)]
            for r in range(w.N)]


def to_dev_u16(arr, pad_before=0, pad_after=0, fill=0x7FC1):
    """Copy a uint16 array to the GPU inside a guard band of sentinel values.

    Returns (view, backing): ``view`` holds the data, ``backing`` the guards.
    """
    n = arr.size
    backing = torch.full((pad_before + n + pad_after,), fill - 65536 if fill > 32767 else fill,
                         dtype=torch.int16, device=DEV)
    view = backing[pad_before:pad_before + n]
    if n:
        view.copy_(torch.from_numpy(arr.view(np.int16)))
    return view, backing


def f32_guarded(n, pad_before=0, pad_after=0, fill=float("nan")):
    backing = torch.full((pad_before + n + pad_after,), fill, dtype=torch.float32, device=DEV)
    return backing[pad_before:pad_before + n], backing


def u16_of(t):
    return t.cpu().numpy().view(np.uint16)


def f32_bits(t):
    return t.cpu().numpy().view(np.uint32)


def run_rs(plan, dev_grads, shards, stream=None):
    """dev_grads[r][p] -> call with the ABI's r*P + p ordering."""
    flat = [dev_grads[r][p] for r in range(plan.N) for p in range(plan.P)]
    plan.rs_reduce(flat, shards, stream)


def oracle_rs(w, grads):
    geo = O.geometry(w.shapes, w.N)
    return geo, O.rs_reduce(geo, grads, w.M, w.L)


def device_grads(w, stream=None):
    """A workload's gradients generated in HBM by the seeded device generator."""
    from synth import device
    out = []
    for r in range(w.N):
        row = []
        for p in range(w.P):
            t = torch.empty(w.numel(p), dtype=torch.int16, device=DEV)
            device.fill_bf16(t, w.grad_key(r, p), w.dists[p], w.sigma, stream=stream)
            row.append(t)
        out.append(row)
    return out


def device_ag_shards(w, S, stream=None):
    from synth import device
    out = []
    for r in range(w.N):
        t = torch.empty(S, dtype=torch.int16, device=DEV)
        device.fill_bf16(t, w.ag_key(r), gen.UNIFORM, stream=stream)
        out.append(t)
    return out


def workload(cfg):
    return configs.get(cfg)

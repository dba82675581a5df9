#!/usr/bin/env python
"""Benchmark of the TIDE single-GPU hot path.

One step = tide_rs_reduce (bf16 gradients of all N emulated ranks -> N packed
fp32 shards) + tide_ag_place (N packed bf16 shards -> P parameter-major
blocks) over one synthetic parameter group, everything resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload wan22dit]
    python bench.py --impl reference ...   # the CPU oracle, timed on all host cores

Prints one JSON line.  `value` is the effective HBM bandwidth of the step in
GB/s of algorithmic bytes: reduce-scatter 2*N*G (every contributor's real bf16
element read once) + 4*N*S (every fp32 shard element written once), all-gather
2*2*N*S (every bf16 piece read once and written once).  The headline workload
is the largest group, the Wan2.2 DiT block (N = 64); the same step is then
timed on the other three measured groups (Llama-3.1-70B layer, Qwen3-30B-A3B
MoE layer, the uneven padding group), one after another with each group's
buffers freed before the next, and reported under `per_config`.  Under
torchrun each rank runs its own replica on its own GPU (no data-path
collective), `value` sums all ranks' bytes over the slowest rank's time.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RS/AG effective HBM GB/s and % of GB300 HBM peak (1 GPU); elements/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, vendor figure (context beside the measured peak)
L2_FLUSH_BELOW = 1 << 30   # steps moving fewer bytes than this get an L2 flush before each timed step
L2_FLUSH_BYTES = 512 << 20
DEFAULT_WORKLOAD = "wan22dit"
# The four full-size groups the step is measured on; the default run times
# the headline workload, then the other three under `per_config`.
MEASURED_GROUPS = ("wan22dit", "llama70b", "qwen3moe", "uneven")
CLOCK_QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
               "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
               "clocks_event_reasons.sw_power_cap")
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", choices=["fused", "staged-rs", "rd-ag", "variants", "ag-ceiling"], default="fused",
                    help="fused: the hot path (RS + AG per step); staged-rs: the two-stage reduce-scatter "
                         "through an inbox; rd-ag: the all-gather by recursive-doubling exchange and stage "
                         "placement; variants: bulk-copy RS kernel, averaging / accumulating RS, "
                         "Slot-Reuse pack + RS from slots, unpadded AG, AG transports; ag-ceiling: "
                         "tide_ag_place against a plain device copy of the same bytes, each after an L2 flush")
    ap.add_argument("--variants", default="all",
                    help="variants: comma-separated subset of the timed variants (default all)")
    ap.add_argument("--ag-transport", choices=["sm", "bulk", "copy-engines"], default="sm",
                    help="how tide_ag_place moves the pieces (default: the SM kernel)")
    ap.add_argument("--nodes", type=int, default=0,
                    help="regroup the workload's N ranks as this many nodes of N / nodes GPUs (e.g. 16 for "
                         "wan22dit as 16 x 4: more nodes than GPUs per node)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="wan22dit (default), llama70b, qwen3moe, uneven or tiny")
    ap.add_argument("--per-config", default="auto",
                    help="groups also timed after the headline, under per_config: 'auto' (the other measured "
                         "groups when the headline is one of them), 'none', or a comma-separated list")
    ap.add_argument("--row-div", type=int, default=1,
                    help="divide every parameter's rows (a smaller case of the same layer, for profiling)")
    ap.add_argument("--staged-budget", choices=["both", "fill", "pages"], default="both",
                    help="staged-rs: CTA budgets timed (fill the GPU, the pages' 16 + 4 per rank, or both)")
    ap.add_argument("--inbox-offset", type=int, default=0,
                    help="staged-rs: place the inbox this many floats past a 256-byte boundary (1 forces the "
                         "4-byte landing kernels)")
    ap.add_argument("--rd-exchange", choices=["both", "copy-engines", "sm"], default="both",
                    help="rd-ag: exchange transports timed")
    ap.add_argument("--rd-mode", choices=["both", "rails", "per-rail"], default="both",
                    help="rd-ag: every rail at once, rail by rail, or both")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle time budget of cpu_baseline")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- plumbing

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(local_seconds, local_units, world, device="cpu"):
    """(max seconds over ranks, summed units over ranks)."""
    if world == 1:
        return local_seconds, local_units
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    u = torch.tensor([local_units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def algorithmic_bytes(w, geo):
    """RS: 2*N*G + 4*N*S; AG (bf16): 2*2*N*S.  Also the element counts."""
    G = w.total_grad_elems()
    N, S = w.N, geo.S
    return {"rs_bytes": 2 * N * G + 4 * N * S, "ag_bytes": 4 * N * S,
            "rs_elems": N * G, "ag_elems": N * S, "G": G, "S": S}


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest(name):
    path = os.path.join(ROOT, "fsdp_layout_aware_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def profile_fields(summary_name):
    """The `key: value` lines of a committed ncu summary under profiles/."""
    fields = {}
    with open(os.path.join(ROOT, "profiles", summary_name)) as f:
        for line in f:
            if ":" in line and not line.startswith(" "):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    return fields


def profiled_traffic(summary_name, kernel_file, alg_read_full, alg_write_full):
    """DRAM traffic of one full-size launch, from a committed ncu summary of a
    smaller capture of the same kernel (a rows/k case of the same group), if
    the kernel source it was taken on is the current one; otherwise None.

    Reads grow with the contributor bytes, so the captured DRAM reads are
    scaled by (full-size algorithmic reads / captured algorithmic reads).
    Writes are not scaled: at the end of a launch part of them is still dirty
    in L2 (tens of MB whatever the size), so a scaled capture would credit
    that residue many times over; the full launch's algorithmic writes stand
    in for them."""
    try:
        f = profile_fields(summary_name)
        if f.get("kernel_source_sha256") != kernel_source_digest(kernel_file):
            return None
        reads, writes = float(f["dram_bytes_read"]), float(f["dram_bytes_write"])
        alg_r, alg_w = float(f["algorithmic_read_bytes_captured"]), float(f["algorithmic_write_bytes_captured"])
    except (OSError, KeyError, ValueError):
        return None
    scale = alg_read_full / alg_r
    return {"bytes": round(reads * scale + alg_write_full),
            "source": (f"{f.get('workload_captured', 'a smaller capture')}: DRAM reads x {scale:g} "
                       f"+ the full launch's algorithmic writes ({summary_name})"),
            "captured_dram_read_over_algorithmic": round(reads / alg_r, 4),
            "captured_dram_write_over_algorithmic": round(writes / alg_w, 4)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    MIN_RUN_S = 1.5   # nvidia-smi needs about a second before its first sample

    def start(self):
        self.t_start = time.time()
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + CLOCK_QUERY, "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu_index)], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self, windows):
        """Median SM clock and the throttle reasons seen in samples taken
        inside any of the (t0, t1) wall-clock windows (all samples if none)."""
        if self.proc is None:
            return None
        time.sleep(max(0.0, self.t_start + self.MIN_RUN_S - time.time()))
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) != 9:
                    continue
                try:
                    ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if any(t0 <= r[0] <= t1 for t0, t1 in windows)] or rows
        if not inside:
            return None
        reasons = sorted({REASON_NAMES[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------- our arm

def get_workload(args):
    from synth import configs
    w = configs.get(args.workload)
    if args.row_div > 1:
        w = configs.scaled(w, row_div=args.row_div, name=f"{w.name}_rows{args.row_div}")
    if args.nodes:
        if w.N % args.nodes:
            raise SystemExit(f"--nodes {args.nodes} does not divide N = {w.N}")
        w = configs.scaled(w, M=args.nodes, L=w.N // args.nodes, name=f"{w.name}_{args.nodes}x{w.N // args.nodes}")
    return w


def per_config_groups(args):
    """Groups timed after the headline one, under per_config."""
    if args.per_config == "none":
        return []
    if args.per_config == "auto":
        if args.workload not in MEASURED_GROUPS or args.nodes:
            return []
        return [g for g in MEASURED_GROUPS if g != args.workload]
    from synth import configs
    names = [g.strip() for g in args.per_config.split(",") if g.strip()]
    unknown = [g for g in names if g not in configs.BY_NAME]
    if unknown:
        raise SystemExit(f"--per-config: unknown group(s) {', '.join(unknown)} (known: {', '.join(configs.BY_NAME)})")
    return names


def allocate_group(w, plan, dev, stream):
    """Every rank's bf16 gradients and bf16 packed all-gather shards, filled
    in HBM by the seeded generator, plus the outputs of both calls."""
    import torch

    from synth import device, gen
    S = plan.S
    with torch.cuda.stream(stream):
        grads = []
        for r in range(w.N):
            for p in range(w.P):
                t = torch.empty(w.numel(p), dtype=torch.int16, device=dev)
                device.fill_bf16(t, w.grad_key(r, p), w.dists[p], w.sigma, stream=stream)
                grads.append(t)
        rs_out = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(w.N)]
        ag_in = []
        for r in range(w.N):
            t = torch.empty(S, dtype=torch.int16, device=dev)
            device.fill_bf16(t, w.ag_key(r), gen.UNIFORM, stream=stream)
            ag_in.append(t)
        ag_out = [torch.empty(w.N * plan.e[p], dtype=torch.int16, device=dev) for p in range(w.P)]
    stream.synchronize()
    return grads, rs_out, ag_in, ag_out


def time_group(args, w, world, dev, stream, windows, keep=False):
    """Warm-up, then K timed steps of one group: one tide_rs_reduce and one
    tide_ag_place per step on one stream, CUDA events around every call and
    around the K steps, a barrier and a device synchronisation on both sides.
    Appends the timed wall-clock window to `windows`."""
    import torch

    import fsdp_layout_aware_gb300 as tide
    plan = tide.TidePlan(w.shapes, w.N, w.M, w.L)
    plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, {"sm": tide.TIDE_AG_SM, "bulk": tide.TIDE_AG_BULK,
                                                 "copy-engines": tide.TIDE_AG_COPY_ENGINES}[args.ag_transport])
    nbytes = algorithmic_bytes(w, plan)
    grads, rs_out, ag_in, ag_out = allocate_group(w, plan, dev, stream)
    # Device addresses marshalled once, as a caller reusing its buffers would.
    ptrs = (tide.pointer_array(grads), tide.pointer_array(rs_out), tide.pointer_array(ag_in),
            tide.pointer_array(ag_out))

    for _ in range(args.warmup):
        plan.rs_reduce(ptrs[0], ptrs[1], stream)
        plan.ag_place(ptrs[2], ptrs[3], 2, stream)
    stream.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # A step whose bytes would largely fit in the 129 MB L2 gets an L2 flush
    # (a 512 MiB fill) before each timed step; the fill is outside the
    # per-step events and the step time is then their sum.
    flush = (torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
             if nbytes["rs_bytes"] + nbytes["ag_bytes"] < L2_FLUSH_BELOW else None)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    launches = [0, 0]  # kernels launched by the RS and AG calls (the library's own count)
    start.record(stream)
    for k in range(K):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(k & 0xFF)
        ev[k][0].record(stream)
        plan.rs_reduce(ptrs[0], ptrs[1], stream)
        launches[0] += plan.last_launches()
        ev[k][1].record(stream)
        plan.ag_place(ptrs[2], ptrs[3], 2, stream)
        launches[1] += plan.last_launches()
        ev[k][2].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    windows.append((t_wall0, time.time()))
    barrier(world)
    plan.check()

    rs_all = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    ag_all = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)]
    flush_used = flush is not None
    if flush is None:
        local_s = start.elapsed_time(stop) / 1e3
    else:
        local_s = sum(ev[k][0].elapsed_time(ev[k][2]) for k in range(K)) / 1e3
        del flush
    rs_ms, ag_ms = statistics.mean(rs_all), statistics.mean(ag_all)
    step_bytes = nbytes["rs_bytes"] + nbytes["ag_bytes"]
    max_s, total_bytes = aggregate(local_s, float(step_bytes * K), world, device=dev)
    _, total_elems = aggregate(local_s, float((nbytes["rs_elems"] + nbytes["ag_elems"]) * K), world, device=dev)
    res = {"w": w, "plan": plan, "nbytes": nbytes, "max_s": max_s, "total_bytes": total_bytes,
           "total_elems": total_elems, "rs_ms": rs_ms, "ag_ms": ag_ms, "launches": launches,
           "rs_ms_median": statistics.median(rs_all), "ag_ms_median": statistics.median(ag_all),
           "l2": (f"no flush: {(nbytes['rs_bytes'] + nbytes['ag_bytes']) / 1e9:.1f} GB of inputs and outputs "
                  f"per step >> 129 MB L2" if flush_used is False else
                  f"L2 flushed (512 MiB fill) before each timed step, outside the step's events: "
                  f"{nbytes['rs_bytes'] + nbytes['ag_bytes']} bytes per step")}
    res["rs_ms_uploading"], res["ag_ms_uploading"] = time_table_uploads(plan, w, dev, stream, grads, ag_in, ptrs,
                                                                        min(K, 10))
    if keep:
        res["buffers"] = (grads, rs_out, ag_in, ag_out, ptrs)
    else:
        plan.close()
        del grads, rs_out, ag_in, ag_out, ptrs
        torch.cuda.empty_cache()
    return res


def time_table_uploads(plan, w, dev, stream, grads, ag_in, ptrs, K):
    """Mean time of a call that must upload its pointer table: calls
    alternate between the timed output buffers and a second set, so each
    call's table differs from the one before (outside the timed region of
    the step; the steady state of the step reuses its tables)."""
    import torch

    import fsdp_layout_aware_gb300 as tide
    rs_out2 = [torch.empty(plan.S, dtype=torch.float32, device=dev) for _ in range(w.N)]
    ag_out2 = [torch.empty(w.N * plan.e[p], dtype=torch.int16, device=dev) for p in range(w.P)]
    rs_sets = [ptrs[1], tide.pointer_array(rs_out2)]
    ag_sets = [ptrs[3], tide.pointer_array(ag_out2)]
    out = []
    for call in (lambda k: plan.rs_reduce(ptrs[0], rs_sets[k % 2], stream),
                 lambda k: plan.ag_place(ptrs[2], ag_sets[k % 2], 2, stream)):
        call(1)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
        torch.cuda.synchronize()
        ev[0].record(stream)
        for k in range(K):
            call(k)
            ev[k + 1].record(stream)
        torch.cuda.synchronize()
        out.append(statistics.mean(ev[k].elapsed_time(ev[k + 1]) for k in range(K)))
    del rs_out2, ag_out2
    return out[0], out[1]


def call_stats(g, peak):
    """Per-call figures of a timed group: mean over the K timed calls (what
    GB/s and frac use) and the median beside it."""
    nbytes = g["nbytes"]
    out = []
    for call in ("rs", "ag"):
        ms = g[call + "_ms"]
        gbs = nbytes[call + "_bytes"] / ms / 1e6
        out.append({"ms": round(ms, 4), "ms_median": round(g[call + "_ms_median"], 4), "GB_s": round(gbs, 2),
                    "frac": round(gbs / peak, 4), "elements_per_s": round(nbytes[call + "_elems"] / ms * 1e3, 1),
                    "ms_uploading_pointer_table": round(g[call + "_ms_uploading"], 4)})
    return out[0], out[1]


def run_ours(args, rank, world, local_rank):
    import torch

    groups = per_config_groups(args)   # validated before any GPU work
    torch.cuda.set_device(local_rank)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=dev)
    peak, peak_kind = measured_hbm_peak()
    K = args.steps
    windows = []
    sampler = ClockSampler(local_rank).start() if rank == 0 else None
    if sampler:
        time.sleep(0.4)   # let nvidia-smi come up before the first timed region

    head = time_group(args, get_workload(args), world, dev, stream, windows, keep=True)
    w, plan, nbytes = head["w"], head["plan"], head["nbytes"]
    grads, rs_out, ag_in, ag_out, ptrs = head.pop("buffers")
    e2e = None if args.no_e2e else run_e2e(args, plan, w, nbytes, grads, rs_out, ag_in, ag_out, stream, world, dev,
                                            ptrs)
    plan.close()
    del grads, rs_out, ag_in, ag_out, ptrs, head["plan"]
    torch.cuda.empty_cache()

    per_config = {}
    for name in groups:
        sub = argparse.Namespace(**{**vars(args), "workload": name, "nodes": 0})
        g = time_group(args, get_workload(sub), world, dev, stream, windows)
        rs, ag = call_stats(g, peak)
        step_gbs = g["total_bytes"] / g["max_s"] / 1e9
        per_config[name] = {
            "workload": f"{g['w'].name}: {g['w'].notes}", "N": g["w"].N, "M": g["w"].M, "L": g["w"].L,
            "P": g["w"].P, "rs_bytes_per_step": g["nbytes"]["rs_bytes"],
            "ag_bytes_per_step": g["nbytes"]["ag_bytes"], "ms_per_step": round(g["max_s"] / K * 1e3, 4),
            "GB_s": round(step_gbs, 2), "frac": round(step_gbs / peak, 4), "rs": rs, "ag": ag,
            "gpu_launches": g["launches"][0] + g["launches"][1], "l2": g["l2"]}
    clocks = sampler.stop(windows) if sampler else None

    if rank != 0:
        return None
    max_s, launches = head["max_s"], head["launches"]
    value = head["total_bytes"] / max_s / 1e9
    rs, ag = call_stats(head, peak)
    traffic = profiled_traffic(f"rs_fused_{w.name}.txt", "rs_kernel.cu", 2 * nbytes["rs_elems"],
                               4 * w.N * nbytes["S"])
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(max_s / K * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 bf16; shapes of the named layer)",
        "config": {"workload": f"{w.name}: {w.notes}", "N": w.N, "M": w.M, "L": w.L, "P": w.P,
                   "G_elems": nbytes["G"], "S_elems": nbytes["S"], "rs_bytes_per_step": nbytes["rs_bytes"],
                   "ag_bytes_per_step": nbytes["ag_bytes"],
                   "l2": head["l2"],
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "elements_per_s": round(head["total_elems"] / max_s, 1),
        "rs": rs,
        "ag": ag,
        "roofline": {"kernel": "rs_fused", "bound": "hbm", "achieved": rs["GB_s"], "peak": peak,
                     "peak_source": peak_kind, "unit": "GB/s", "frac": rs["frac"],
                     "traffic": traffic["bytes"] if traffic else None,
                     "traffic_source": traffic["source"] if traffic else None,
                     "algorithmic_bytes_per_launch": nbytes["rs_bytes"],
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": round(rs["GB_s"] / NOMINAL_HBM_GBS, 4)},
        "per_config": per_config,
        "gpu_launches": launches[0] + launches[1],
        "kernels_per_step": {"rs": launches[0] / K, "ag": launches[1] / K},
        "ag_transport": args.ag_transport,
        "clocks": clocks,
        "e2e": e2e,
    }
    if traffic:
        line["roofline"]["traffic_captured_ratios"] = {
            "dram_read_over_algorithmic": traffic["captured_dram_read_over_algorithmic"],
            "dram_write_over_algorithmic": traffic["captured_dram_write_over_algorithmic"]}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], line["cpu_baseline_all_cores"] = cpu_baselines(args.workload, args.cpu_seconds)
    return line


def _time_steps(step, K, stream, world, dev, nbytes):
    import torch
    step()
    stream.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(K):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return aggregate(a.elapsed_time(b) / 1e3, float((nbytes["rs_bytes"] + nbytes["ag_bytes"]) * K), world, device=dev)


def host_available_bytes():
    """Host memory this process can still take: MemAvailable, capped by the
    cgroup's limit when one is set; None if neither can be read."""
    vals = []
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    vals.append(int(line.split()[1]) * 1024)
    except (OSError, ValueError, IndexError):
        pass
    try:
        with open("/sys/fs/cgroup/memory.max") as f:
            lim = f.read().strip()
        with open("/sys/fs/cgroup/memory.current") as f:
            cur = int(f.read().strip())
        if lim != "max":
            vals.append(int(lim) - cur)
    except (OSError, ValueError):
        pass
    return min(vals) if vals else None


def all_ranks_ok(ok, world, dev):
    """True only if `ok` holds on every rank (so all ranks take the same branch)."""
    if world == 1:
        return ok
    import torch
    import torch.distributed as dist
    t = torch.tensor([1 if ok else 0], dtype=torch.int32, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return bool(t.item())


def run_e2e(args, plan, w, nbytes, grads, rs_out, ag_in, ag_out, stream, world, dev, ptrs):
    """The step through the C ABI with HOST buffers.

    Inputs (every rank's gradients and packed shards) live in pinned host
    memory and outputs are written to pinned host memory.  On GB300 a pinned
    host address is a valid device address, so the library's kernels read the
    inputs and write the results across NVLink-C2C themselves (45.7 GB in and
    2.1 GB out per wan22dit step, 15.4 GB in and 5.1 GB out per llama70b
    step); the link is the bound.  For context the
    same step is also timed with explicit staging: copy every input to device
    buffers, run on the device, copy every output back.
    """
    import torch

    import fsdp_layout_aware_gb300 as tide
    need = sum(t.numel() * t.element_size() for t in grads + ag_in + rs_out + ag_out)
    local = int(os.environ.get("LOCAL_WORLD_SIZE", world))
    avail = host_available_bytes()
    why = None
    if avail is not None and need * local > 0.6 * avail:
        why = (f"needs {need / 1e9:.1f} GB of pinned host memory per rank x {local} ranks; "
               f"{avail / 1e9:.1f} GB available")
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h_grads = h_ag_in = h_rs_out = h_ag_out = []
    if why is None:
        try:
            h_grads, h_ag_in = [pin(t) for t in grads], [pin(t) for t in ag_in]
            h_rs_out, h_ag_out = [pin(t) for t in rs_out], [pin(t) for t in ag_out]
        except RuntimeError as err:
            why = f"pinned host allocation of {need / 1e9:.1f} GB failed: {str(err).splitlines()[0][:120]}"
    if not all_ranks_ok(why is None, world, dev):
        del h_grads, h_ag_in, h_rs_out, h_ag_out
        return {"value": None, "unit": "GB/s", "unavailable": why or "another rank could not pin its host buffers"}
    with torch.cuda.stream(stream):
        for h, d in zip(h_grads + h_ag_in, grads + ag_in):
            h.copy_(d, non_blocking=True)
    stream.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in h_grads + h_ag_in)
    d2h = sum(t.numel() * t.element_size() for t in h_rs_out + h_ag_out)
    hp = [tide.pointer_array(x) for x in (h_grads, h_rs_out, h_ag_in, h_ag_out)]

    def step_host():
        plan.rs_reduce(hp[0], hp[1], stream)
        plan.ag_place(hp[2], hp[3], 2, stream)

    def step_staged():
        with torch.cuda.stream(stream):
            for d, h in zip(grads + ag_in, h_grads + h_ag_in):
                d.copy_(h, non_blocking=True)
            plan.rs_reduce(ptrs[0], ptrs[1], stream)
            plan.ag_place(ptrs[2], ptrs[3], 2, stream)
            for h, d in zip(h_rs_out + h_ag_out, rs_out + ag_out):
                h.copy_(d, non_blocking=True)

    K = max(1, args.e2e_steps)
    max_s, tot = _time_steps(step_host, K, stream, world, dev, nbytes)
    st_s, st_tot = _time_steps(step_staged, K, stream, world, dev, nbytes)
    return {"value": round(tot / max_s / 1e9, 3), "unit": "GB/s", "steps": K,
            "ms_per_step": round(max_s / K * 1e3, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "mode": "host buffers passed to the C ABI; kernels read inputs and write outputs over NVLink-C2C",
            "staged": {"value": round(st_tot / st_s / 1e9, 3), "ms_per_step": round(st_s / K * 1e3, 3),
                       "mode": "cudaMemcpy of every input in and every output out around the device call"}}


# ---------------------------------------------------------------- CPU oracle

# Row divisors of the CPU samples: every large parameter keeps whole per-rank
# pieces (wan22dit rows/80: one row of every 5120-row parameter per rank).
SAMPLE_ROW_DIV = {"llama70b": 64, "qwen3moe": 16, "wan22dit": 80, "uneven": 8, "tiny": 1}


def oracle_sample(workload_name):
    """A row subset of the workload (same row lengths, N, M, L) for CPU timing."""
    from synth import configs
    div = SAMPLE_ROW_DIV.get(workload_name, 16)
    w = configs.get(workload_name)
    return (configs.scaled(w, row_div=div, name=f"{w.name}_rows{div}") if div > 1 else w), div


def rank_bytes(w, geo, ranks):
    """Algorithmic bytes of the reduce-scatter and all-gather work of the
    given destination ranks (summed over all ranks: 2*N*G + 4*N*S + 4*N*S)."""
    import oracle.tide_oracle as O
    return sum(2 * w.N * sum(O.valid_elems(geo, p, r) for p in range(geo.P)) + 4 * geo.S + 4 * geo.S
               for r in ranks)


def host_info():
    """The host the CPU baseline ran on: architecture, logical cores, CPU model."""
    import platform
    model = platform.processor() or ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"machine": platform.machine(), "nproc": os.cpu_count(), "cpu": model}


def usable_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baselines(name, seconds):
    """The oracle as it stands, timed on a row sample of the workload: on one
    host core (every destination rank in one process), and on all host cores
    (the destination ranks dealt to one process per core, each running the
    same oracle functions on its own ranks; oracle.parallel).  Each leg runs
    whole passes until `seconds` have gone by."""
    import oracle.parallel as OP
    import oracle.tide_oracle as O
    ws, div = oracle_sample(name)
    geo = O.geometry(ws.shapes, ws.N)
    nb = algorithmic_bytes(ws, geo)
    host = host_info()
    one = OP.run(ws, 1, passes=None, seconds=seconds, warmup=1)
    el, passes = one["seconds"][0], one["passes"][0]
    single = {"value": round((nb["rs_bytes"] + nb["ag_bytes"]) * passes / el / 1e9, 4), "unit": "GB/s",
              "cores": 1, "kind": "oracle", "host": host,
              "sample": f"{name} rows/{div} (N={ws.N}, G={nb['G']}, S={nb['S']}): {passes} passes of RS+AG "
                        f"in {el:.1f} s in one process (numpy)",
              "elements_per_s": round((nb["rs_elems"] + nb["ag_elems"]) * passes / el, 1)}
    cores = usable_cores()
    mt = OP.run(ws, cores, passes=None, seconds=seconds, warmup=1)
    done = sum(rank_bytes(ws, geo, ranks) * n for ranks, n in zip(mt["ranks"], mt["passes"]))
    multi = {"value": round(done / mt["wall"] / 1e9, 4), "unit": "GB/s", "cores": mt["workers"],
             "kind": "oracle, destination ranks split over one process per core", "host": host,
             "sample": f"{name} rows/{div}: {mt['workers']} processes, {min(mt['passes'])}-{max(mt['passes'])} "
                       f"passes each over their ranks in {mt['wall']:.1f} s (numpy)",
             "speedup_over_one_core": None}
    multi["speedup_over_one_core"] = round(multi["value"] / single["value"], 2) if single["value"] else None
    return single, multi


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: rank 0 times K steps, each one
    RS+AG pass over a row subset of the workload, on all host cores (the
    destination ranks dealt to one process per core, each running the
    oracle's own functions on its ranks; oracle.parallel), after W untimed
    passes in every process."""
    if rank != 0:
        return None
    import oracle.parallel as OP
    import oracle.tide_oracle as O
    ws, div = oracle_sample(args.workload)
    geo = O.geometry(ws.shapes, ws.N)
    nb = algorithmic_bytes(ws, geo)
    K = max(1, args.steps)
    res = OP.run(ws, usable_cores(), passes=K, warmup=args.warmup)
    el = res["wall"]
    value = (nb["rs_bytes"] + nb["ag_bytes"]) * K / el / 1e9
    sample = (f"{args.workload} rows/{div} (N={ws.N}, G={nb['G']}, S={nb['S']}) per step, "
              f"{res['workers']} processes on the host cores, destination ranks split among them (numpy)")
    w = get_workload(args)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(el / K * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 bf16)",
        "config": {"workload": f"{w.name}: {w.notes}", "N": w.N, "M": w.M, "L": w.L, "P": w.P,
                   "sample_row_div": div},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": res["workers"], "kind": "oracle",
                         "sample": sample, "host": host_info()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "elements_per_s": round((nb["rs_elems"] + nb["ag_elems"]) * K / el, 1),
    }


def _setup_inputs(args, local_rank, need_grads=True, need_ag=True):
    import torch

    import fsdp_layout_aware_gb300 as tide
    from synth import device, gen
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = get_workload(args)
    plan = tide.TidePlan(w.shapes, w.N, w.M, w.L)
    stream = torch.cuda.Stream(device=dev)
    grads, ag_in = [], []
    with torch.cuda.stream(stream):
        if need_grads:
            for r in range(w.N):
                for p in range(w.P):
                    t = torch.empty(w.numel(p), dtype=torch.int16, device=dev)
                    device.fill_bf16(t, w.grad_key(r, p), w.dists[p], w.sigma, stream=stream)
                    grads.append(t)
        if need_ag:
            for r in range(w.N):
                t = torch.empty(plan.S, dtype=torch.int16, device=dev)
                device.fill_bf16(t, w.ag_key(r), gen.UNIFORM, stream=stream)
                ag_in.append(t)
    stream.synchronize()
    return w, plan, stream, dev, grads, ag_in


def _event_time(fn, K, W, stream):
    import torch
    for _ in range(W):
        fn()
    stream.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(K):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / K


def run_staged_rs(args, local_rank):
    """The two-stage reduce-scatter (summing kernel into the inbox, landing
    kernel), filling the GPU and with the pages' 16 + 4 CTAs per rank."""
    import torch

    import fsdp_layout_aware_gb300 as tide
    w, plan, stream, dev, grads, _ = _setup_inputs(args, local_rank, need_ag=False)
    nb = algorithmic_bytes(w, plan)
    shards = [torch.empty(plan.S, dtype=torch.float32, device=dev) for _ in range(w.N)]
    inbox_store = torch.empty(tide.tide_plan_inbox_elems(plan.handle) + args.inbox_offset, dtype=torch.float32,
                              device=dev)
    inbox = inbox_store[args.inbox_offset:]
    gp, sp = tide.pointer_array(grads), tide.pointer_array(shards)
    inbox_bytes = 8 * w.M * w.N * plan.S
    out = {"path": "staged-rs", "metric": METRIC, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
           "warmup": args.warmup, "dtype": "f32", "data": "synthetic",
           "config": {"workload": f"{w.name}: {w.notes}", "N": w.N, "M": w.M, "L": w.L,
                      "rs_bytes_per_step": nb["rs_bytes"], "inbox_extra_bytes_per_step": inbox_bytes,
                      "inbox_offset_floats": args.inbox_offset}}
    budgets = [("fill", (0, 0)), ("pages_16_4", (16, 4))]
    budgets = [b for b in budgets if args.staged_budget == "both" or b[0].startswith(args.staged_budget)]
    for name, budget in budgets:
        t = _event_time(lambda: tide.tide_rs_staged(plan.handle, gp, sp, inbox, *budget, stream=stream),
                        args.steps, args.warmup, stream)
        out[name] = {"ms": round(t * 1e3, 4), "GB_s_algorithmic": round(nb["rs_bytes"] / t / 1e9, 1),
                     "GB_s_with_inbox": round((nb["rs_bytes"] + inbox_bytes) / t / 1e9, 1)}
    t = _event_time(lambda: plan.rs_reduce(gp, sp, stream), args.steps, args.warmup, stream)
    out["fused_ms"] = round(t * 1e3, 4)
    out["value"] = out[budgets[0][0]]["GB_s_algorithmic"]
    return out


def run_rd_ag(args, local_rank):
    """The all-gather the pages' way for one destination node: the
    recursive-doubling exchange between the M nodes' stage buffers (copy
    engines or SM kernel), then the strided stage placement into the
    parameters; timed rail by rail, and for every rail at once (stage init,
    the exchange of all rails, one placement), which is `value`."""
    import torch

    import fsdp_layout_aware_gb300 as tide
    w, plan, stream, dev, _, ag_in = _setup_inputs(args, local_rank, need_grads=False)
    M, L, S = w.M, w.L, plan.S
    stage_rows = torch.empty((M, M * S), dtype=torch.int16, device=dev)   # rows of one buffer
    stages = [stage_rows[n] for n in range(M)]
    params = [torch.empty(w.N * plan.e[p], dtype=torch.int16, device=dev) for p in range(w.P)]
    pp = tide.pointer_array(params)

    def step():
        for rail in range(L):
            for n in range(M):
                stages[n][:S].copy_(ag_in[n * L + rail], non_blocking=True)
            tide.tide_ag_rd_exchange(plan.handle, stages, 2, stream)
            tide.tide_ag_stage_place(plan.handle, stages[0], 0, rail, pp, 2, stream)

    # Every rail at once (the rails run concurrently on the pages): one stage
    # init launch, the rounds of all rails, one placement from the slots.
    all_rows = torch.empty((L * M, M * S), dtype=torch.int16, device=dev)
    all_stages = [all_rows[i] for i in range(L * M)]
    sh_p, st_p = tide.pointer_array(ag_in), tide.pointer_array(all_stages)
    slot_p = tide.pointer_array(tide.stage_shard_pointers(all_stages, 0, M, L, S, 2))

    def step_rails():
        tide.tide_ag_stage_init(plan.handle, sh_p, st_p, 2, stream)
        tide.tide_ag_rd_exchange_rails(plan.handle, st_p, 2, stream)
        plan.ag_place(slot_p, pp, 2, stream)

    # bytes moved per step (read + write): every shard into its slot 0, the
    # M - 1 pieces every node receives per rail, and the placement
    init_bytes = 4 * w.N * S
    place_bytes = 4 * w.N * S
    exch_bytes = L * M * (M - 1) * S * 2 * 2
    moved = init_bytes + place_bytes + exch_bytes
    res, res_rails = {}, {}
    picked = {"both": ("copy_engines", "sm_kernel"), "copy-engines": ("copy_engines",), "sm": ("sm_kernel",)}
    transports = [(n, m) for n, m in (("copy_engines", 0), ("sm_kernel", 1)) if n in picked[args.rd_exchange]]
    with torch.cuda.stream(stream):
        for name, mode in transports:
            plan.set_option(tide.TIDE_OPT_RD_EXCHANGE, mode)
            if args.rd_mode in ("both", "per-rail"):
                t = _event_time(step, max(1, args.steps // 8), args.warmup, stream)
                res[name] = {"ms_per_step": round(t * 1e3, 4), "GB_s": round(moved / t / 1e9, 1)}
            if args.rd_mode in ("both", "rails"):
                t = _event_time(step_rails, args.steps, args.warmup, stream)
                res_rails[name] = {"ms_per_step": round(t * 1e3, 4), "GB_s": round(moved / t / 1e9, 1)}
        ta = _event_time(lambda: plan.ag_place(tide.pointer_array(ag_in), pp, 2, stream), args.steps, args.warmup,
                         stream)
    plan.check()
    head = (res_rails or res)[transports[0][0]]
    return {"path": "rd-ag", "metric": METRIC, "unit": "GB/s", "n_gpus": 1, "dtype": "bf16 copy", "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.notes}", "N": w.N, "M": M, "L": L,
                       "rounds": tide.tide_rd_rounds(M)},
            "stage_init_bytes": init_bytes, "placement_bytes": place_bytes, "exchange_bytes": exch_bytes,
            "exchange": res, "exchange_all_rails": res_rails,
            "ms_per_step": head["ms_per_step"], "value": head["GB_s"],
            "direct_landing_ms": round(ta * 1e3, 4)}


def run_variants(args, local_rank):
    """The listed variants, each timed alone on the workload: the reduce-scatter
    on the bulk-copy kernel (M <= 8) and through the entry point without
    device allocation, averaged over N and/or accumulated into
    the previous shard, Slot-Reuse
    (pack into the vacated all-gather slot, then the reduce-scatter reading
    the slots), and the all-gather writing only the real rows."""
    import torch

    import fsdp_layout_aware_gb300 as tide
    w, plan, stream, dev, grads, ag_in = _setup_inputs(args, local_rank)
    nb = algorithmic_bytes(w, plan)
    N, S, G = w.N, plan.S, nb["G"]
    shards = [torch.zeros(S, dtype=torch.float32, device=dev) for _ in range(N)]
    gp, sp, ap = tide.pointer_array(grads), tide.pointer_array(shards), tide.pointer_array(ag_in)
    params = [torch.empty(N * plan.e[p], dtype=torch.int16, device=dev) for p in range(w.P)]
    pp = tide.pointer_array(params)
    res = {}

    picked = None if args.variants == "all" else {v.strip() for v in args.variants.split(",")}

    def timed(name, fn, nbytes, setup=None):
        if picked is not None and name not in picked:
            return
        with torch.cuda.stream(stream):
            t = _event_time(fn, args.steps, args.warmup, stream)
        res[name] = {"ms": round(t * 1e3, 4), "bytes": nbytes, "GB_s": round(nbytes / t / 1e9, 1)}

    timed("rs_plain", lambda: plan.rs_reduce(gp, sp, stream), nb["rs_bytes"])
    # the entry point without device allocation: tables built per call in its static buffer
    timed("rs_noalloc", lambda: tide.tide_rs_reduce_noalloc(plan.handle, gp, sp, stream), nb["rs_bytes"])
    if w.M <= 8:  # the bulk-copy pipeline holds at most 8 node partials per thread
        plan.set_option(tide.TIDE_OPT_RS_KERNEL, 1)
        timed("rs_bulk", lambda: plan.rs_reduce(gp, sp, stream), nb["rs_bytes"])
        plan.set_option(tide.TIDE_OPT_RS_KERNEL, 0)
    plan.set_option(tide.TIDE_OPT_RS_AVERAGE, 1)
    timed("rs_average", lambda: plan.rs_reduce(gp, sp, stream), nb["rs_bytes"])
    plan.set_option(tide.TIDE_OPT_RS_ACCUMULATE, 1)
    timed("rs_average_accumulate", lambda: plan.rs_reduce(gp, sp, stream), nb["rs_bytes"] + 4 * N * S)
    plan.set_option(tide.TIDE_OPT_RS_AVERAGE, 0)
    plan.set_option(tide.TIDE_OPT_RS_ACCUMULATE, 0)
    plan.set_option(tide.TIDE_OPT_AG_UNPADDED, 1)
    timed("ag_unpadded", lambda: plan.ag_place(ap, pp, 2, stream), 4 * G)
    plan.set_option(tide.TIDE_OPT_AG_UNPADDED, 0)
    for name, transport in (("ag_copy_engines", tide.TIDE_AG_COPY_ENGINES), ("ag_bulk", tide.TIDE_AG_BULK),
                            ("ag_sm", tide.TIDE_AG_SM)):
        plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, transport)
        timed(name, lambda: plan.ag_place(ap, pp, 2, stream), nb["ag_bytes"])
    # copy engines with the shards as rows of one buffer: one strided copy per parameter
    ag_rows = torch.empty((N, S), dtype=torch.int16, device=dev)
    for r in range(N):
        ag_rows[r].copy_(ag_in[r])
    rows_p = tide.pointer_array([ag_rows[r] for r in range(N)])
    plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, tide.TIDE_AG_COPY_ENGINES)
    timed("ag_copy_engines_rows", lambda: plan.ag_place(rows_p, pp, 2, stream), nb["ag_bytes"])
    plan.set_option(tide.TIDE_OPT_AG_TRANSPORT, tide.TIDE_AG_SM)
    del params, pp, ag_rows
    # Slot-Reuse: every rank's slot is its N*S-element all-gather destination
    slots = [torch.empty(N * S, dtype=torch.int16, device=dev) for _ in range(N)]
    slp = tide.pointer_array(slots)
    timed("slot_pack", lambda: tide.tide_slot_pack(plan.handle, gp, slp, stream), 4 * N * G)
    timed("rs_from_slots", lambda: tide.tide_rs_reduce_slots(plan.handle, slp, sp, stream), nb["rs_bytes"])
    plan.check()
    head = res.get("rs_average_accumulate") or next(iter(res.values()), {"GB_s": None})
    return {"path": "variants", "metric": METRIC, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "dtype": "f32 sums of bf16", "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.notes}", "N": N, "M": w.M, "L": w.L, "G": G, "S": S},
            "value": head["GB_s"], "variants": res}


def run_ag_ceiling(args, local_rank):
    """The all-gather against the copy ceiling at its own size: for each
    group, tide_ag_place and a plain device-to-device copy (torch copy_) of
    the same bytes (N*S bf16 read and written), each timed alone with CUDA
    events right after a 512 MiB fill that flushes L2, median of K."""
    import torch

    import fsdp_layout_aware_gb300 as tide
    from synth import device, gen
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    peak, _ = measured_hbm_peak()

    def median_ms(fn):
        ts = []
        for _ in range(max(1, args.steps)):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    groups = [args.workload] + (per_config_groups(args) if args.workload in MEASURED_GROUPS else [])
    out = {}
    for name in groups:
        sub = argparse.Namespace(**{**vars(args), "workload": name, "nodes": 0})
        w = get_workload(sub)
        plan = tide.TidePlan(w.shapes, w.N, w.M, w.L)
        shards = []
        for r in range(w.N):
            t = torch.empty(plan.S, dtype=torch.int16, device=dev)
            device.fill_bf16(t, w.ag_key(r), gen.UNIFORM)
            shards.append(t)
        params = [torch.empty(w.N * plan.e[p], dtype=torch.int16, device=dev) for p in range(w.P)]
        sp, pp = tide.pointer_array(shards), tide.pointer_array(params)
        src = torch.empty(w.N * plan.S, dtype=torch.int16, device=dev)
        dst = torch.empty_like(src)
        for _ in range(max(1, args.warmup)):
            plan.ag_place(sp, pp, 2, stream)
            dst.copy_(src)
        nbytes = 4 * w.N * plan.S
        ag = median_ms(lambda: plan.ag_place(sp, pp, 2, stream))
        cp = median_ms(lambda: dst.copy_(src))
        plan.check()
        out[name] = {"bytes_read_plus_written": nbytes, "ag_ms": round(ag, 4), "copy_ms": round(cp, 4),
                     "ag_frac": round(nbytes / ag / 1e6 / peak, 4), "copy_frac": round(nbytes / cp / 1e6 / peak, 4),
                     "ag_over_copy": round(cp / ag, 4)}
        plan.close()
        del shards, params, src, dst
        torch.cuda.empty_cache()
    return {"path": "ag-ceiling", "metric": "all-gather and same-size copy, fraction of measured copy bandwidth",
            "unit": "fraction", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "data": "synthetic",
            "value": out[groups[0]]["ag_over_copy"], "groups": out}


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.path == "staged-rs":
        line = run_staged_rs(args, local_rank) if rank == 0 else None
    elif args.path == "rd-ag":
        line = run_rd_ag(args, local_rank) if rank == 0 else None
    elif args.path == "variants":
        line = run_variants(args, local_rank) if rank == 0 else None
    elif args.path == "ag-ceiling":
        line = run_ag_ceiling(args, local_rank) if rank == 0 else None
    else:
        line = run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

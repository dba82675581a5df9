"""bench.py host logic without a GPU: the reference (oracle) arm, the byte
accounting, and the multi-rank aggregation over gloo with world_size 2."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle.tide_oracle as O  # noqa: E402
from synth import configs  # noqa: E402


def test_algorithmic_bytes_match_closed_form():
    w = configs.get(2)
    geo = O.geometry(w.shapes, w.N)
    nb = bench.algorithmic_bytes(w, geo)
    assert nb["rs_bytes"] == 2 * 8 * 855_654_400 + 4 * 8 * 106_956_800
    assert nb["ag_bytes"] == 4 * 8 * 106_956_800
    w = configs.get(4)
    geo = O.geometry(w.shapes, w.N)
    assert bench.algorithmic_bytes(w, geo)["rs_bytes"] == 2 * 64 * 351_288_320 + 4 * 64 * 5_488_880


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1", "--workload", "tiny"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    secs = [1.5, 2.5][rank]
    units = [10.0, 30.0][rank]
    agreed = (bench.all_ranks_ok(True, world, "cpu"), bench.all_ranks_ok(rank == 0, world, "cpu"))
    q.put((rank, (bench.aggregate(secs, units, world), agreed)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_aggregate_and_agreement_over_gloo():
    """Max time and summed units over the ranks; and a yes/no that holds only
    if every rank says yes (the e2e leg runs on all ranks or on none)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == ((2.5, 40.0), (True, False))


def test_reference_arm_only_rank0_prints(monkeypatch):
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "tiny"])
    assert bench.run_reference(args, rank=1, world=2) is None
    rec = bench.run_reference(args, rank=0, world=2)
    assert rec["n_gpus"] == 2 and rec["impl"] == "reference"


def test_per_config_groups_selection():
    pick = lambda *argv: bench.per_config_groups(bench.parse_args(list(argv)))
    assert pick() == ["llama70b", "qwen3moe", "uneven"]                      # headline wan22dit
    assert pick("--workload", "uneven") == ["wan22dit", "llama70b", "qwen3moe"]
    assert pick("--workload", "tiny") == []                                   # not a measured group
    assert pick("--nodes", "16") == []                                        # a regrouped headline
    assert pick("--per-config", "none") == []
    assert pick("--per-config", "uneven, llama70b") == ["uneven", "llama70b"]
    with pytest.raises(SystemExit):
        pick("--per-config", "llama70b,nosuchgroup")


def test_rank_bytes_sum_to_the_algorithmic_bytes():
    for name in ("tiny", "uneven"):
        w, _ = bench.oracle_sample(name)
        geo = O.geometry(w.shapes, w.N)
        nb = bench.algorithmic_bytes(w, geo)
        assert bench.rank_bytes(w, geo, range(w.N)) == nb["rs_bytes"] + nb["ag_bytes"]
        half = list(range(0, w.N, 2))
        rest = list(range(1, w.N, 2))
        assert bench.rank_bytes(w, geo, half) + bench.rank_bytes(w, geo, rest) == nb["rs_bytes"] + nb["ag_bytes"]


def test_profiled_traffic_scales_reads_and_adds_algorithmic_writes(tmp_path, monkeypatch):
    """Reads of the captured launch scale by the ratio of contributor bytes;
    writes are the full launch's algorithmic writes; a summary taken on other
    kernel source gives None."""
    (tmp_path / "profiles").mkdir()
    (tmp_path / "fsdp_layout_aware_gb300" / "csrc").mkdir(parents=True)
    src = tmp_path / "fsdp_layout_aware_gb300" / "csrc" / "k.cu"
    src.write_bytes(b"kernel source")
    import hashlib
    digest = hashlib.sha256(b"kernel source").hexdigest()
    (tmp_path / "profiles" / "p.txt").write_text(
        f"workload_captured: g rows/4\nkernel_source_sha256: {digest}\n"
        "algorithmic_read_bytes_captured: 1000\nalgorithmic_write_bytes_captured: 100\n"
        "dram_bytes_read: 1010\ndram_bytes_write: 90\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    t = bench.profiled_traffic("p.txt", "k.cu", 4000, 400)
    assert t["bytes"] == 1010 * 4 + 400
    assert t["captured_dram_read_over_algorithmic"] == 1.01 and t["captured_dram_write_over_algorithmic"] == 0.9
    assert "g rows/4" in t["source"] and "x 4" in t["source"]
    src.write_bytes(b"changed source")
    assert bench.profiled_traffic("p.txt", "k.cu", 4000, 400) is None
    assert bench.profiled_traffic("missing.txt", "k.cu", 4000, 400) is None


def test_committed_headline_traffic_covers_the_algorithmic_bytes():
    """The committed rs_fused summaries give a full-launch traffic at least the
    algorithmic bytes (nothing is read less than once) for every measured group
    whose summary matches the current kernel source."""
    for name in ("wan22dit", "llama70b", "qwen3moe", "uneven"):
        w = configs.get(name)
        geo = O.geometry(w.shapes, w.N)
        nb = bench.algorithmic_bytes(w, geo)
        t = bench.profiled_traffic(f"rs_fused_{name}.txt", "rs_kernel.cu", 2 * nb["rs_elems"], 4 * w.N * geo.S)
        if t is None:
            pytest.skip(f"profiles/rs_fused_{name}.txt was taken on other kernel source (bench reports null)")
        assert nb["rs_bytes"] <= t["bytes"] <= 1.01 * nb["rs_bytes"], name

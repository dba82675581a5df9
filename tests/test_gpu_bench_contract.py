"""bench.py on the GPU at small sizes: every path exits 0 and prints one JSON
line, and the default line carries every key of the measurement contract
(roofline, CPU baseline, end-to-end, clocks, launch count)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMALL = ["--workload", "llama70b", "--row-div", "64"]


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_default_line_has_every_contract_key():
    K, W = 3, 3
    rec = _run(*SMALL, "--steps", str(K), "--warmup", str(W), "--cpu-seconds", "1", "--e2e-steps", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
                "gpu_launches"):
        assert key in rec, key
    assert rec["n_gpus"] == 1 and rec["steps"] == K and rec["warmup"] == W and rec["value"] > 0
    assert rec["higher_is_better"] is True and rec["scaling"] == "weak" and rec["vs_baseline"] is None
    assert "workload" in rec["config"]
    assert rec["config"]["l2"].startswith("L2 flushed")   # llama70b rows/64 moves 320 MB per step
    roof = rec["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-3)
    assert roof["frac_of_nominal"] == pytest.approx(roof["achieved"] / roof["nominal_peak"], rel=1e-3)
    for call in ("rs", "ag"):
        assert rec[call]["ms_median"] > 0 and rec[call]["ms"] > 0 and rec[call]["ms_uploading_pointer_table"] > 0
    cpu = rec["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0 and cpu["sample"]
    e2e = rec["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(rec["clocks"] or {})
    assert rec["gpu_launches"] == 2 * K   # one reduce-scatter and one all-gather kernel per step
    mt = rec["cpu_baseline_all_cores"]
    assert mt["cores"] >= 1 and mt["value"] > 0 and mt["sample"]
    # the other three measured groups, at the same row divisor, each with its own calls' figures
    assert set(rec["per_config"]) == {"wan22dit", "qwen3moe", "uneven"}
    for name, g in rec["per_config"].items():
        assert g["gpu_launches"] == 2 * K and g["GB_s"] > 0, name
        for call in ("rs", "ag"):
            assert g[call]["frac"] == pytest.approx(g[call]["GB_s"] / roof["peak"], rel=1e-3), (name, call)
        assert g["rs"]["GB_s"] == pytest.approx(g["rs_bytes_per_step"] / g["rs"]["ms"] / 1e6, rel=1e-3)


@pytest.mark.parametrize("path", ["staged-rs", "rd-ag", "variants", "ag-ceiling"])
def test_other_paths_print_one_line(path):
    rec = _run("--path", path, *SMALL, "--steps", "2", "--warmup", "1")
    assert rec["path"] == path and rec["value"] > 0


def test_path_options_select_what_is_timed():
    rec = _run("--path", "variants", "--variants", "rs_bulk,ag_sm", *SMALL, "--steps", "2", "--warmup", "1")
    assert set(rec["variants"]) == {"rs_bulk", "ag_sm"}
    rec = _run("--path", "staged-rs", "--staged-budget", "pages", "--inbox-offset", "1", *SMALL, "--steps", "2",
               "--warmup", "1")
    assert "pages_16_4" in rec and "fill" not in rec and rec["config"]["inbox_offset_floats"] == 1
    rec = _run("--path", "rd-ag", "--rd-exchange", "sm", "--rd-mode", "rails", *SMALL, "--steps", "2", "--warmup", "1")
    assert set(rec["exchange_all_rails"]) == {"sm_kernel"} and rec["exchange"] == {}
    rec = _run("--path", "ag-ceiling", "--per-config", "none", *SMALL, "--steps", "3", "--warmup", "1")
    g = rec["groups"]["llama70b"]
    assert set(rec["groups"]) == {"llama70b"} and g["ag_ms"] > 0 and g["copy_ms"] > 0

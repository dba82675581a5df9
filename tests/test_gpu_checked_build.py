"""The kernels store only inside their own work items.

Builds libtide_checked.so (every global store compared with the range of the
item it belongs to; a store outside is skipped and counted) and runs the
small-case GPU parity tests against it in a child process: they must pass
and the count must be zero.  With the plan's items checked on the host to
tile the caller's buffers exactly, this rules out stores outside the buffers
and stores into a neighbouring item that a later write would have hidden.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_kernels_store_only_inside_their_items(tmp_path):
    import importlib.util
    spec = importlib.util.spec_from_file_location("tide_build", os.path.join(ROOT, "fsdp_layout_aware_gb300",
                                                                               "build.py"))
    build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build)
    build.build_lib("tide_checked")
    report = tmp_path / "bounds.txt"
    env = dict(os.environ, TIDE_LIBRARY="checked", TIDE_BOUNDS_REPORT=str(report))
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_parity.py", "tests/test_gpu_many_nodes.py", "tests/test_gpu_fuzz.py",
           "tests/test_gpu_graphs.py", "tests/test_gpu_table_reuse.py",
           "-k", "not full_size"]
    proc = subprocess.run(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True,
                          timeout=1800)
    assert proc.returncode == 0, proc.stdout[-4000:]
    assert report.read_text().strip() == "0", "kernels stored outside their items: " + report.read_text()
    # positive control: the check does count (one made-up address, no memory access)
    probe = ("import fsdp_layout_aware_gb300 as t\n"
             "t.tide_debug_bounds_violations(True)\n"
             "t.tide_debug_bounds_selftest()\n"
             "print(t.tide_debug_bounds_violations(True))\n")
    out = subprocess.run([sys.executable, "-c", probe], cwd=ROOT, env=env, stdout=subprocess.PIPE,
                         stderr=subprocess.STDOUT, text=True, timeout=600)
    assert out.returncode == 0 and out.stdout.strip().splitlines()[-1] == "1", out.stdout

"""The boundary is a C ABI: a plain C99 program, compiled against
include/tide.h alone and linked with libtide.so, creates a plan, queries it,
gets error statuses and destroys it (no GPU call)."""

import os
import shutil
import subprocess

import pytest

import fsdp_layout_aware_gb300 as tide

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_library_is_usable_from_c(tmp_path):
    exe = tmp_path / "abi_from_c"
    libdir = os.path.dirname(tide.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_from_c.c"),
                    "-L", libdir, "-l:" + os.path.basename(tide.LIB_PATH), "-Wl,-rpath," + libdir,
                    "-o", str(exe)], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr

"""In-tree build of the CUDA libraries for sm_103a (GB300).

``build_all()`` compiles, with nvcc and in parallel:
  * ``fsdp_layout_aware_gb300/libtide.so``  -- the C-ABI library (include/tide.h)
  * ``synth/libtide_synth.so``              -- the seeded input generator's
                                               device twin (tests and bench only)
and, on request (``build_lib("tide_checked")``, ``--checked``):
  * ``fsdp_layout_aware_gb300/libtide_checked.so`` -- the same library compiled
                                               with TIDE_CHECKED: every kernel
                                               store checked against its work
                                               item (check.cuh; tests only)
A library is rebuilt only when its sources, headers or flags changed (a
content hash is kept next to the objects in ``_build/``).
"""

import concurrent.futures
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libtide")
    return cand


def _cuda_lib_dir(nvcc):
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]

TIDE_SRCS = [os.path.join(HERE, "csrc", f) for f in ("plan.cpp", "runtime.cu", "rs_kernel.cu", "rs_bulk.cu",
                                                     "rs_staged.cu", "ag_kernel.cu", "ag_bulk.cu", "rs_noalloc.cu")]
TIDE_DEPS = [os.path.join(HERE, "csrc", f) for f in ("tide_internal.h", "rs_device.cuh", "bulk_ptx.cuh",
                                                     "check.cuh")] + [os.path.join(ROOT, "include", "tide.h")]

LIBS = {
    "tide": {
        "out": os.path.join(HERE, "libtide.so"),
        "srcs": TIDE_SRCS,
        "deps": TIDE_DEPS,
        "build": os.path.join(HERE, "_build"),
    },
    "tide_checked": {
        "out": os.path.join(HERE, "libtide_checked.so"),
        "srcs": TIDE_SRCS,
        "deps": TIDE_DEPS,
        "build": os.path.join(HERE, "_build_checked"),
        "flags": ["-DTIDE_CHECKED"],
        "on_request": True,
    },
    "synth": {
        "out": os.path.join(ROOT, "synth", "libtide_synth.so"),
        "srcs": [os.path.join(ROOT, "synth", "csrc", "synth_gen.cu")],
        "deps": [],
        "build": os.path.join(ROOT, "synth", "_build"),
    },
}


def _digest(spec, flags):
    h = hashlib.sha256(" ".join(flags).encode())
    for path in spec["srcs"] + spec["deps"]:
        with open(path, "rb") as f:
            h.update(path.encode() + b"\0" + f.read())
    return h.hexdigest()


def _run(cmd):
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if proc.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + proc.stdout)
    return proc.stdout


def build_lib(name, force=False, verbose=False, extra_flags=()):
    spec = LIBS[name]
    nvcc = _nvcc()
    flags = ARCH + CFLAGS + spec.get("flags", []) + list(extra_flags)
    os.makedirs(spec["build"], exist_ok=True)
    stamp = os.path.join(spec["build"], "stamp")
    digest = _digest(spec, flags)
    if not force and os.path.exists(spec["out"]) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return spec["out"]
    objs = [os.path.join(spec["build"], os.path.basename(s) + ".o") for s in spec["srcs"]]
    cmds = [[nvcc] + flags + ["-c", s, "-o", o] for s, o in zip(spec["srcs"], objs)]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(cmds)) as pool:
        outs = list(pool.map(_run, cmds))
    if verbose:
        for o in outs:
            if o.strip():
                print(o)
    tmp = spec["out"] + ".tmp"
    _run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs +
         ["-Xlinker", "-rpath=" + _cuda_lib_dir(nvcc)])
    os.replace(tmp, spec["out"])
    with open(stamp, "w") as f:
        f.write(digest)
    return spec["out"]


def build_all(force=False, verbose=False, checked=False):
    """The libraries the package needs; the checked variant only if asked."""
    return [build_lib(n, force=force, verbose=verbose) for n, spec in LIBS.items()
            if checked or not spec.get("on_request")]


if __name__ == "__main__":
    import sys
    for path in build_all(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv):
        print(path)

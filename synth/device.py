"""Device-side fill of seeded bf16 inputs (``libtide_synth.so``).

Produces, on the GPU, exactly the bits ``synth.gen.bf16_values`` produces on
the host, so multi-gigabyte gradient groups can be generated in HBM while the
oracle regenerates any sampled element on the CPU.
"""

import ctypes
import os

import numpy as np

from . import gen

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtide_synth.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; run the build first")
        lib = ctypes.CDLL(LIB_PATH)
        lib.synth_fill_bf16.restype = ctypes.c_int
        lib.synth_fill_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32,
                                        ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p]
        _lib = lib
    return _lib


def fill_bf16(tensor, key, dist, sigma=1e-3, idx0=0, stream=None):
    """Fill a contiguous 2-byte CUDA tensor with stream ``key`` from index idx0."""
    import torch
    assert tensor.is_cuda and tensor.element_size() == 2 and tensor.is_contiguous()
    scale_bits = int(np.array([gen.normal_scale_f32(sigma)], dtype=np.float32).view(np.uint32)[0])
    s = (stream or torch.cuda.current_stream()).cuda_stream
    err = _load().synth_fill_bf16(tensor.data_ptr(), tensor.numel(), key & ((1 << 64) - 1), dist,
                                  scale_bits, idx0, s)
    if err != 0:
        raise RuntimeError(f"synth_fill_bf16 failed with CUDA error {err}")

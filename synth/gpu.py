"""ctypes binding of synth/libmhsynth.so: fills torch CUDA tensors with the
generator's draws (bit-identical to ``synth.normal``)."""
from __future__ import annotations

import ctypes
import os

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmhsynth.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: build it first")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.synth_normal_fill.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                          ctypes.c_float, ctypes.c_void_p]
        lib.synth_normal_fill.restype = ctypes.c_int
        _lib = lib
    return _lib


def fill_normal(t, seed: int, tensor_id: int, std=1.0, offset: int = 0, stream=None):
    """Overwrite contiguous CUDA tensor ``t`` (float32 or bfloat16) in place."""
    import torch
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("fill_normal needs a contiguous CUDA tensor")
    code = {torch.float32: 0, torch.bfloat16: 1}.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    s = torch.cuda.current_stream() if stream is None else stream
    err = _load().synth_normal_fill(t.data_ptr(), code, t.numel(), seed & ((1 << 64) - 1),
                                    tensor_id & ((1 << 64) - 1), offset, float(np.float32(std)),
                                    s.cuda_stream)
    if err != 0:
        raise RuntimeError(f"synth_normal_fill failed with cudaError {err}")
    return t

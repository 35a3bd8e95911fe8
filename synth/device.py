"""Device-side fill of synthetic values (the same generator as synth.values, in CUDA), for inputs
too large to generate on the host. Input generation only; shares nothing with librc."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

from . import TENSOR_K, TENSOR_Q, TENSOR_V, VALUE_SCALE

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "fill.cu")
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(src):
        return _LIB
    os.makedirs(_BUILD, exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                           "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", src, "-o", tmp])
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.synth_fill_rows.restype = ctypes.c_int
        L.synth_fill_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                      ctypes.c_void_p, ctypes.c_void_p]
        _lib = L
    return _lib


def fill_rows(hashes_dev, tensor: int, layer: int, dst, head0: int = 0, slots_dev=None,
              stream=None) -> None:
    """dst[i (or slots[i]), h, :] = values(hashes[i], tensor, layer, head0 + h) for all rows i.

    hashes_dev: int64 CUDA tensor (uint64 bits); dst: CUDA tensor [rows, H, D] (bf16 or fp32)."""
    import torch
    H, D = dst.shape[-2], dst.shape[-1]
    s = torch.cuda.current_stream() if stream is None else stream
    rc = lib().synth_fill_rows(
        ctypes.c_void_p(hashes_dev.data_ptr()),
        None if slots_dev is None else ctypes.c_void_p(slots_dev.data_ptr()),
        hashes_dev.numel(), tensor, layer, head0, H, D, int(dst.dtype == torch.bfloat16),
        float(VALUE_SCALE), ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_rows failed ({rc})")


def hashes_to_device(hashes: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(hashes, dtype=np.uint64).view(np.int64)).to(device)

"""GPU fill of the synthetic IQ4_NL expert tensors (``synth/synth_gen.cu``).

Input generation only: the same generator as ``synth/__init__.py``; a test
checks the two byte for byte."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gen.cu")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(_SRC)):
        return LIB_PATH
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", _SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {_SRC}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_fill_iq4nl.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                         ctypes.c_int64, ctypes.c_void_p]
        lib.synth_fill_iq4nl.restype = ctypes.c_int
        _lib = lib
    return _lib


def fill_iq4nl(dst, n_experts: int, blocks_per_expert: int, seed: int, layer: int, tensor: int,
               expert0: int = 0, stream=None):
    """Fill a uint8 CUDA tensor with n_experts * blocks_per_expert blocks."""
    import torch
    assert dst.dtype == torch.uint8 and dst.is_cuda and dst.is_contiguous()
    assert dst.numel() >= n_experts * blocks_per_expert * 18
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream.cuda_stream
    rc = _load().synth_fill_iq4nl(dst.data_ptr(), n_experts, blocks_per_expert, seed, layer,
                                  tensor, expert0, s)
    if rc != 0:
        raise RuntimeError(f"synth_fill_iq4nl failed ({rc})")
    return dst

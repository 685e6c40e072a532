"""ctypes binding for the plain C++ CPU oracle (``oracle/oracle.cpp``).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module. The CUDA library and its
Python binding never do.

The oracle computes the IQ4_NL routed-expert MoE layer with plain loops in
double precision (Red Lite, "What we learned", section 7: every native stage
has a double-precision CPU reference). See the header of ``oracle.cpp`` for the
source of each definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

EXACT = 0
MMA16 = 1
MMA8 = 2     # E4M3 operands with power-of-two row / vector exponents (oracle.cpp header)


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (OpenMP when available). Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
            _SRC, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c = ctypes
        P = c.c_void_p
        lib.orc_table.argtypes = [P]
        lib.orc_half_to_double.argtypes = [c.c_uint16]
        lib.orc_half_to_double.restype = c.c_double
        lib.orc_bf16_to_double.argtypes = [c.c_uint16]
        lib.orc_bf16_to_double.restype = c.c_double
        lib.orc_double_to_half.argtypes = [c.c_double]
        lib.orc_double_to_half.restype = c.c_uint16
        lib.orc_e4m3_to_double.argtypes = [c.c_uint8]
        lib.orc_e4m3_to_double.restype = c.c_double
        lib.orc_double_to_e4m3.argtypes = [c.c_double]
        lib.orc_double_to_e4m3.restype = c.c_uint8
        lib.orc_dequant_rows_e4m3.argtypes = [P, c.c_int64, c.c_int, P, P]
        lib.orc_dequant_blocks.argtypes = [P, c.c_int64, c.c_int, P]
        lib.orc_sanitize.argtypes = [P, P, c.c_int64, c.c_int, P, P]
        lib.orc_route.argtypes = [c.c_int, c.c_int, c.c_int, P, P, P, c.c_int, P, P, P, P]
        lib.orc_expert_ffn.argtypes = [c.c_int, c.c_int, P, P, P, P, c.c_int, P]
        lib.orc_moe_layer.argtypes = ([c.c_int] * 6 + [P, P, P, P, P, P, P, c.c_int, P, P,
                                                        c.c_int, c.c_int, P])
        lib.orc_max_threads.restype = c.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def table() -> np.ndarray:
    out = np.zeros(16, np.int32)
    _load().orc_table(_ptr(out))
    return out


def half_to_double(bits: int) -> float:
    return _load().orc_half_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits))


def double_to_half(v: float) -> int:
    return int(_load().orc_double_to_half(float(v)))


def e4m3_to_double(code: int) -> float:
    return _load().orc_e4m3_to_double(int(code) & 0xFF)


def double_to_e4m3(v: float) -> int:
    return int(_load().orc_double_to_e4m3(float(v)))


def dequant_rows_e4m3(mat: np.ndarray, rows: int, K: int):
    """Mode-2 (mma8) weights of `rows` rows of a K-input IQ4_NL matrix: float64
    [rows][K] and each row's exponent E_m (int32 [rows])."""
    b = np.ascontiguousarray(mat, dtype=np.uint8).reshape(-1)
    assert b.size >= rows * (K // 32) * 18
    out = np.empty((rows, K), np.float64)
    ex = np.empty(rows, np.int32)
    rc = _load().orc_dequant_rows_e4m3(_ptr(b), int(rows), int(K), _ptr(out), _ptr(ex))
    assert rc == 0
    return out, ex


def max_threads() -> int:
    return int(_load().orc_max_threads())


def dequant(blocks: np.ndarray, mode: int = EXACT) -> np.ndarray:
    """blocks: uint8 array whose size is a multiple of 18. Returns float64 [n*32]."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    assert b.size % 18 == 0
    n = b.size // 18
    out = np.empty(n * 32, np.float64)
    rc = _load().orc_dequant_blocks(_ptr(b), n, int(mode), _ptr(out))
    assert rc == 0
    return out


def sanitize(ids: np.ndarray, w: np.ndarray, n_experts: int):
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    io = np.empty_like(ids)
    wo = np.empty_like(w)
    bad = _load().orc_sanitize(_ptr(ids), _ptr(w), ids.size, int(n_experts), _ptr(io), _ptr(wo))
    return io, wo, int(bad)


def route(router_w: np.ndarray, bias: np.ndarray | None, x: np.ndarray, k: int):
    """router_w: uint16 (bf16 bits) [E, H]; bias: float32 [E] or None;
    x: uint16 (bf16 bits) [T, H]. Returns ids int32 [T,k], w float64 [T,k],
    gap float64 [T], scores float64 [T,E]."""
    Wr = np.ascontiguousarray(router_w, np.uint16)
    E, H = Wr.shape
    xx = np.ascontiguousarray(x, np.uint16).reshape(-1, H)
    T = xx.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, np.float32)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    gap = np.empty(T, np.float64)
    scores = np.empty((T, E), np.float64)
    rc = _load().orc_route(H, E, k, _ptr(Wr), _ptr(b), _ptr(xx), T, _ptr(ids), _ptr(w),
                           _ptr(gap), _ptr(scores))
    assert rc == 0, rc
    return ids, w, gap, scores


def expert_ffn(gate: np.ndarray, up: np.ndarray, down: np.ndarray, x_row: np.ndarray,
               H: int, F: int, mode: int = EXACT) -> np.ndarray:
    """One expert on one bf16 row; gate/up/down are this expert's blocks."""
    g = np.ascontiguousarray(gate, np.uint8)
    u = np.ascontiguousarray(up, np.uint8)
    d = np.ascontiguousarray(down, np.uint8)
    xr = np.ascontiguousarray(x_row, np.uint16).reshape(-1)
    assert xr.size == H
    out = np.empty(H, np.float64)
    rc = _load().orc_expert_ffn(H, F, _ptr(g), _ptr(u), _ptr(d), _ptr(xr), int(mode), _ptr(out))
    assert rc == 0, rc
    return out


def moe_layer(H: int, F: int, Fs: int, E: int, k: int, n_shared: int,
              experts: dict, shared, x: np.ndarray, ids: np.ndarray, w: np.ndarray,
              mode: int = EXACT, threads: int = 1) -> np.ndarray:
    """The whole layer. ``experts`` maps expert id -> (gate, up, down) uint8
    arrays of that expert's blocks (only the experts the routes use are needed).
    ``shared`` is (gate, up, down) or None. Returns y float64 [T, H]."""
    xx = np.ascontiguousarray(x, np.uint16).reshape(-1, H)
    T = xx.shape[0]
    ids = np.ascontiguousarray(ids, np.int32).reshape(T, k)
    w = np.ascontiguousarray(w, np.float64).reshape(T, k)
    keep = []
    ptrs = [(ctypes.c_void_p * E)() for _ in range(3)]
    for e, mats in experts.items():
        for m in range(3):
            a = np.ascontiguousarray(mats[m], np.uint8)
            keep.append(a)
            ptrs[m][int(e)] = a.ctypes.data
    if n_shared:
        sh = [np.ascontiguousarray(m, np.uint8) for m in shared]
        keep.extend(sh)
        shp = [_ptr(m) for m in sh]
    else:
        shp = [None, None, None]
    y = np.empty((T, H), np.float64)
    rc = _load().orc_moe_layer(H, F, Fs, E, k, n_shared, ptrs[0], ptrs[1], ptrs[2],
                               shp[0], shp[1], shp[2], _ptr(xx), T, _ptr(ids), _ptr(w),
                               int(mode), int(threads), _ptr(y))
    assert rc == 0, f"orc_moe_layer returned {rc}"
    del keep
    return y

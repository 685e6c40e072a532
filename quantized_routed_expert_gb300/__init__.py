"""Python binding of libmoe: the IQ4_NL routed-expert MoE layer on one GB300.

Argument marshalling only. Every step of the layer runs in libmoe's CUDA
kernels (``csrc/``), reached through the C ABI of ``include/moe.h``; PyTorch
provides device memory and streams. There is no CPU fallback: importing this
package fails if ``_build/libmoe.so`` has not been built, and every call
raises ``MoeError`` on a non-zero status.

Functions keep the C names without the ``moe_`` prefix: ``route_topk``,
``workspace_bytes``, ``iq4nl_decode``, ``iq4nl_prefill_grouped``,
``iq4nl_dequantize``, ``sanitize_routes``, ``set_pdl``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_LIBRARY may name another build of libmoe (the phase-stamp profiling
# build, _build_profile/libmoe.so); there is no other implementation.
LIB_PATH = os.environ.get("MOE_LIBRARY") or os.path.join(_HERE, "_build", "libmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libmoe is not built ({LIB_PATH} missing); run "
        "`python -c 'import __graft_entry__ as g; g.build()'` or "
        "`python quantized_routed_expert_gb300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_MISALIGNED = -4
MOE_ERR_CUDA = -5
STATUS_INVALID_ROUTE_MASK = 0x0000FFFF
STATUS_TIMEOUT = 0x80000000
MAX_DECODE_TOKENS = 16
STATIC_SCRATCH_BYTES = 8 << 20
DECODE, PREFILL, PREFILL_FP8 = 0, 1, 2
DEQUANT_FP32, DEQUANT_FP16, DEQUANT_FP32_ONE_TOKEN = 0, 1, 2


class Shape(ctypes.Structure):
    """moe_shape: hidden, ffn, ffn_shared, n_experts, top_k, n_shared."""
    _fields_ = [("hidden", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("ffn_shared", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")]


class _LayerWeights(ctypes.Structure):
    _fields_ = [("experts", _Weights), ("router_w", ctypes.c_void_p),
                ("router_bias", ctypes.c_void_p)]


_P = ctypes.c_void_p
_lib.moe_route_topk.argtypes = [ctypes.POINTER(Shape), _P, _P, _P, ctypes.c_int32, _P, _P, _P]
_lib.moe_route_topk.restype = ctypes.c_int
_lib.moe_workspace_bytes.argtypes = [ctypes.POINTER(Shape), ctypes.c_int32, ctypes.c_int32]
_lib.moe_workspace_bytes.restype = ctypes.c_size_t
for _fn in (_lib.moe_iq4nl_decode, _lib.moe_iq4nl_prefill_grouped):
    _fn.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(_Weights), _P, ctypes.c_int32, _P, _P,
                    _P, _P, ctypes.c_size_t, _P, _P]
    _fn.restype = ctypes.c_int
_lib.moe_iq4nl_decode_routed.argtypes = [ctypes.POINTER(Shape), _P, _P, ctypes.POINTER(_Weights),
                                         _P, ctypes.c_int32, _P, _P, _P, _P, ctypes.c_size_t, _P,
                                         _P]
_lib.moe_iq4nl_decode_routed.restype = ctypes.c_int
_lib.moe_iq4nl_decode_layers.argtypes = [ctypes.POINTER(Shape), ctypes.c_int32,
                                         ctypes.POINTER(_LayerWeights), _P, ctypes.c_int32,
                                         ctypes.c_int32, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
_lib.moe_iq4nl_decode_layers.restype = ctypes.c_int
_lib.moe_iq4nl_decode_static.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(_Weights), _P,
                                         ctypes.c_int32, _P, _P, _P, _P, _P]
_lib.moe_iq4nl_decode_static.restype = ctypes.c_int
_lib.moe_iq4nl_prefill_grouped_fp8.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(_Weights),
                                               _P, _P, ctypes.c_int32, _P, _P, _P, _P,
                                               ctypes.c_size_t, _P, _P]
_lib.moe_iq4nl_prefill_grouped_fp8.restype = ctypes.c_int
_lib.moe_fp8_row_exponent_count.argtypes = [ctypes.POINTER(Shape)]
_lib.moe_fp8_row_exponent_count.restype = ctypes.c_int64
_lib.moe_iq4nl_fp8_row_exponents.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(_Weights), _P,
                                             _P]
_lib.moe_iq4nl_fp8_row_exponents.restype = ctypes.c_int
_lib.moe_iq4nl_dequantize_e4m3.argtypes = [_P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P]
_lib.moe_iq4nl_dequantize_e4m3.restype = ctypes.c_int
_lib.moe_iq4nl_dequantize.argtypes = [_P, ctypes.c_int64, ctypes.c_int32, _P, _P]
_lib.moe_iq4nl_dequantize.restype = ctypes.c_int
_lib.moe_sanitize_routes.argtypes = [_P, _P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P, _P]
_lib.moe_sanitize_routes.restype = ctypes.c_int
_lib.moe_launches_per_call.argtypes = [ctypes.POINTER(Shape), ctypes.c_int32, ctypes.c_int32]
_lib.moe_launches_per_call.restype = ctypes.c_int32
_lib.moe_set_pdl.argtypes = [ctypes.c_int32]
_lib.moe_set_pdl.restype = ctypes.c_int32
_lib.moe_set_barrier_wait_ns.argtypes = [ctypes.c_uint64]
_lib.moe_set_barrier_wait_ns.restype = ctypes.c_uint64
_lib.moe_status_string.argtypes = [ctypes.c_int32]
_lib.moe_status_string.restype = ctypes.c_char_p
_lib.moe_version.restype = ctypes.c_char_p

EXPORTS = ("moe_route_topk", "moe_workspace_bytes", "moe_iq4nl_decode", "moe_iq4nl_decode_routed",
           "moe_iq4nl_decode_layers",
           "moe_iq4nl_decode_static", "moe_iq4nl_prefill_grouped", "moe_iq4nl_prefill_grouped_fp8",
           "moe_fp8_row_exponent_count", "moe_iq4nl_fp8_row_exponents", "moe_iq4nl_dequantize_e4m3",
           "moe_iq4nl_dequantize", "moe_sanitize_routes",
           "moe_launches_per_call", "moe_set_pdl", "moe_set_barrier_wait_ns", "moe_status_string",
           "moe_version")


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib.moe_status_string(status).decode()} ({status})")


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def version() -> str:
    return _lib.moe_version().decode()


def status_string(status: int) -> str:
    return _lib.moe_status_string(int(status)).decode()


CALL_ROUTE, CALL_DECODE, CALL_DECODE_ROUTED, CALL_PREFILL = 0, 1, 2, 3
CALL_PREFILL_FP8 = 5
MAX_LAYERS = 128


def call_decode_layers(n_layers: int, chained: bool) -> int:
    """The `call` code of moe_iq4nl_decode_layers for launches_per_call."""
    return 4 + 2 * int(n_layers) + (1 if chained else 0)


def launches_per_call(shape: Shape, T: int, call: int) -> int:
    """Kernel launches one call makes (host query)."""
    n = int(_lib.moe_launches_per_call(ctypes.byref(shape), int(T), int(call)))
    if n < 0:
        raise MoeError(n, "moe_launches_per_call")
    return n


def set_pdl(enable: bool) -> bool:
    return bool(_lib.moe_set_pdl(1 if enable else 0))


def set_barrier_wait_ns(ns: int) -> int:
    """Limit of a CTA's waits on the other CTAs of its grid (grid barriers of
    the single-launch decode kernels), in ns; returns the previous limit."""
    return int(_lib.moe_set_barrier_wait_ns(int(ns)))


def make_shape(hidden, ffn, n_experts, top_k, ffn_shared=None, n_shared=1) -> Shape:
    return Shape(int(hidden), int(ffn), int(ffn if ffn_shared is None else ffn_shared),
                 int(n_experts), int(top_k), int(n_shared))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _meta(t, dtype, name, shape=None):
    """Type, dtype and shape (when given) of one tensor argument."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _on_cuda(t, name):
    """A contiguous CUDA tensor."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _dev(t, dtype, name, shape=None):
    """Check one tensor argument: type, dtype, shape (when given), then that it
    is a contiguous CUDA tensor."""
    return _on_cuda(_meta(t, dtype, name, shape), name)


def _same_device(*tensors):
    """All tensor arguments on one CUDA device, and that device current (the
    library launches on the current device)."""
    devs = {t.device for t in tensors if isinstance(t, torch.Tensor)}
    if len(devs) > 1:
        raise ValueError(f"arguments are on different devices: {sorted(map(str, devs))}")
    if devs:
        d = devs.pop()
        if d.type == "cuda" and d.index is not None and d.index != torch.cuda.current_device():
            raise ValueError(f"arguments are on {d}, but the current device is "
                             f"cuda:{torch.cuda.current_device()}")


def _status_arg(status):
    if status is None:
        return
    if not isinstance(status, torch.Tensor) or status.dtype not in (torch.int32, torch.uint32) \
            or status.numel() < 1:
        raise TypeError("status must be an int32 or uint32 tensor with at least one element")
    if not status.is_cuda:
        raise ValueError("status must be on a CUDA device")


def _block_bytes(rows: int, K: int) -> int:
    return rows * (K // 32) * 18


class ExpertWeights:
    """Device tensors (uint8, IQ4_NL blocks) of one layer; keeps them alive.
    Entries may also be raw device addresses (int), which are not checked."""

    def __init__(self, gate, up, down, sh_gate=None, sh_up=None, sh_down=None):
        self.tensors = (gate, up, down, sh_gate, sh_up, sh_down)
        self.c = _Weights(*[_ptr(t) for t in self.tensors])

    def check(self, shape: "Shape"):
        """Each weight tensor holds at least the bytes the shape reads."""
        H, F, E = shape.hidden, shape.ffn, shape.n_experts
        need = [E * _block_bytes(F, H), E * _block_bytes(F, H), E * _block_bytes(H, F)]
        if shape.n_shared:
            Fs = shape.ffn_shared
            need += [_block_bytes(Fs, H), _block_bytes(Fs, H), _block_bytes(H, Fs)]
        names = ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")
        for name, t, n in zip(names, self.tensors, need):
            if t is None:
                raise ValueError(f"expert weights: {name} is missing")
            if isinstance(t, torch.Tensor):
                nb = t.numel() * t.element_size()
                if nb < n:
                    raise ValueError(f"expert weights: {name} holds {nb} bytes, the shape "
                                     f"reads {n}")
        return [t for t in self.tensors if isinstance(t, torch.Tensor)]

    def check_device(self):
        names = ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")
        for name, t in zip(names, self.tensors):
            if isinstance(t, torch.Tensor):
                if not t.is_cuda:
                    raise ValueError(f"expert weights: {name} must be on a CUDA device")
                if not t.is_contiguous():
                    raise ValueError(f"expert weights: {name} must be contiguous")


def workspace_bytes(shape: Shape, max_tokens: int, mode: int = DECODE) -> int:
    return int(_lib.moe_workspace_bytes(ctypes.byref(shape), int(max_tokens), int(mode)))


def workspace(shape: Shape, max_tokens: int, mode: int = DECODE, device="cuda"):
    """A zero-filled workspace (uint8) of the size libmoe asks for."""
    n = workspace_bytes(shape, max_tokens, mode)
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def route_topk(shape: Shape, router_w, router_bias, x, ids=None, weights=None, stream=None):
    """router_w: bf16 [E,H]; router_bias: fp32 [E] or None; x: bf16 [T,H].
    Returns (ids int32 [T,k], weights fp32 [T,k])."""
    ok = _shape_ok(shape)
    E, H, k = shape.n_experts, shape.hidden, shape.top_k
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a [T, hidden] tensor")
    T = x.shape[0]
    _meta(router_w, torch.bfloat16, "router_w", (E, H) if ok else None)
    _meta(x, torch.bfloat16, "x", (T, H) if ok else None)
    if router_bias is not None:
        _meta(router_bias, torch.float32, "router_bias", (E,) if ok else None)
    for t, name, dt in ((ids, "ids", torch.int32), (weights, "weights", torch.float32)):
        if t is not None:
            _meta(t, dt, name, (T, k) if ok else None)
    _on_cuda(router_w, "router_w")
    _on_cuda(x, "x")
    if router_bias is not None:
        _on_cuda(router_bias, "router_bias")
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=x.device)
    _on_cuda(ids, "ids")
    _on_cuda(weights, "weights")
    _same_device(router_w, router_bias, x, ids, weights)
    _check(_lib.moe_route_topk(ctypes.byref(shape), _ptr(router_w), _ptr(router_bias), _ptr(x),
                               int(T), _ptr(ids), _ptr(weights), _stream(stream)),
           "moe_route_topk")
    return ids, weights


def _shape_ok(shape: Shape) -> bool:
    """The library's own shape rule (an invalid shape is left to the C call,
    which refuses it with its status code)."""
    return int(_lib.moe_workspace_bytes(ctypes.byref(shape), 1, DECODE)) > 0


def _layer_args(shape, w: ExpertWeights, x, ids, weights, y, status):
    """Shapes, dtypes and devices of a layer call's tensors; returns (T, y)."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a [T, hidden] tensor")
    T = x.shape[0]
    ok = _shape_ok(shape)
    H, k = shape.hidden, shape.top_k
    wts = w.check(shape) if ok else []
    _meta(x, torch.bfloat16, "x", (T, H) if ok else None)
    _meta(ids, torch.int32, "ids", (T, k) if ok else None)
    _meta(weights, torch.float32, "weights", (T, k) if ok else None)
    if y is not None:
        _meta(y, torch.float32, "y", (T, H) if ok else None)
    if status is not None and (not isinstance(status, torch.Tensor) or status.dtype not in (
            torch.int32, torch.uint32) or status.numel() < 1):
        raise TypeError("status must be an int32 or uint32 tensor with at least one element")
    for t, name in ((x, "x"), (ids, "ids"), (weights, "weights")):
        _on_cuda(t, name)
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _on_cuda(y, "y")
    _status_arg(status)
    if ok:
        w.check_device()
    _same_device(x, ids, weights, y, status, *wts)
    return T, y


def _layer(fn, name, shape, w: ExpertWeights, x, ids, weights, y, ws, status, stream):
    T, y = _layer_args(shape, w, x, ids, weights, y, status)
    if ws is not None:
        _dev(ws, torch.uint8, "ws")
        _same_device(x, ws)
    _check(fn(ctypes.byref(shape), ctypes.byref(w.c), _ptr(x), int(T), _ptr(ids),
              _ptr(weights), _ptr(y), _ptr(ws), int(ws.numel() if ws is not None else 0),
              _ptr(status), _stream(stream)), name)
    return y


def iq4nl_decode(shape: Shape, w: ExpertWeights, x, ids, weights, ws, y=None, status=None,
                 stream=None):
    """Decode 1..16 tokens: y fp32 [T,H]."""
    return _layer(_lib.moe_iq4nl_decode, "moe_iq4nl_decode", shape, w, x, ids, weights, y, ws,
                  status, stream)


def iq4nl_decode_static(shape: Shape, w: ExpertWeights, x, ids, weights, y=None, status=None,
                        stream=None):
    """Decode 1..16 tokens on the library's own fixed scratch (no workspace
    argument, nothing allocated by libmoe). For callers that cannot allocate
    device memory where they run the layer. One scratch per device: calls that
    may overlap on the GPU race, so keep them on one stream. The first call on
    a device sets the scratch up and should come before any stream capture.
    Pass ``y`` to keep this wrapper from allocating the output itself."""
    T, y = _layer_args(shape, w, x, ids, weights, y, status)
    _check(_lib.moe_iq4nl_decode_static(ctypes.byref(shape), ctypes.byref(w.c), _ptr(x), int(T),
                                        _ptr(ids), _ptr(weights), _ptr(y), _ptr(status),
                                        _stream(stream)), "moe_iq4nl_decode_static")
    return y


def iq4nl_decode_routed(shape: Shape, router_w, router_bias, w: ExpertWeights, x, ws, ids=None,
                        weights=None, y=None, status=None, stream=None):
    """Route and decode 1..16 tokens in one call. Returns (ids, weights, y)."""
    ok = _shape_ok(shape)
    E, H, k = shape.n_experts, shape.hidden, shape.top_k
    _meta(router_w, torch.bfloat16, "router_w", (E, H) if ok else None)
    if router_bias is not None:
        _meta(router_bias, torch.float32, "router_bias", (E,) if ok else None)
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a [T, hidden] tensor")
    T = x.shape[0]
    for t, name, dt in ((ids, "ids", torch.int32), (weights, "weights", torch.float32)):
        if t is not None:
            _meta(t, dt, name, (T, k) if ok else None)
    _on_cuda(router_w, "router_w")
    if router_bias is not None:
        _on_cuda(router_bias, "router_bias")
    _on_cuda(x, "x")
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=x.device)
    T, y = _layer_args(shape, w, x, ids, weights, y, status)
    if ws is not None:
        _dev(ws, torch.uint8, "ws")
    _same_device(router_w, router_bias, x, ws)
    _check(_lib.moe_iq4nl_decode_routed(ctypes.byref(shape), _ptr(router_w), _ptr(router_bias),
                                        ctypes.byref(w.c), _ptr(x), int(T), _ptr(ids),
                                        _ptr(weights), _ptr(y), _ptr(ws),
                                        int(ws.numel() if ws is not None else 0), _ptr(status),
                                        _stream(stream)), "moe_iq4nl_decode_routed")
    return ids, weights, y


def iq4nl_decode_layers(shape: Shape, layers, x, ws, chained: bool = False, ids=None,
                        weights=None, y=None, status=None, stream=None):
    """Route and decode several layers of one shape in one call.
    layers: a sequence of (ExpertWeights, router_w bf16 [E,H], router_bias fp32 [E] or None).
    x: bf16 [L,T,H] (each layer's input) or, with chained=True, [T,H] (the first
    layer's; layer l+1 then takes bf16(y_l)). Returns (ids [L,T,k], weights [L,T,k],
    y fp32 [L,T,H])."""
    L = len(layers)
    if L < 1 or L > MAX_LAYERS:
        raise ValueError(f"1..{MAX_LAYERS} layers, got {L}")
    ok = _shape_ok(shape)
    E, H, k = shape.n_experts, shape.hidden, shape.top_k
    if not isinstance(x, torch.Tensor):
        raise TypeError("x must be a torch tensor")
    if chained:
        if x.dim() != 2:
            raise ValueError("x must be [T, hidden] for a chained call")
        T = x.shape[0]
        _meta(x, torch.bfloat16, "x", (T, H) if ok else None)
    else:
        if x.dim() != 3 or x.shape[0] != L:
            raise ValueError(f"x must be [{L}, T, hidden] (one input per layer)")
        T = x.shape[1]
        _meta(x, torch.bfloat16, "x", (L, T, H) if ok else None)
    keep, arr = [], (_LayerWeights * L)()
    for i, (w, wr, b) in enumerate(layers):
        if ok:
            keep += w.check(shape)
        _meta(wr, torch.bfloat16, f"layers[{i}] router_w", (E, H) if ok else None)
        if b is not None:
            _meta(b, torch.float32, f"layers[{i}] router_bias", (E,) if ok else None)
        arr[i].experts = w.c
        arr[i].router_w = _ptr(wr)
        arr[i].router_bias = _ptr(b)
        keep += [wr] + ([b] if b is not None else [])
    for t, name, dt, shp in ((ids, "ids", torch.int32, (L, T, k)),
                             (weights, "weights", torch.float32, (L, T, k)),
                             (y, "y", torch.float32, (L, T, H))):
        if t is not None:
            _meta(t, dt, name, shp if ok else None)
    _on_cuda(x, "x")
    for w, _, _ in layers:
        if ok:
            w.check_device()
    for t in keep:
        _on_cuda(t, "layer weights")
    if ids is None:
        ids = torch.empty((L, T, k), dtype=torch.int32, device=x.device)
    if weights is None:
        weights = torch.empty((L, T, k), dtype=torch.float32, device=x.device)
    if y is None:
        y = torch.empty((L, T, H), dtype=torch.float32, device=x.device)
    for t, name in ((ids, "ids"), (weights, "weights"), (y, "y")):
        _on_cuda(t, name)
    _status_arg(status)
    if ws is not None:
        _dev(ws, torch.uint8, "ws")
    _same_device(x, ids, weights, y, status, ws, *keep)
    _check(_lib.moe_iq4nl_decode_layers(ctypes.byref(shape), L, arr, _ptr(x), int(T),
                                        1 if chained else 0, _ptr(ids), _ptr(weights), _ptr(y),
                                        _ptr(ws), int(ws.numel() if ws is not None else 0),
                                        _ptr(status), _stream(stream)),
           "moe_iq4nl_decode_layers")
    return ids, weights, y


def iq4nl_prefill_grouped(shape: Shape, w: ExpertWeights, x, ids, weights, ws, y=None,
                          status=None, stream=None):
    """Prefill a chunk of tokens: y fp32 [T,H]."""
    return _layer(_lib.moe_iq4nl_prefill_grouped, "moe_iq4nl_prefill_grouped", shape, w, x, ids,
                  weights, y, ws, status, stream)


def fp8_row_exponents(shape: Shape, w: ExpertWeights, out=None, stream=None):
    """The row-exponent table of the 8-bit prefill for these weights: int8 [n]
    (gate rows, up rows, down rows, then the shared expert's), made once per
    set of weights."""
    n = int(_lib.moe_fp8_row_exponent_count(ctypes.byref(shape)))
    if n <= 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_fp8_row_exponent_count")
    keep = w.check(shape)
    w.check_device()
    dev = keep[0].device
    if out is None:
        out = torch.empty(n, dtype=torch.int8, device=dev)
    _dev(out, torch.int8, "out", (n,))
    _same_device(out, *keep)
    _check(_lib.moe_iq4nl_fp8_row_exponents(ctypes.byref(shape), ctypes.byref(w.c), _ptr(out),
                                            _stream(stream)), "moe_iq4nl_fp8_row_exponents")
    return out


def iq4nl_prefill_grouped_fp8(shape: Shape, w: ExpertWeights, row_exp, x, ids, weights, ws,
                              y=None, status=None, stream=None):
    """Prefill a chunk of tokens with E4M3 operands: y fp32 [T,H]. row_exp from
    fp8_row_exponents(shape, w); ws from workspace(shape, T, PREFILL_FP8)."""
    n = int(_lib.moe_fp8_row_exponent_count(ctypes.byref(shape)))
    _meta(row_exp, torch.int8, "row_exp", (n,) if n > 0 else None)
    T, y = _layer_args(shape, w, x, ids, weights, y, status)
    _on_cuda(row_exp, "row_exp")
    if ws is not None:
        _dev(ws, torch.uint8, "ws")
    _same_device(x, row_exp, ws)
    _check(_lib.moe_iq4nl_prefill_grouped_fp8(
        ctypes.byref(shape), ctypes.byref(w.c), _ptr(row_exp), _ptr(x), int(T), _ptr(ids),
        _ptr(weights), _ptr(y), _ptr(ws), int(ws.numel() if ws is not None else 0),
        _ptr(status), _stream(stream)), "moe_iq4nl_prefill_grouped_fp8")
    return y


def iq4nl_dequantize_e4m3(mat, rows: int, K: int, stream=None):
    """mat: uint8 device tensor of rows x K/32 IQ4_NL blocks -> (row exponents
    int8 [rows], E4M3 codes uint8 [rows, K]) through the 8-bit prefill's decoder."""
    if not isinstance(mat, torch.Tensor) or K % 32 or mat.numel() != rows * (K // 32) * 18:
        raise ValueError("mat must hold rows x K/32 blocks of 18 bytes")
    _dev(mat, torch.uint8, "mat")
    row_exp = torch.empty(rows, dtype=torch.int8, device=mat.device)
    out = torch.empty((rows, K), dtype=torch.uint8, device=mat.device)
    _check(_lib.moe_iq4nl_dequantize_e4m3(_ptr(mat), int(rows), int(K), _ptr(row_exp), _ptr(out),
                                          _stream(stream)), "moe_iq4nl_dequantize_e4m3")
    return row_exp, out


def iq4nl_dequantize(blocks, fp16: bool = False, out=None, stream=None, mode=None):
    """blocks: uint8 device tensor of 18-byte blocks -> fp32 (exact) or fp16 [n*32].
    ``mode`` picks the decoder: DEQUANT_FP32 (the decode lookup for experts
    with several tokens; the default), DEQUANT_FP16 (the prefill decoder;
    also ``fp16=True``) or DEQUANT_FP32_ONE_TOKEN (the decode split table)."""
    if mode is None:
        mode = DEQUANT_FP16 if fp16 else DEQUANT_FP32
    if mode not in (DEQUANT_FP32, DEQUANT_FP16, DEQUANT_FP32_ONE_TOKEN):
        raise ValueError(f"unknown dequantisation mode {mode}")
    if not isinstance(blocks, torch.Tensor) or blocks.numel() % 18:
        raise ValueError("blocks must be a tensor of a whole number of 18-byte blocks")
    _dev(blocks, torch.uint8, "blocks")
    n = blocks.numel() // 18
    dt = torch.float16 if mode == DEQUANT_FP16 else torch.float32
    if out is None:
        out = torch.empty(n * 32, dtype=dt, device=blocks.device)
    _dev(out, dt, "out", (n * 32,))
    _same_device(blocks, out)
    _check(_lib.moe_iq4nl_dequantize(_ptr(blocks), n, int(mode), _ptr(out),
                                     _stream(stream)), "moe_iq4nl_dequantize")
    return out


def sanitize_routes(ids, weights, n_experts: int, ids_out=None, weights_out=None, status=None,
                    stream=None):
    _dev(ids, torch.int32, "ids")
    _dev(weights, torch.float32, "weights", tuple(ids.shape))
    ids_out = torch.empty_like(ids) if ids_out is None else ids_out
    weights_out = torch.empty_like(weights) if weights_out is None else weights_out
    _dev(ids_out, torch.int32, "ids_out", tuple(ids.shape))
    _dev(weights_out, torch.float32, "weights_out", tuple(ids.shape))
    _status_arg(status)
    _same_device(ids, weights, ids_out, weights_out, status)
    _check(_lib.moe_sanitize_routes(_ptr(ids), _ptr(weights), ids.numel(), int(n_experts),
                                    _ptr(ids_out), _ptr(weights_out), _ptr(status),
                                    _stream(stream)), "moe_sanitize_routes")
    return ids_out, weights_out

"""A shared expert whose width differs from the routed experts' (ffn_shared !=
ffn): every layer path against the oracle. The pages' models all give the
shared expert the routed width; the calls take any width their rules allow, so
the other case is checked here: the decode kernels (fused, for a few tokens,
and the two-kernel path), the fp16-operand prefill and the E4M3 prefill."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV, check_close, lib, moe_shape, oracle_layer, run_decode, weights_of

pytestmark = pytest.mark.gpu

# widths that every path takes (multiples of 256); the shared expert is 3x as wide
WIDE = synth.Shape("shared-wide", 512, 256, 16, 4, 64, 1, Fs=768, n_shared=1)
NARROW = synth.Shape("shared-narrow", 512, 768, 16, 4, 64, 1, Fs=256, n_shared=1)

_layers = {}


def layer_of(s):
    from synth.layers import Layer
    if s.name not in _layers:
        _layers[s.name] = Layer(s, 13, 0, device=DEV)
    return _layers[s.name]


def _inputs(s, T, seed):
    rng = np.random.default_rng(seed)
    x_host = synth.to_bf16_bits(rng.standard_normal((T, s.H)))
    ids = np.stack([rng.choice(s.E, s.k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, s.k)).astype(np.float32)
    return x_host, ids, w


@pytest.mark.parametrize("s", [WIDE, NARROW], ids=["wide", "narrow"])
@pytest.mark.parametrize("T", [3, 11])
def test_decode_shared_width(s, T):
    L = layer_of(s)
    x_host, ids, w = _inputs(s, T, T)
    _, _, y = run_decode(L, x_host, ids, w)
    check_close(y, oracle_layer(L, x_host, ids, w), f"decode {s.name} T={T}")


def _prefill(L, x_host, ids, w, fp8):
    moe = lib()
    from synth.layers import bf16_tensor
    s = L.shape
    shape = moe_shape(s)
    x = bf16_tensor(x_host, DEV)
    ids_t = torch.as_tensor(ids, device=DEV).contiguous()
    w_t = torch.as_tensor(w, device=DEV).contiguous()
    T = x_host.shape[0]
    wts = weights_of(L)
    if fp8:
        ws = moe.workspace(shape, T, moe.PREFILL_FP8, DEV)
        y = moe.iq4nl_prefill_grouped_fp8(shape, wts, moe.fp8_row_exponents(shape, wts), x,
                                          ids_t, w_t, ws)
    else:
        ws = moe.workspace(shape, T, moe.PREFILL, DEV)
        y = moe.iq4nl_prefill_grouped(shape, wts, x, ids_t, w_t, ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("s", [WIDE, NARROW], ids=["wide", "narrow"])
@pytest.mark.parametrize("fp8", [False, True], ids=["fp16", "e4m3"])
def test_prefill_shared_width(s, fp8):
    L = layer_of(s)
    T = 300
    x_host, ids, w = _inputs(s, T, 7)
    y = _prefill(L, x_host, ids, w, fp8)
    rows = np.sort(np.random.default_rng(3).choice(T, 40, replace=False))
    ref = oracle_layer(L, x_host[rows], ids[rows], w[rows], oracle.MMA8 if fp8 else oracle.MMA16)
    check_close(y[rows], ref, f"prefill {'e4m3' if fp8 else 'fp16'} {s.name}")

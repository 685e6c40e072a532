"""GPU test helpers: device layers, C-ABI calls and the matching oracle runs."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import synth
from _util import GAP_MIN, check_close

DEV = torch.device("cuda:0")
THREADS = max(1, min(os.cpu_count() or 1, 16))


def lib():
    import quantized_routed_expert_gb300 as moe
    return moe


def moe_shape(s: synth.Shape):
    moe = lib()
    return moe.make_shape(s.H, s.F, s.E, s.k, s.Fs, s.n_shared)


def weights_of(layer):
    moe = lib()
    return moe.ExpertWeights(layer.gate, layer.up, layer.down, layer.sh_gate, layer.sh_up,
                             layer.sh_down)


def gapped_rows(layer, T: int, input_set: int = 0, max_tries: int = 64) -> np.ndarray:
    """x rows (bf16 bits [T,H]) whose k-th key beats the (k+1)-th by > 1e-3."""
    s = layer.shape
    rows = []
    for t in range(T):
        for r in range(max_tries):
            xr = synth.x_row(layer.seed, layer.layer, s.H, t, input_set, r)
            _, _, gap, _ = oracle.route(layer.router_w_host, layer.bias_host, xr[None], s.k)
            if gap[0] > GAP_MIN:
                break
        else:
            raise RuntimeError("no gapped row")
        rows.append(xr)
    return np.stack(rows)


def oracle_layer(layer, x_host: np.ndarray, ids: np.ndarray, w: np.ndarray,
                 mode=oracle.EXACT) -> np.ndarray:
    s = layer.shape
    ids = np.asarray(ids, np.int32)
    used = sorted({int(e) for e in ids.reshape(-1) if 0 <= e < s.E} | {0})
    experts = {e: layer.expert_bytes_host(e) for e in used}
    sh = layer.shared_bytes_host() if s.n_shared else None
    return oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, s.n_shared, experts, sh, x_host, ids,
                            np.asarray(w, np.float64), mode=mode, threads=THREADS)


def check_route(ids_g: np.ndarray, w_g: np.ndarray, layer, x_host: np.ndarray):
    """Chosen expert sets bit-exact against the oracle; the order within a token
    valid (non-increasing oracle key, up to fp32 noise); weights within 1e-6."""
    ids_ref, w_ref, gap, scores = oracle.route(layer.router_w_host, layer.bias_host, x_host,
                                               layer.shape.k)
    assert np.all(gap > GAP_MIN)
    assert np.array_equal(np.sort(ids_g, 1), np.sort(ids_ref, 1)), (ids_g, ids_ref)
    p = 1.0 / (1.0 + np.exp(-scores))
    key = p + layer.bias_host.astype(np.float64)[None, :]
    kg = np.take_along_axis(key, ids_g.astype(np.int64), 1)
    assert np.all(np.diff(kg, axis=1) <= 1e-5), kg
    # weights: compare per expert id
    for t in range(ids_g.shape[0]):
        ref = dict(zip(ids_ref[t].tolist(), w_ref[t].tolist()))
        got = np.array([ref[int(e)] for e in ids_g[t]])
        assert np.allclose(w_g[t], got, rtol=2e-6, atol=1e-7), (w_g[t], got)
    assert np.all(np.abs(w_g.sum(1) - 1.0) <= 1e-6)


def run_decode(layer, x_host: np.ndarray, ids=None, w=None, ws=None, status=None):
    moe = lib()
    from synth.layers import bf16_tensor
    s = layer.shape
    shape = moe_shape(s)
    x = bf16_tensor(x_host, DEV)
    if ids is None:
        ids_t, w_t = moe.route_topk(shape, layer.router_w, layer.bias, x)
    else:
        ids_t = torch.as_tensor(np.asarray(ids, np.int32), device=DEV).contiguous()
        w_t = torch.as_tensor(np.asarray(w, np.float32), device=DEV).contiguous()
    T = x_host.shape[0]
    if ws is None:
        ws = moe.workspace(shape, T, moe.DECODE, DEV)
    y = moe.iq4nl_decode(shape, weights_of(layer), x, ids_t, w_t, ws, status=status)
    torch.cuda.synchronize()
    return ids_t.cpu().numpy(), w_t.cpu().numpy(), y.cpu().numpy()


__all__ = ["DEV", "lib", "moe_shape", "weights_of", "gapped_rows", "oracle_layer",
           "check_route", "run_decode", "check_close"]

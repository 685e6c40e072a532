"""Shared test helpers: golden-file readers, independent numpy references for
the oracle pins, routing-gap resampling, and the parity comparison."""
from __future__ import annotations

import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden(name: str) -> list[str]:
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


def golden_table() -> np.ndarray:
    return np.array([int(v) for v in read_golden("iq4nl_table.txt")[0].split()], np.int64)


def golden_kv(name: str) -> dict:
    out = {}
    for ln in read_golden(name):
        k, *v = ln.split()
        out[k] = v
    return out


# ---------------------------------------------------------------------------
# Independent numpy references (library conversions + BLAS), used to pin the
# oracle. They decode fp16 with numpy's float16 and use scipy's expit.

def np_dequant(blocks: np.ndarray) -> np.ndarray:
    """IQ4_NL blocks uint8 [n, 18] -> float64 [n, 32] via numpy's float16."""
    b = np.ascontiguousarray(blocks, np.uint8).reshape(-1, 18)
    table = golden_table().astype(np.float64)
    d = b[:, 0:2].copy().view("<f2").astype(np.float64).reshape(-1, 1)
    qs = b[:, 2:18]
    return np.concatenate([table[qs & 0x0F], table[qs >> 4]], axis=1) * d


def np_dense(blocks: np.ndarray, rows: int, K: int) -> np.ndarray:
    return np_dequant(blocks).reshape(rows, K)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def np_swiglu_expert(mats, H: int, F: int, x: np.ndarray, fp16: bool = False) -> np.ndarray:
    """Dense SwiGLU expert: x float64 [T, H] -> [T, H]. fp16=True rounds the
    dequantised weights, x and h to float16 with numpy (the mma16 reading)."""
    from scipy.special import expit
    Wg = np_dense(mats[0], F, H)
    Wu = np_dense(mats[1], F, H)
    Wd = np_dense(mats[2], H, F)
    if fp16:
        Wg, Wu, Wd = (m.astype(np.float16).astype(np.float64) for m in (Wg, Wu, Wd))
        x = x.astype(np.float16).astype(np.float64)
    g = x @ Wg.T
    u = x @ Wu.T
    h = g * expit(g) * u
    if fp16:
        h = h.astype(np.float16).astype(np.float64)
    return h @ Wd.T


def torch_e4m3(v: np.ndarray) -> np.ndarray:
    """Round values to E4M3 with PyTorch's float8_e4m3fn conversion (round to
    nearest even); the library routine the mma8 pins check against. Values must
    lie within +-464, where PyTorch and the saturating reading agree. PyTorch
    converts through float32, so a float64 input is rounded twice: exact for
    the pins' weights and activations (which are float32 values), and for h it
    differs only for a value within a float32 ulp of an E4M3 midpoint."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, np.float64))
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def np_row_exponents(blocks: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Largest fp16 scale exponent of each row (field - 15; -14 for field 0)."""
    b = np.ascontiguousarray(blocks, np.uint8).reshape(rows, K // 32, 18)
    f = ((b[:, :, 0].astype(np.int32) | (b[:, :, 1].astype(np.int32) << 8)) >> 10) & 0x1F
    return np.where(f == 0, -14, f - 15).max(axis=1)


def np_e4m3_rows(M: np.ndarray, E: np.ndarray) -> np.ndarray:
    """Rows of M rounded as 2^E e4m3(M 2^-E), E per row."""
    sc = np.ldexp(1.0, E.astype(np.int64))[:, None]
    return torch_e4m3(M / sc) * sc


def np_e4m3_vectors(V: np.ndarray) -> np.ndarray:
    """Each row v of V rounded as 2^X e4m3(v 2^-X), X = floor(log2 max|v|) - 6."""
    m = np.abs(V).max(axis=1)
    _, e = np.frexp(m)
    X = np.where(m > 0, e - 1 - 6, 0)
    return np_e4m3_rows(V, X)


def np_swiglu_expert_e4m3(mats, H: int, F: int, x: np.ndarray) -> np.ndarray:
    """Dense SwiGLU expert with the mma8 reading's roundings, from numpy
    (dequantisation, exponents, BLAS) and PyTorch (E4M3 rounding)."""
    from scipy.special import expit
    out = []
    for m, rows, K in ((mats[0], F, H), (mats[1], F, H), (mats[2], H, F)):
        out.append(np_e4m3_rows(np_dense(m, rows, K), np_row_exponents(m, rows, K)))
    Wg, Wu, Wd = out
    x8 = np_e4m3_vectors(x)
    g = x8 @ Wg.T
    u = x8 @ Wu.T
    h8 = np_e4m3_vectors(g * expit(g) * u)
    return h8 @ Wd.T


def np_route(Wr_bits: np.ndarray, bias, x_bits: np.ndarray, k: int):
    """Keys from numpy (row by row np.dot), selection by brute force over all
    k-subsets (only for small E)."""
    from itertools import combinations
    from scipy.special import expit
    Wr = bf16_to_f64(Wr_bits)
    X = bf16_to_f64(x_bits).reshape(-1, Wr.shape[1])
    E = Wr.shape[0]
    b = np.zeros(E) if bias is None else np.asarray(bias, np.float64)
    ids_all, w_all = [], []
    for x in X:
        s = np.array([np.dot(Wr[e], x) for e in range(E)])
        p = expit(s)
        key = p + b
        best = None
        for S in combinations(range(E), k):
            cand = sorted(((-key[e], e) for e in S))
            if best is None or cand < best:
                best = cand
        ids = [e for _, e in best]
        ids_all.append(ids)
        w_all.append(p[ids] / p[ids].sum())
    return np.array(ids_all, np.int32), np.array(w_all)


# ---------------------------------------------------------------------------
# Routing gap: inputs are resampled per token until the k-th key exceeds the
# (k+1)-th by more than 1e-3 (both sides then take the same top-k decision).

GAP_MIN = 1e-3


def gapped_x(shape, seed: int, layer: int, T: int, input_set: int = 0, max_tries: int = 64):
    import oracle
    import synth
    Wr, b = synth.router(shape, seed, layer)
    rows, rs = [], []
    for t in range(T):
        for r in range(max_tries):
            xr = synth.x_row(seed, layer, shape.H, t, input_set, r)
            _, _, gap, _ = oracle.route(Wr, b, xr.reshape(1, -1), shape.k)
            if gap[0] > GAP_MIN:
                break
        else:
            raise RuntimeError("no gapped row found")
        rows.append(xr)
        rs.append(r)
    return np.stack(rows), np.array(rs, np.int64)


# ---------------------------------------------------------------------------
# Parity bar for floating outputs: max|diff| <= 1e-3 * max|ref| and
# relative L2 <= 5e-4.

MAX_REL = 1e-3
L2_REL = 5e-4


def check_close(got: np.ndarray, ref: np.ndarray, what: str = "", max_rel=MAX_REL,
                l2_rel=L2_REL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert got.size > 0, f"{what}: empty output"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    scale = np.abs(ref).max()
    assert scale > 0, f"{what}: all-zero reference"
    diff = np.abs(got - ref)
    md = diff.max() / scale
    l2 = np.sqrt((diff ** 2).sum() / (ref ** 2).sum())
    assert md <= max_rel and l2 <= l2_rel, (
        f"{what}: max|diff|/max|ref| = {md:.3e} (bar {max_rel}), rel-L2 = {l2:.3e} (bar {l2_rel})")
    return md, l2

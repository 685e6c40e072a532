"""Parity of the 8-bit-operand prefill with the oracle's E4M3 mode (MMA8).

The call runs the prompt contraction on the 8-bit tensor cores: weights enter
as E4M3 codes of d*T[q] scaled by a power of two per weight row, x and h as
E4M3 codes of each row scaled by a power of two per token / per (token,
expert). The weight and x codes are a fixed function of the inputs, so the
decoder is checked bit for bit; h comes from fp32 accumulators on the GPU and
from exact arithmetic in the oracle, so a code of h whose value lies within
the accumulation error of a rounding midpoint can round the other way. Such a
flip moves one h by one E4M3 step (2^-3 of its binade) and y by that times one
column of the down matrix, far inside the layer's float bar over thousands of
terms; the bar is the same as for the other layer paths.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV, check_close, gapped_rows, lib, moe_shape, weights_of

pytestmark = pytest.mark.gpu

_layers = {}


def layer_of(cfg_or_shape, layer=0, seed=None):
    from synth.layers import Layer
    s = synth.SHAPES[cfg_or_shape] if isinstance(cfg_or_shape, int) else cfg_or_shape
    seed = synth.seed_of(cfg_or_shape) if seed is None else seed
    key = (s.name, s.H, s.F, s.E, s.k, s.n_shared, seed, layer)
    if key not in _layers:
        if len(_layers) > 3:
            _layers.clear()
            torch.cuda.empty_cache()
        _layers[key] = Layer(s, seed, layer, device=DEV)
    return _layers[key]


# a small layer the 8-bit path takes (reduction lengths multiples of 256)
SMALL = synth.Shape("pf8-small", 256, 256, 8, 2, 4, 1, n_shared=1)


def run_prefill_fp8(L, x_host, ids=None, w=None, status=None):
    moe = lib()
    from synth.layers import bf16_tensor
    s = L.shape
    shape = moe_shape(s)
    x = bf16_tensor(x_host, DEV)
    if ids is None:
        ids_t, w_t = moe.route_topk(shape, L.router_w, L.bias, x)
    else:
        ids_t = torch.as_tensor(np.asarray(ids, np.int32), device=DEV).contiguous()
        w_t = torch.as_tensor(np.asarray(w, np.float32), device=DEV).contiguous()
    T = x_host.shape[0]
    wts = weights_of(L)
    rexp = moe.fp8_row_exponents(shape, wts)
    ws = moe.workspace(shape, T, moe.PREFILL_FP8, DEV)
    y = moe.iq4nl_prefill_grouped_fp8(shape, wts, rexp, x, ids_t, w_t, ws, status=status)
    torch.cuda.synchronize()
    return ids_t.cpu().numpy(), w_t.cpu().numpy(), y.cpu().numpy()


def oracle_rows(L, x_host, ids, w, rows, mode=oracle.MMA8):
    s = L.shape
    ids = np.asarray(ids, np.int32)
    used = sorted({int(e) for e in ids[rows].reshape(-1) if 0 <= e < s.E} | {0})
    experts = {e: L.expert_bytes_host(e) for e in used}
    sh = L.shared_bytes_host() if s.n_shared else None
    return oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, s.n_shared, experts, sh, x_host[rows],
                            ids[rows], np.asarray(w, np.float64)[rows], mode=mode, threads=16)


def _e4m3_values():
    return np.array([oracle.e4m3_to_double(c) for c in range(256)], np.float64)


def _check_codes(mat_host, rows, K, what):
    """GPU E4M3 decoder of rows x K weights against the oracle's, bit for bit."""
    moe = lib()
    mat = torch.as_tensor(np.ascontiguousarray(mat_host, np.uint8).reshape(-1), device=DEV)
    rexp, codes = moe.iq4nl_dequantize_e4m3(mat, rows, K)
    torch.cuda.synchronize()
    rexp = rexp.cpu().numpy().astype(np.int32)
    codes = codes.cpu().numpy()
    want, want_e = oracle.dequant_rows_e4m3(mat_host, rows, K)
    assert np.array_equal(rexp, want_e), f"{what}: row exponents differ"
    got = _e4m3_values()[codes] * np.ldexp(1.0, rexp)[:, None]
    bad = np.argwhere((got != want) | (np.signbit(got) != np.signbit(want)))
    assert bad.size == 0, (f"{what}: {len(bad)} codes differ, first at {bad[0]}: "
                           f"code {codes[tuple(bad[0])]:#04x} -> {got[tuple(bad[0])]!r}, "
                           f"oracle {want[tuple(bad[0])]!r}")
    assert not np.any((codes & 0x7F) == 0x7F), f"{what}: NaN code"


def _blocks(rng, rows, K, dbits):
    """rows x K/32 IQ4_NL blocks with the given fp16 scale bits [rows, K/32]
    and random index nibbles."""
    nb = K // 32
    b = np.zeros((rows, nb, 18), np.uint8)
    d = np.asarray(dbits, np.uint16).reshape(rows, nb)
    b[:, :, 0] = d & 0xFF
    b[:, :, 1] = d >> 8
    b[:, :, 2:] = rng.integers(0, 256, (rows, nb, 16), dtype=np.uint8)
    return b.reshape(rows, nb * 18)


def test_e4m3_decoder_layer_weights():
    # every matrix of a synthetic layer, through the prefill's decoder
    L = layer_of(SMALL, 0, seed=3)
    s = L.shape
    g, u, d = L.expert_bytes_host(0)
    for name, m, rows, K in (("gate", g, s.F, s.H), ("up", u, s.F, s.H), ("down", d, s.H, s.F)):
        _check_codes(m, rows, K, f"expert 0 {name}")


def test_e4m3_decoder_extreme_scales():
    # rows whose block scales span the fp16 range: zero and negative zero,
    # subnormals, the largest finite, and rows mixing a large scale with small
    # ones (those blocks land on E4M3 subnormals or round to zero)
    rng = np.random.default_rng(7)
    K, rows = 256, 12
    special = [0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x0400, 0x7BFF, 0xFBFF, 0x3C00, 0xBC00,
               0x1234, 0x5678]
    dbits = np.empty((rows, K // 32), np.uint16)
    for r in range(rows):
        if r < 4:
            dbits[r] = rng.choice(special, K // 32)
        elif r < 8:
            dbits[r] = rng.integers(0x0001, 0x7BFF, K // 32) | (rng.integers(0, 2, K // 32) << 15)
            dbits[r, 0] = 0x7800 | rng.integers(0, 0x3FF)      # one large scale
        else:
            dbits[r] = rng.integers(0, 0x0400, K // 32)        # subnormal scales only
    dbits[11] = 0                                              # an all-zero row: E = -14
    _check_codes(_blocks(rng, rows, K, dbits), rows, K, "extreme scales")


def test_fp8_row_exponent_table():
    moe = lib()
    L = layer_of(SMALL, 0, seed=3)
    s = L.shape
    shape = moe_shape(s)
    n = moe._lib.moe_fp8_row_exponent_count(__import__("ctypes").byref(shape))
    assert n == 2 * s.E * s.F + s.E * s.H + 2 * s.Fs + s.H
    got = moe.fp8_row_exponents(shape, weights_of(L)).cpu().numpy().astype(np.int32)
    want = {"gate": [], "up": [], "down": []}
    for e in range(s.E):
        g, u, d = L.expert_bytes_host(e)
        want["gate"].append(oracle.dequant_rows_e4m3(g, s.F, s.H)[1])
        want["up"].append(oracle.dequant_rows_e4m3(u, s.F, s.H)[1])
        want["down"].append(oracle.dequant_rows_e4m3(d, s.H, s.F)[1])
    sg, su, sd = L.shared_bytes_host()
    ref = np.concatenate(want["gate"] + want["up"] + want["down"] +
                         [oracle.dequant_rows_e4m3(sg, s.Fs, s.H)[1],
                          oracle.dequant_rows_e4m3(su, s.Fs, s.H)[1],
                          oracle.dequant_rows_e4m3(sd, s.H, s.Fs)[1]])
    assert np.array_equal(got, ref)


def test_prefill_fp8_small_layer():
    L = layer_of(SMALL, 0, seed=3)
    s = L.shape
    rng = np.random.default_rng(5)
    T = 37
    x_host = synth.to_bf16_bits(rng.standard_normal((T, s.H)))
    x_host[3] = 0                                   # an all-zero token: X = 0
    x_host[4] = synth.to_bf16_bits(rng.standard_normal(s.H) * 1e-5)    # small values
    x_host[5] = synth.to_bf16_bits(rng.standard_normal(s.H) * 1e5)     # large values
    ids = np.stack([rng.choice(s.E, s.k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, s.k)).astype(np.float32)
    _, _, y = run_prefill_fp8(L, x_host, ids, w)
    rows = np.array([t for t in range(T) if t not in (4, 5)])
    check_close(y[rows], oracle_rows(L, x_host, ids, w, rows), "prefill fp8 small vs mma8")
    assert np.all(y[3] == 0)
    for t in (4, 5):                                # each token on its own scale
        check_close(y[[t]], oracle_rows(L, x_host, ids, w, np.array([t])), f"fp8 token {t}")
    md, l2 = check_close(y[rows], oracle_rows(L, x_host, ids, w, rows, oracle.EXACT),
                         "prefill fp8 small vs exact", max_rel=0.15, l2_rel=0.1)
    print(f"fp8 small vs exact: max {md:.3e}, rel-L2 {l2:.3e}")


def test_prefill_fp8_ragged_chunk_xing_shape():
    s = synth.SHAPES[4]
    L = layer_of(4, 0)
    rng = np.random.default_rng(11)
    T = 200
    x_host = synth.to_bf16_bits(rng.standard_normal((T, s.H)))
    ids, w, y = run_prefill_fp8(L, x_host)
    rows = np.arange(T)
    md, l2 = check_close(y, oracle_rows(L, x_host, ids, w, rows), "prefill fp8 T=200 vs mma8")
    print(f"fp8 T=200 vs mma8: max {md:.3e}, rel-L2 {l2:.3e}")


def test_prefill_fp8_full_chunk_sampled_tokens():
    s = synth.SHAPES[4]
    L = layer_of(4, 1)
    T = s.T
    x_host = synth.x_rows(L.seed, 1, s.H, T)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, w, y = run_prefill_fp8(L, x_host, status=status)
    assert int(status.item()) == 0
    rows = np.random.default_rng(0).choice(T, 12, replace=False)
    rows = np.sort(np.concatenate([rows, [0, T - 1]]))
    check_close(y[rows], oracle_rows(L, x_host, ids, w, rows), "prefill fp8 T=2048 sampled")
    md, l2 = check_close(y[rows], oracle_rows(L, x_host, ids, w, rows, oracle.EXACT),
                         "prefill fp8 T=2048 vs exact", max_rel=0.15, l2_rel=0.1)
    print(f"fp8 T=2048 vs exact: max {md:.3e}, rel-L2 {l2:.3e}")
    _, _, y2 = run_prefill_fp8(L, x_host, ids, w)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_prefill_fp8_largest_chunk_sampled_tokens():
    # the largest chunk the call takes (16384 tokens), Xing shape: bucketing,
    # tile schedule, token exponents and h conversion at their maximum
    moe = lib()
    s = synth.SHAPES[4]
    L = layer_of(4, 2)
    T = 16384
    shape = moe_shape(s)
    assert moe.workspace_bytes(shape, T, moe.PREFILL_FP8) > 0
    assert moe.workspace_bytes(shape, T + 1, moe.PREFILL_FP8) == 0
    x_host = synth.x_rows(L.seed, 2, s.H, T)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, w, y = run_prefill_fp8(L, x_host, status=status)
    assert int(status.item()) == 0
    rows = np.random.default_rng(1).choice(T, 10, replace=False)
    rows = np.sort(np.concatenate([rows, [0, T - 1]]))
    check_close(y[rows], oracle_rows(L, x_host, ids, w, rows), "prefill fp8 T=16384 sampled")


def test_prefill_fp8_empty_chunk():
    # T = 0: nothing to do, nothing launched, y untouched
    moe = lib()
    L = layer_of(SMALL, 0, seed=3)
    s = L.shape
    shape = moe_shape(s)
    wts = weights_of(L)
    rexp = moe.fp8_row_exponents(shape, wts)
    x = torch.zeros((0, s.H), dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros((0, s.k), dtype=torch.int32, device=DEV)
    w = torch.zeros((0, s.k), dtype=torch.float32, device=DEV)
    y = moe.iq4nl_prefill_grouped_fp8(shape, wts, rexp, x, ids, w,
                                      moe.workspace(shape, 1, moe.PREFILL_FP8, DEV))
    torch.cuda.synchronize()
    assert tuple(y.shape) == (0, s.H)
    assert moe.launches_per_call(shape, 0, 5) == 0


@pytest.mark.parametrize("H,F,E,k,T,ns", [
    (256, 256, 1, 1, 3, 0),        # one expert, no shared expert
    (256, 512, 16, 4, 300, 1),     # four 128-row weight tiles, ragged token tiles
    (512, 256, 64, 6, 257, 0),     # many nearly empty buckets
])
def test_prefill_fp8_edge_shapes(H, F, E, k, T, ns):
    s = synth.Shape("pf8-edge", H, F, E, k, T, 1, n_shared=ns)
    L = layer_of(s, 0, seed=5)
    rng = np.random.default_rng(H + F + T)
    x_host = synth.to_bf16_bits(rng.standard_normal((T, H)))
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    _, _, y = run_prefill_fp8(L, x_host, ids, w)
    rows = np.arange(T) if T <= 64 else np.sort(rng.choice(T, 40, replace=False))
    check_close(y[rows], oracle_rows(L, x_host, ids, w, rows), f"prefill fp8 edge H{H} F{F} E{E}")


def test_prefill_fp8_invalid_and_duplicate_routes():
    L = layer_of(SMALL, 0, seed=3)
    s = L.shape
    rng = np.random.default_rng(2)
    x_host = synth.to_bf16_bits(rng.standard_normal((4, s.H)))
    ids = np.stack([rng.choice(s.E, s.k, replace=False) for _ in range(4)]).astype(np.int32)
    w = rng.random((4, s.k)).astype(np.float32)
    ids[0, 1] = -3
    ids[2, 0] = s.E
    ids[3, 1] = ids[3, 0]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _, _, y = run_prefill_fp8(L, x_host, ids, w, status=status)
    assert int(status.item()) & 0xFFFF == 2
    check_close(y, oracle_rows(L, x_host, ids, w, np.arange(4)), "prefill fp8 invalid routes")


def test_prefill_fp8_argument_errors():
    moe = lib()
    from synth.layers import bf16_tensor
    L = layer_of(SMALL, 0, seed=3)
    s = L.shape
    shape = moe_shape(s)
    rng = np.random.default_rng(1)
    x = bf16_tensor(synth.to_bf16_bits(rng.standard_normal((4, s.H))), DEV)
    ids, w = moe.route_topk(shape, L.router_w, L.bias, x)
    wts = weights_of(L)
    rexp = moe.fp8_row_exponents(shape, wts)
    # the fp16 path's workspace is smaller than the 8-bit path's
    assert moe.workspace_bytes(shape, 4, moe.PREFILL_FP8) > moe.workspace_bytes(shape, 4, moe.PREFILL)
    with pytest.raises(moe.MoeError) as e:
        moe.iq4nl_prefill_grouped_fp8(shape, wts, rexp, x, ids, w,
                                      moe.workspace(shape, 4, moe.PREFILL, DEV))
    assert e.value.status == moe.MOE_ERR_WORKSPACE
    # ffn a multiple of 128 but not of 256: the fp16 path runs, the 8-bit one refuses
    T0 = layer_of(0)
    s0 = moe_shape(T0.shape)
    x0 = bf16_tensor(gapped_rows(T0, 4), DEV)
    ids0, w0 = moe.route_topk(s0, T0.router_w, T0.bias, x0)
    z = torch.zeros(1 << 22, dtype=torch.uint8, device=DEV)
    r0 = torch.zeros(1 << 16, dtype=torch.int8, device=DEV)
    with pytest.raises(moe.MoeError) as e:
        moe._check(moe._lib.moe_iq4nl_prefill_grouped_fp8(
            __import__("ctypes").byref(s0), __import__("ctypes").byref(weights_of(T0).c),
            moe._ptr(r0), moe._ptr(x0), 4, moe._ptr(ids0), moe._ptr(w0),
            moe._ptr(torch.empty((4, T0.shape.H), dtype=torch.float32, device=DEV)), moe._ptr(z),
            z.numel(), None, None), "fp8")
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    assert moe.launches_per_call(s0, 4, 5) == 0
    assert moe.launches_per_call(shape, 4, 5) == 6

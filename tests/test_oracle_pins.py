"""Pins of the CPU oracle against facts fixed outside it: the printed IQ4_NL
table, hand-built blocks, numpy's IEEE conversions, PyTorch's E4M3 conversion,
brute-force top-k, a dense numpy SwiGLU, the vLLM article's route-sanitiser
example, and invariances."""
import numpy as np
import pytest

import oracle
import synth
from _util import (bf16_to_f64, check_close, golden_kv, golden_table, np_dense,
                   np_e4m3_rows, np_route, np_row_exponents, np_swiglu_expert,
                   np_swiglu_expert_e4m3)


# ---------------------------------------------------------------- table/layout

def test_table_is_the_printed_table():
    t = golden_table()
    assert t.size == 16
    assert np.array_equal(oracle.table(), t)
    assert np.all(np.diff(t) > 0)                       # strictly increasing
    assert t.min() >= -128 and t.max() <= 127           # int8 range
    assert t.sum() == -94
    assert np.count_nonzero((t >= 1) & (t < 13)) == 1 and t[8] == 1


def _block(d_bits: int, qs) -> np.ndarray:
    b = np.zeros(18, np.uint8)
    b[0] = d_bits & 0xFF
    b[1] = d_bits >> 8
    b[2:] = np.asarray(qs, np.uint8)
    return b


def test_block_layout_hand_built():
    T = golden_table().astype(np.float64)
    qs = [j | ((15 - j) << 4) for j in range(16)]
    # d = 1.0: low nibble of byte j is weight j, high nibble is weight j+16
    w = oracle.dequant(_block(0x3C00, qs))
    assert np.array_equal(w[:16], T[np.arange(16)])
    assert np.array_equal(w[16:], T[15 - np.arange(16)])
    # little-endian scale: 0x0400 = 2^-14 (smallest normal), 0x0001 = 2^-24
    assert np.array_equal(oracle.dequant(_block(0x0400, qs))[:16], T * 2.0 ** -14)
    assert np.array_equal(oracle.dequant(_block(0x0001, qs))[16:], T[::-1] * 2.0 ** -24)
    # negative scale flips every sign; 0x4000 = 2.0
    assert np.array_equal(oracle.dequant(_block(0xBC00, qs))[:16], -T)
    assert np.array_equal(oracle.dequant(_block(0x4000, qs))[:16], 2 * T)
    # consecutive blocks are 18 bytes apart
    two = np.concatenate([_block(0x3C00, qs), _block(0x4000, [0x88] * 16)])
    w2 = oracle.dequant(two)
    assert w2.size == 64 and np.all(w2[32:] == 2.0 * T[8])


def test_mma16_dequant_rounds_each_product_to_half():
    rng = np.random.default_rng(7)
    blocks = synth.iq4nl_blocks(99, 0, synth.GATE, 0, 64)
    exact = oracle.dequant(blocks, oracle.EXACT)
    r16 = oracle.dequant(blocks, oracle.MMA16)
    assert np.array_equal(r16, exact.astype(np.float16).astype(np.float64))
    # products are exact in double: d has 11 significant bits and |T| <= 127
    d = blocks[:, 0:2].copy().view("<f2").astype(np.float64)
    assert np.all(np.abs(exact.reshape(-1, 32)) <= 127 * np.abs(d) + 0)
    del rng


# ---------------------------------------------------------------- IEEE decoders

def test_half_decoder_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32)
    ref = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_half_encoder_round_to_nearest_even():
    rng = np.random.default_rng(1)
    vals = [1 + 2 ** -11, 1 + 3 * 2 ** -11, 65504.0, 65519.99, 65520.0, 70000.0, 2 ** -25,
            3 * 2 ** -25, 2 ** -24, 2 ** -14, 2 ** -14 - 2 ** -25, 1e-8, -0.0, 0.0,
            float("inf"), -float("inf"), 1e-4, 3.3333e-4, -2.5]
    vals += list(rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 6, 3000))
    vals += list((np.arange(1, 3000) + 0.5) * 2.0 ** -24)          # subnormal ties
    for v in vals:
        ref = int(np.array([v], np.float64).astype(np.float16).view(np.uint16)[0])
        assert oracle.double_to_half(v) == ref, (v, hex(ref))


# ---------------------------------------------------------------- router

def _tiny_router(E, H, seed):
    rng = np.random.default_rng(seed)
    Wr = synth.to_bf16_bits(rng.standard_normal((E, H)) * 0.1)
    b = (rng.standard_normal(E) * 0.01).astype(np.float32)
    x = synth.to_bf16_bits(rng.standard_normal((6, H)))
    return Wr, b, x


@pytest.mark.parametrize("E,k", [(1, 1), (4, 1), (5, 2), (8, 3), (10, 4), (6, 6)])
def test_topk_brute_force(E, k):
    Wr, b, x = _tiny_router(E, 64, seed=E * 10 + k)
    ids, w, gap, _ = oracle.route(Wr, b, x, k)
    ids_ref, w_ref = np_route(Wr, b, x, k)
    assert np.array_equal(ids, ids_ref)
    assert np.allclose(w, w_ref, rtol=0, atol=1e-13)


def test_topk_exact_ties_go_to_lower_index():
    E, H = 8, 64
    Wr, _, x = _tiny_router(E, H, seed=3)
    Wr[5] = Wr[2]                        # experts 2 and 5 always tie
    Wr[7] = Wr[2]
    b = np.zeros(E, np.float32)
    b[[2, 5, 7]] = 1.0                   # ... and are always the top three
    ids, w, gap, _ = oracle.route(Wr, b, x, 2)
    assert np.all(ids == np.array([2, 5]))
    assert np.all(gap == 0.0)            # 5 and 7 tie for the 2nd place
    ids_ref, _ = np_route(Wr, b, x, 2)
    assert np.array_equal(ids, ids_ref)


def test_route_weights_sum_to_one_and_bias_only_selects():
    s = synth.SHAPES[0]
    Wr, b = synth.router(s, 5, 0)
    x = synth.x_rows(5, 0, s.H, 16)
    ids, w, _, scores = oracle.route(Wr, b, x, s.k)
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-12)
    p = 1.0 / (1.0 + np.exp(-scores))
    sel = np.take_along_axis(p, ids, 1)
    assert np.allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-13, atol=0)
    ids1, w1, _, _ = oracle.route(Wr, b, x, 1)
    assert np.all(w1 == 1.0)


def test_sanitizer_worked_example():
    g = golden_kv("route_sanitizer.txt")
    E = int(g["n_experts"][0])
    ids, w, bad = oracle.sanitize(np.array(g["ids_in"], np.int32),
                                  np.array(g["w_in"], np.float64), E)
    assert ids.tolist() == [int(v) for v in g["ids_out"]]
    assert w.tolist() == [float(v) for v in g["w_out"]]
    assert bad == 2


# ---------------------------------------------------------------- expert / layer

def _layer_inputs(shape, seed, T=None, layer=0):
    T = shape.T if T is None else T
    Wr, b = synth.router(shape, seed, layer)
    x = synth.x_rows(seed, layer, shape.H, T)
    ex = {e: synth.expert_mats(shape, seed, layer, e) for e in range(shape.E)}
    sh = synth.shared_mats(shape, seed, layer)
    return Wr, b, x, ex, sh


@pytest.mark.parametrize("mode", [oracle.EXACT, oracle.MMA16])
def test_top1_single_expert_equals_dense_swiglu(mode):
    # E = 1, k = 1, no shared expert: the layer is one dense SwiGLU FFN.
    s = synth.Shape("t", 128, 96, 1, 1, 5, 1, n_shared=0)
    _, _, x, ex, _ = _layer_inputs(s, 11)
    ids = np.zeros((5, 1), np.int32)
    w = np.ones((5, 1))
    y = oracle.moe_layer(s.H, s.F, s.F, 1, 1, 0, ex, None, x, ids, w, mode=mode)
    ref = np_swiglu_expert(ex[0], s.H, s.F, bf16_to_f64(x), fp16=(mode == oracle.MMA16))
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15 * np.abs(ref).max())


def test_layer_equals_dense_masked_evaluation():
    # every expert on every token, densely, then masked by the route table
    s = synth.SHAPES[0]
    Wr, b, x, ex, sh = _layer_inputs(s, 21)
    ids, w, _, _ = oracle.route(Wr, b, x, s.k)
    y = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, ids, w)
    X = bf16_to_f64(x)
    dense = np.stack([np_swiglu_expert(ex[e], s.H, s.F, X) for e in range(s.E)])  # [E,T,H]
    shared = np_swiglu_expert(sh, s.H, s.Fs, X)
    ref = np.zeros_like(y)
    for t in range(s.T):
        mask = np.zeros(s.E)
        mask[ids[t]] = w[t]
        ref[t] = (mask[:, None] * dense[:, t, :]).sum(0) + shared[t]
    assert np.allclose(y, ref, rtol=1e-11, atol=1e-14 * np.abs(ref).max())


def test_closed_form_constant_weights():
    # gate/up/down blocks all index 8 (T = 1) with scales c_g, c_u, c_d and x = 1:
    # g = c_g H, u = c_u H, h = silu(g) u for every f, y = c_d F h (+ nothing shared)
    H, F = 64, 32
    def const_mat(rows, K, dbits):
        blk = _block(dbits, [0x88] * 16)
        return np.tile(blk, rows * K // 32)
    cg, cu, cd = 0x2000, 0x2400, 0x1C00        # 2^-7, 2^-6, 2^-8
    mats = (const_mat(F, H, cg), const_mat(F, H, cu), const_mat(H, F, cd))
    x = np.full((1, H), 0x3F80, np.uint16)      # bf16 1.0
    y = oracle.moe_layer(H, F, F, 1, 1, 0, {0: mats}, None, x, np.zeros((1, 1), np.int32),
                         np.ones((1, 1)))
    g, u = 2.0 ** -7 * H, 2.0 ** -6 * H
    h = g / (1.0 + np.exp(-g)) * u
    assert np.allclose(y, 2.0 ** -8 * F * h, rtol=1e-14)


def test_invariances():
    s = synth.SHAPES[0]
    Wr, b, x, ex, sh = _layer_inputs(s, 31)
    ids, w, _, _ = oracle.route(Wr, b, x, s.k)
    y = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, ids, w)
    # relabelling experts permutes the ids and leaves y unchanged
    perm = np.random.default_rng(0).permutation(s.E)          # new label of old expert e
    Wr_p = np.empty_like(Wr); Wr_p[perm] = Wr
    b_p = np.empty_like(b); b_p[perm] = b
    ex_p = {int(perm[e]): ex[e] for e in ex}
    ids_p, w_p, _, _ = oracle.route(Wr_p, b_p, x, s.k)
    assert np.array_equal(ids_p, perm[ids])
    y_p = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex_p, sh, x, ids_p, w_p)
    assert np.array_equal(y, y_p)
    # doubling every down-projection scale (an exact fp16 exponent step) doubles y
    def dbl(m):
        m = m.copy()
        d = m[:, 0:2].copy().view("<u2")
        m[:, 0:2] = (d + np.uint16(0x0400)).view(np.uint8).reshape(-1, 2)
        return m
    ex2 = {e: (g_, u_, dbl(d_)) for e, (g_, u_, d_) in ex.items()}
    sh2 = (sh[0], sh[1], dbl(sh[2]))
    y2 = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex2, sh2, x, ids, w)
    assert np.array_equal(y2, 2.0 * y)
    # batch invariance: each token alone gives the same row
    for t in range(s.T):
        yt = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x[t:t + 1], ids[t:t + 1],
                              w[t:t + 1])
        assert np.array_equal(yt[0], y[t])


def test_invalid_routes_contribute_nothing():
    s = synth.SHAPES[0]
    Wr, b, x, ex, sh = _layer_inputs(s, 41)
    ids, w, _, _ = oracle.route(Wr, b, x, s.k)
    bad = ids.copy(); bad[0, 1] = -1; bad[2, 0] = s.E + 3
    y = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, bad, w)
    keep = ids.copy(); keep[0, 1] = 0; keep[2, 0] = 0
    w0 = w.copy(); w0[0, 1] = 0; w0[2, 0] = 0
    y_ref = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, keep, w0)
    assert np.array_equal(y, y_ref)


def test_threads_do_not_change_results():
    s = synth.SHAPES[0]
    Wr, b, x, ex, sh = _layer_inputs(s, 51)
    ids, w, _, _ = oracle.route(Wr, b, x, s.k)
    y1 = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, ids, w, threads=1)
    y4 = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, ids, w, threads=4)
    assert np.array_equal(y1, y4)


def test_mma16_is_close_to_exact():
    # information for the prefill reading: fp16 operands move y by ~1e-4 rel-L2
    s = synth.SHAPES[0]
    Wr, b, x, ex, sh = _layer_inputs(s, 61)
    ids, w, _, _ = oracle.route(Wr, b, x, s.k)
    ye = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, ids, w, mode=oracle.EXACT)
    y16 = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, ids, w, mode=oracle.MMA16)
    check_close(y16, ye, "mma16 vs exact", max_rel=5e-3, l2_rel=2e-3)
    assert not np.array_equal(y16, ye)


# ---------------------------------------------------------------- mma8 (E4M3 operands)

def test_e4m3_decoder_all_codes():
    # every one of the 256 codes against PyTorch's float8_e4m3fn decoder
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2      # 0x7F, 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encoder_round_to_nearest_even():
    # every finite code value, every midpoint between neighbours (ties go to the
    # even fraction), the float32 values just around each midpoint, and random
    # values, both signs, against PyTorch's conversion (which agrees up to 464).
    # All are float32 values: PyTorch converts a float64 through float32 first,
    # which would round a double just below a midpoint onto it.
    import torch
    vals = np.array(sorted({oracle.e4m3_to_double(c) for c in range(0x7F)}))   # 0 .. 448
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    near = np.concatenate([np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    rnd = np.random.default_rng(5).uniform(-460, 460, 4000).astype(np.float32)
    small = np.random.default_rng(6).uniform(-2.0 ** -5, 2.0 ** -5, 2000).astype(np.float32)
    v = np.concatenate([vals.astype(np.float32), mids, near, rnd, small, [np.float32(464.0)]])
    v = np.concatenate([v, -v])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.double_to_e4m3(float(x)) for x in v], np.uint8)
    assert np.array_equal(got, ref)
    assert oracle.double_to_e4m3(1.0625) == 0x38 and oracle.double_to_e4m3(1.1875) == 0x3A


def test_e4m3_encoder_saturates():
    # the saturating reading (finite overflow and infinities to +-448, NaN to NaN)
    for v, c in ((448.0, 0x7E), (449.0, 0x7E), (480.0, 0x7E), (1e30, 0x7E),
                 (float("inf"), 0x7E), (-1e30, 0xFE), (-float("inf"), 0xFE)):
        assert oracle.double_to_e4m3(v) == c, v
    assert oracle.double_to_e4m3(float("nan")) & 0x7F == 0x7F


def test_mma8_weights_against_pytorch_rounding():
    s = synth.Shape("t8", 256, 128, 2, 1, 2, 1)
    g, u, d = synth.expert_mats(s, 17, 0, 1)
    for m, rows, K in ((g, 128, 256), (d, 256, 128)):
        w8, ex = oracle.dequant_rows_e4m3(m, rows, K)
        assert np.array_equal(ex, np_row_exponents(m, rows, K))
        ref = np_e4m3_rows(np_dense(m, rows, K), np_row_exponents(m, rows, K))
        assert np.array_equal(w8, ref)
        assert not np.array_equal(w8, np_dense(m, rows, K))           # rounding happened


def test_mma8_single_expert_equals_dense_reference():
    # E = 1, k = 1, no shared expert: one dense SwiGLU FFN with the mma8 roundings
    s = synth.Shape("t", 128, 96, 1, 1, 5, 1, n_shared=0)
    _, _, x, ex, _ = _layer_inputs(s, 11)
    ids = np.zeros((5, 1), np.int32)
    w = np.ones((5, 1))
    y = oracle.moe_layer(s.H, s.F, s.F, 1, 1, 0, ex, None, x, ids, w, mode=oracle.MMA8)
    ref = np_swiglu_expert_e4m3(ex[0], s.H, s.F, bf16_to_f64(x))
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15 * np.abs(ref).max())


@pytest.mark.parametrize("s", [synth.SHAPES[0],
                               synth.Shape("sw", 256, 128, 8, 2, 4, 1, Fs=384),
                               synth.Shape("sn", 256, 384, 8, 2, 4, 1, Fs=128)],
                         ids=["tiny", "shared-wider", "shared-narrower"])
def test_mma8_layer_equals_dense_masked_evaluation(s):
    # also with a shared expert of another width than the routed ones (its h
    # row gets its own exponent)
    Wr, b, x, ex, sh = _layer_inputs(s, 22)
    ids, w, _, _ = oracle.route(Wr, b, x, s.k)
    y = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, ids, w, mode=oracle.MMA8)
    X = bf16_to_f64(x)
    dense = np.stack([np_swiglu_expert_e4m3(ex[e], s.H, s.F, X) for e in range(s.E)])
    shared = np_swiglu_expert_e4m3(sh, s.H, s.Fs, X)
    ref = np.zeros_like(y)
    for t in range(s.T):
        mask = np.zeros(s.E)
        mask[ids[t]] = w[t]
        ref[t] = (mask[:, None] * dense[:, t, :]).sum(0) + shared[t]
    assert np.allclose(y, ref, rtol=1e-11, atol=1e-14 * np.abs(ref).max())


def test_mma8_exponent_steps_scale_exactly():
    # doubling every scale of the up matrices doubles u, so h, and (the h
    # exponent follows) y exactly; doubling every down scale doubles y exactly
    s = synth.SHAPES[0]
    Wr, b, x, ex, sh = _layer_inputs(s, 33)
    ids, w, _, _ = oracle.route(Wr, b, x, s.k)
    def run(ex_, sh_):
        return oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex_, sh_, x, ids, w,
                                mode=oracle.MMA8)
    y = run(ex, sh)
    def dbl(m):
        m = m.copy()
        dd = m[:, 0:2].copy().view("<u2")
        m[:, 0:2] = (dd + np.uint16(0x0400)).view(np.uint8).reshape(-1, 2)
        return m
    y_up = run({e: (g_, dbl(u_), d_) for e, (g_, u_, d_) in ex.items()}, (sh[0], dbl(sh[1]), sh[2]))
    y_dn = run({e: (g_, u_, dbl(d_)) for e, (g_, u_, d_) in ex.items()}, (sh[0], sh[1], dbl(sh[2])))
    assert np.array_equal(y_up, 2.0 * y)
    assert np.array_equal(y_dn, 2.0 * y)


def test_mma8_is_close_to_exact():
    # information: E4M3 operands (3 fraction bits) move y by a few percent
    s = synth.SHAPES[0]
    Wr, b, x, ex, sh = _layer_inputs(s, 61)
    ids, w, _, _ = oracle.route(Wr, b, x, s.k)
    ye = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, ids, w, mode=oracle.EXACT)
    y8 = oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, 1, ex, sh, x, ids, w, mode=oracle.MMA8)
    rel = np.linalg.norm(y8 - ye) / np.linalg.norm(ye)
    assert 1e-3 < rel < 0.1, rel


# ---------------------------------------------------------------- byte budget

def test_xing_byte_budget_matches_page():
    g = golden_kv("xing_byte_budget.txt")
    H, F = int(g["hidden"][0]), int(g["expert_ffn"][0])
    k, L = int(g["top_k"][0]), int(g["moe_layers"][0])
    s = synth.SHAPES[1]
    assert (s.H, s.F, s.k, s.L) == (H, F, k, L)
    per_expert = 3 * H * F * 18 // 32
    assert per_expert == s.expert_bytes()
    routed = per_expert * k * L / 2 ** 30
    shared = per_expert * L / 2 ** 30
    assert round(routed, 3) == float(g["routed_gib"][0])
    assert round(shared, 3) == float(g["shared_gib"][0])

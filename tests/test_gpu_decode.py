"""Parity of the CUDA router, dequantiser and decode path with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import (DEV, check_close, check_route, gapped_rows, lib, moe_shape, oracle_layer,
                  run_decode, weights_of)
from _util import golden_kv

pytestmark = pytest.mark.gpu

_layers = {}


def layer_of(cfg_or_shape, layer=0, seed=None):
    from synth.layers import Layer
    s = synth.SHAPES[cfg_or_shape] if isinstance(cfg_or_shape, int) else cfg_or_shape
    seed = synth.seed_of(cfg_or_shape) if seed is None else seed
    key = (s.name, s.H, s.F, s.E, s.k, s.n_shared, seed, layer)
    if key not in _layers:
        if len(_layers) > 6:
            _layers.clear()
            torch.cuda.empty_cache()
        _layers[key] = Layer(s, seed, layer, device=DEV)
    return _layers[key]


# ---------------------------------------------------------------- inputs, dequant

def test_device_generator_matches_host():
    from synth import device as sdev
    for (layer, tensor, e, nb) in [(0, synth.GATE, 0, 300), (3, synth.DOWN, 7, 1000),
                                   (17, synth.SH_UP, 0, 64)]:
        t = torch.empty((e + 1) * nb * 18, dtype=torch.uint8, device=DEV)
        sdev.fill_iq4nl(t, e + 1, nb, 1235, layer, tensor)
        got = t.view(e + 1, nb, 18)[e].cpu().numpy()
        ref = synth.iq4nl_blocks(1235, layer, tensor, e, nb)
        assert np.array_equal(got, ref)


def _edge_blocks():
    rng = np.random.default_rng(5)
    blocks = synth.iq4nl_blocks(77, 0, synth.GATE, 0, 512)
    edge = [0x0001, 0x03FF, 0x0400, 0x7BFF, 0x8000, 0x0000, 0xFBFF, 0x8001, 0x3C00, 0xBC00,
            0x7C00, 0xFC00]
    extra = np.zeros((len(edge), 18), np.uint8)
    for i, d in enumerate(edge):
        extra[i, 0] = d & 0xFF
        extra[i, 1] = d >> 8
        extra[i, 2:] = rng.integers(0, 256, 16, dtype=np.uint8)
    return np.concatenate([blocks, extra])


@pytest.mark.parametrize("mode", ["multi", "one_token", "fp16"])
@pytest.mark.parametrize("odd", [False, True])
def test_dequant_hot_path_decoders_bit_exact(mode, odd):
    # Each mode runs one of the block decoders the layer kernels call, on the
    # 36-byte block pairs they read: the decode lookup for experts with several
    # tokens (split_pair + iq4_lookup8 + iq4_dot_block), the decode split table
    # for experts with one token (iq4_pair_dot1) and the prefill producers'
    # fp16 decoder (dequant_block_half). The dot-product decoders give each
    # table value through a one-hot activation vector. Every value must equal
    # the oracle's dequantisation bit for bit: exact d*T in fp32, or its
    # round-to-nearest-even fp16 (a last odd block checks the pair tail).
    moe = lib()
    b = _edge_blocks()
    if odd:
        b = b[:-1]
    assert (len(b) % 2 == 1) == odd
    m = {"multi": moe.DEQUANT_FP32, "one_token": moe.DEQUANT_FP32_ONE_TOKEN,
         "fp16": moe.DEQUANT_FP16}[mode]
    out = moe.iq4nl_dequantize(torch.from_numpy(b.reshape(-1)).to(DEV), mode=m).cpu().numpy()
    if mode == "fp16":
        ref = oracle.dequant(b, oracle.MMA16).astype(np.float16)   # already fp16 values
        assert np.array_equal(out.view(np.uint16), ref.reshape(-1).view(np.uint16))
    else:
        ref = oracle.dequant(b, oracle.EXACT).astype(np.float32)   # exact in fp32
        got, want = out.view(np.uint32), ref.reshape(-1).view(np.uint32)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, (mode, bad[:8], out[bad[:8]], ref.reshape(-1)[bad[:8]])


def test_dequant_every_code_in_every_position():
    # 16 blocks whose 32 positions cycle through all 16 codes with a shift per
    # block, so each code sits in each position (low and high nibble) of some
    # block, for each decoder.
    moe = lib()
    blocks = np.zeros((32, 18), np.uint8)
    for i in range(32):
        blocks[i, 0:2] = np.frombuffer(np.float16(0.5 + i / 64).tobytes(), np.uint8)
        for j in range(16):
            lo, hi = (j + i) % 16, (j + 16 + i) % 16
            blocks[i, 2 + j] = lo | (hi << 4)
    flat = torch.from_numpy(blocks.reshape(-1)).to(DEV)
    ref32 = oracle.dequant(blocks, oracle.EXACT).astype(np.float32).reshape(-1)
    ref16 = oracle.dequant(blocks, oracle.MMA16).astype(np.float16).reshape(-1)
    for m in (moe.DEQUANT_FP32, moe.DEQUANT_FP32_ONE_TOKEN):
        out = moe.iq4nl_dequantize(flat, mode=m).cpu().numpy()
        assert np.array_equal(out.view(np.uint32), ref32.view(np.uint32)), m
    out = moe.iq4nl_dequantize(flat, mode=moe.DEQUANT_FP16).cpu().numpy()
    assert np.array_equal(out.view(np.uint16), ref16.view(np.uint16))


def test_dequant_refuses_unknown_mode():
    moe = lib()
    b = torch.zeros(36, dtype=torch.uint8, device=DEV)
    out = torch.zeros(64, dtype=torch.float32, device=DEV)
    st = moe._lib.moe_iq4nl_dequantize(b.data_ptr(), 2, 3, out.data_ptr(), None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_sanitize_worked_example():
    moe = lib()
    g = golden_kv("route_sanitizer.txt")
    ids = torch.tensor([int(v) for v in g["ids_in"]], dtype=torch.int32, device=DEV)
    w = torch.tensor([float(v) for v in g["w_in"]], dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    io, wo = moe.sanitize_routes(ids, w, int(g["n_experts"][0]), status=status)
    assert io.cpu().tolist() == [int(v) for v in g["ids_out"]]
    assert wo.cpu().tolist() == [float(v) for v in g["w_out"]]
    assert int(status.item()) == 2


# ---------------------------------------------------------------- router

@pytest.mark.parametrize("cfg,T", [(0, 4), (1, 1), (2, 2), (3, 1), (3, 16)])
def test_route_parity(cfg, T):
    moe = lib()
    from synth.layers import bf16_tensor
    L = layer_of(cfg)
    x_host = gapped_rows(L, T)
    ids, w = moe.route_topk(moe_shape(L.shape), L.router_w, L.bias, bf16_tensor(x_host, DEV))
    torch.cuda.synchronize()
    check_route(ids.cpu().numpy(), w.cpu().numpy(), L, x_host)


def test_route_token_tiles_ragged():
    # a prefill-sized chunk with a ragged last tile, on the Xing router shape
    moe = lib()
    from synth.layers import bf16_tensor
    L = layer_of(4)
    x_host = gapped_rows(L, 83)
    ids, w = moe.route_topk(moe_shape(L.shape), L.router_w, L.bias, bf16_tensor(x_host, DEV))
    torch.cuda.synchronize()
    check_route(ids.cpu().numpy(), w.cpu().numpy(), L, x_host)


@pytest.mark.parametrize("cfg,T", [(4, 300), (1, 256), (0, 263)])
def test_route_chunk_tensor_cores(cfg, T):
    # chunks of 256+ tokens take the tensor-core router (16-token tiles; 300 =
    # 18 full tiles and a ragged one). The chosen sets must match the oracle
    # exactly. The MMA's fp32 accumulation (its own order and rounding over
    # H/16 steps) moves a score by about 1e-5, and a weight by up to (1 - p)
    # times that, relative: the weights are held to 1e-4 relative, and as a
    # whole to the float bar of the layer outputs.
    moe = lib()
    from synth.layers import bf16_tensor
    L = layer_of(cfg)
    s = L.shape
    x_host = gapped_rows(L, T)
    ids, w = moe.route_topk(moe_shape(s), L.router_w, L.bias, bf16_tensor(x_host, DEV))
    torch.cuda.synchronize()
    ids, w = ids.cpu().numpy(), w.cpu().numpy()
    ids_ref, w_ref, _, scores = oracle.route(L.router_w_host, L.bias_host, x_host, s.k)
    assert np.array_equal(np.sort(ids, 1), np.sort(ids_ref, 1))
    key = 1.0 / (1.0 + np.exp(-scores)) + L.bias_host.astype(np.float64)[None, :]
    assert np.all(np.diff(np.take_along_axis(key, ids.astype(np.int64), 1), axis=1) <= 1e-5)
    got = np.empty_like(w_ref)
    for t in range(T):
        ref = dict(zip(ids_ref[t].tolist(), w_ref[t].tolist()))
        got[t] = [ref[int(e)] for e in ids[t]]
    assert np.allclose(w, got, rtol=1e-4, atol=0)
    check_close(w, got, f"chunk router weights cfg{cfg}")


@pytest.mark.parametrize("T", [4096, 7200])
def test_route_long_chunk_many_experts(T):
    # more than 256 experts keep long chunks on the SIMT router, with 8-token
    # (T = 4096) and 16-token (T = 7200) tiles
    moe = lib()
    from synth.layers import Layer, bf16_tensor
    s = synth.Shape("long chunk E384", 256, 256, 384, 6, T, 1)
    L = Layer(s, 21, 0, device=DEV)
    x_host = gapped_rows(L, T)
    ids, w = moe.route_topk(moe_shape(s), L.router_w, L.bias, bf16_tensor(x_host, DEV))
    torch.cuda.synchronize()
    check_route(ids.cpu().numpy(), w.cpu().numpy(), L, x_host)


def _tied_router(E: int, H: int, seed: int):
    """Zero router rows and biases on a 1/64 grid with many repeats: every
    score is 0, every sigmoid exactly 1/2, every key exactly 1/2 + bias in
    fp32 and fp64 alike, so the k-th choice falls inside a group of equal keys."""
    rng = np.random.default_rng(seed)
    bias = (rng.integers(0, 6, E) / 64.0).astype(np.float32)
    wr_host = np.zeros((E, H), np.uint16)
    return wr_host, bias


@pytest.mark.parametrize("E,k,T", [(64, 4, 1), (64, 4, 40), (64, 4, 2048), (512, 10, 2),
                                   (384, 6, 16), (100, 16, 3)])
def test_route_exact_ties_go_to_lower_index(E, k, T):
    # moe_route_topk on decode batches (cluster tiles) and chunks (token tiles)
    moe = lib()
    from synth.layers import bf16_tensor
    H = 256
    wr_host, bias = _tied_router(E, H, 11 * E + T)
    x_host = synth.x_rows(5, 0, H, T)
    ids_ref, w_ref, gap, _ = oracle.route(wr_host, bias, x_host, k)
    assert gap[0] == 0.0                                         # the cut is inside a tie
    shape = moe.make_shape(H, 256, E, k, 256, 1)
    ids, w = moe.route_topk(shape, bf16_tensor(wr_host, DEV), torch.from_numpy(bias).to(DEV),
                            bf16_tensor(x_host, DEV))
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)           # order included
    assert np.allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=0)


@pytest.mark.parametrize("E,k,T", [(64, 4, 1), (512, 10, 2), (384, 6, 4), (64, 4, 9),
                                   (1024, 16, 2)])
def test_decode_routed_exact_ties(E, k, T):
    # the fused kernel's in-kernel routing (1..4 tokens, up to 512 experts) and
    # the router launched before the layer (5..16 tokens, or more experts), on
    # keys with exact ties
    moe = lib()
    from synth.layers import bf16_tensor
    s = synth.Shape(f"ties E{E}", 256, 256, E, k, T, 1)
    L = layer_of(s, 0, seed=13)
    wr_host, bias = _tied_router(E, s.H, 3 * E + T)
    x_host = synth.x_rows(9, 0, s.H, T)
    ids_ref, w_ref, _, _ = oracle.route(wr_host, bias, x_host, k)
    ws = moe.workspace(moe_shape(s), T, moe.DECODE, DEV)
    ids, w, y = moe.iq4nl_decode_routed(moe_shape(s), bf16_tensor(wr_host, DEV),
                                        torch.from_numpy(bias).to(DEV), weights_of(L),
                                        bf16_tensor(x_host, DEV), ws)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=0)
    check_close(y.cpu().numpy(), oracle_layer(L, x_host, ids_ref, w_ref), f"ties E{E} T{T}")


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("cfg,T,layer", [(0, 4, 0), (0, 1, 0), (1, 1, 0), (1, 1, 37), (2, 2, 0),
                                         (2, 2, 47), (3, 1, 0), (3, 4, 1), (3, 16, 3)])
def test_decode_parity(cfg, T, layer):
    L = layer_of(cfg, layer)
    x_host = gapped_rows(L, T)
    ids, w, y = run_decode(L, x_host)
    check_route(ids, w, L, x_host)
    ref = oracle_layer(L, x_host, ids, w)
    check_close(y, ref, f"decode cfg{cfg} T{T} layer{layer}")


def test_decode_batch_invariance_and_determinism():
    L = layer_of(3, 1)
    x_host = gapped_rows(L, 4)
    ids, w, y = run_decode(L, x_host)
    _, _, y2 = run_decode(L, x_host, ids, w)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
    for t in range(4):
        _, _, yt = run_decode(L, x_host[t:t + 1], ids[t:t + 1], w[t:t + 1])
        assert np.array_equal(yt[0].view(np.uint32), y[t].view(np.uint32)), t


def test_decode_paired_tokens_share_experts():
    # the same token twice (a guess equal to the token): union of experts = k
    L = layer_of(2, 5)
    x1 = gapped_rows(L, 1)
    x_host = np.concatenate([x1, x1])
    ids, w, y = run_decode(L, x_host)
    assert np.array_equal(ids[0], ids[1])
    assert np.array_equal(y[0].view(np.uint32), y[1].view(np.uint32))
    check_close(y, oracle_layer(L, x_host, ids, w), "paired identical tokens")


def test_decode_invalid_and_duplicate_routes():
    L = layer_of(0)
    s = L.shape
    x_host = gapped_rows(L, 4)
    ids, w, _ = run_decode(L, x_host)
    bad = ids.copy()
    bad[0, 1] = -1
    bad[2, 0] = s.E + 5
    bad[3, 1] = bad[3, 0]               # duplicate expert in one token
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _, _, y = run_decode(L, x_host, bad, w, status=status)
    assert int(status.item()) & 0xFFFF == 2
    ref = oracle_layer(L, x_host, bad, w)
    check_close(y, ref, "invalid/duplicate routes")


def _wide_range_x(x_host: np.ndarray) -> np.ndarray:
    """Per token: block 3 holds one value 2^12 times its neighbours' scale,
    block 7 only values near 2^-100, block 11 alternates 2^-20 and 2^10 scales
    (a range of 2^30 inside one 32-value block)."""
    x = synth.bf16_bits_to_f32(x_host).astype(np.float64)
    for t in range(x.shape[0]):
        x[t, 100] = 4096.0 * (1.0 if t % 2 == 0 else -1.0)
        x[t, 224:256] *= 2.0 ** -100
        x[t, 352:384:2] *= 2.0 ** -20
        x[t, 353:384:2] *= 2.0 ** 10
    return synth.to_bf16_bits(x)


# (wide x blocks, shared gate row 5 scaled up, float bar max|diff|/max|ref|, rel-L2)
_WIDE_CASES = {
    "x": (True, False, 1e-3, 5e-4),
    "h": (False, True, 1e-3, 5e-4),
    # Both at once: on the Qwen3-Next shape, u_5 of the shared expert cancels
    # to about 0.5 from terms near 100 while g_5 is near 1e5, so the x
    # rounding (2^-16 of its block's largest value, absolute) becomes a
    # relative error of about 1% in h_5, the largest term of y. A CPU
    # emulation of the int16 arithmetic gives 2.7e-3 / 2.8e-3 here; the bound
    # below records that limit of the 16-bit reading.
    "x+h": (True, True, 5e-3, 5e-3),
}


@pytest.mark.parametrize("case", ["x", "h", "x+h"])
@pytest.mark.parametrize("cfg,T", [(1, 1), (2, 2), (3, 4), (3, 16)])
def test_decode_wide_range_blocks(cfg, T, case):
    # The decode path quantises x and h to 16-bit integers with one power-of-
    # two scale per 32 values; this is where that rounding bites. "x": blocks
    # of x that span up to 2^30. "h": the shared expert's gate row 5 gets block
    # scales 2^10 above its neighbours', so the first 32-value block of the
    # shared expert's h spans more than 2^10. Routes are passed in (taken from
    # the oracle on the same x), so both sides use the same ids.
    from synth.layers import Layer
    wide_x, wide_h, max_rel, l2_rel = _WIDE_CASES[case]
    s = synth.SHAPES[cfg]
    L = Layer(s, synth.seed_of(cfg), 0, device=DEV)
    if wide_h:
        sh = [m.copy() for m in L.shared_bytes_host()]
        nbh = s.H // 32
        big = np.frombuffer(np.float16(0.25).tobytes(), np.uint8)
        sh[0][5 * nbh:6 * nbh, 0:2] = big                 # row 5 of the shared gate
        L.sh_gate.copy_(torch.from_numpy(sh[0].reshape(-1)).to(DEV))
        L.shared_bytes_host = lambda: sh
    x_host = gapped_rows(L, T)
    if wide_x:
        x_host = _wide_range_x(x_host)
    ids, w, _, _ = oracle.route(L.router_w_host, L.bias_host, x_host, s.k)
    _, _, y = run_decode(L, x_host, ids, w.astype(np.float32))
    ref = oracle_layer(L, x_host, ids, w.astype(np.float32).astype(np.float64))
    check_close(y, ref, f"wide-range blocks ({case}) cfg{cfg} T{T}", max_rel, l2_rel)
    del L
    torch.cuda.empty_cache()


def test_barrier_timeout_is_reported_and_recovers():
    # The single-launch decode kernel waits at grid barriers for every CTA.
    # With the barrier limit set to 0, a CTA gives up the first time it finds
    # a barrier incomplete: the call must still return, with MOE_STATUS_TIMEOUT
    # in the status word, and the next call on the same workspace with the
    # default limit must be correct again (the kernel drained its own copies
    # and left the barrier counters at zero).
    moe = lib()
    from synth.layers import bf16_tensor
    L = layer_of(1, 4)
    s = L.shape
    shape = moe_shape(s)
    assert moe.launches_per_call(shape, 1, moe.CALL_DECODE_ROUTED) == 1   # fused path
    x_host = gapped_rows(L, 1)
    x = bf16_tensor(x_host, DEV)
    ws = moe.workspace(shape, 1, moe.DECODE, DEV)
    ids0, w0, y0 = moe.iq4nl_decode_routed(shape, L.router_w, L.bias, weights_of(L), x, ws)
    torch.cuda.synchronize()
    y0 = y0.cpu().numpy()
    check_close(y0, oracle_layer(L, x_host, ids0.cpu().numpy(), w0.cpu().numpy()),
                "before the timeout")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    old = moe.set_barrier_wait_ns(0)
    try:
        moe.iq4nl_decode_routed(shape, L.router_w, L.bias, weights_of(L), x, ws, status=status)
        torch.cuda.synchronize()
    finally:
        assert moe.set_barrier_wait_ns(old) == 0
    assert old == 2_000_000_000
    st = int(status.item()) & 0xFFFFFFFF
    assert st & moe.STATUS_TIMEOUT, hex(st)
    assert st & moe.STATUS_INVALID_ROUTE_MASK == 0
    status.zero_()
    for _ in range(2):
        ids1, w1, y1 = moe.iq4nl_decode_routed(shape, L.router_w, L.bias, weights_of(L), x, ws,
                                               status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(ids1.cpu().numpy(), ids0.cpu().numpy())
        assert np.array_equal(y1.cpu().numpy().view(np.uint32), y0.view(np.uint32))


def test_workspace_reused_across_layers():
    moe = lib()
    s = synth.SHAPES[0]
    L0, L1 = layer_of(0, 0), layer_of(0, 1)
    x0, x1 = gapped_rows(L0, 4), gapped_rows(L1, 4)
    ws = moe.workspace(moe_shape(s), 4, moe.DECODE, DEV)
    ids0, w0, ya = run_decode(L0, x0, ws=ws)
    ids1, w1, yb = run_decode(L1, x1, ws=ws)
    _, _, ya2 = run_decode(L0, x0, ids0, w0)
    _, _, yb2 = run_decode(L1, x1, ids1, w1)
    assert np.array_equal(ya.view(np.uint32), ya2.view(np.uint32))
    assert np.array_equal(yb.view(np.uint32), yb2.view(np.uint32))


@pytest.mark.parametrize("H,F,E,k,T,ns", [
    (64, 64, 1, 1, 1, 0),          # one expert, no shared: a dense SwiGLU
    (64, 64, 1024, 16, 16, 1),     # largest E, k, T: 256 routed pairs
    (128, 192, 5, 3, 7, 1),        # ragged: 3 block pairs per F row, odd T
    (256, 128, 8, 2, 16, 1),       # tiny down rows (72 B, 8-byte multiples)
    (8192, 64, 4, 2, 2, 1),        # widest hidden
    (256, 256, 8, 3, 3, 1),        # single-launch fused path, odd T
    (4096, 512, 2, 2, 4, 0),       # fused path without a shared expert
    (2048, 768, 33, 5, 2, 1),      # fused path, F not a power of two
])
def test_decode_edge_shapes(H, F, E, k, T, ns):
    s = synth.Shape("edge", H, F, E, k, T, 1, n_shared=ns)
    L = layer_of(s, 0, seed=99)
    rng = np.random.default_rng(H + F + E)
    x_host = synth.to_bf16_bits(rng.standard_normal((T, H)))
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    _, _, y = run_decode(L, x_host, ids, w)
    ref = oracle_layer(L, x_host, ids, w.astype(np.float64))
    check_close(y, ref, f"edge H{H} F{F} E{E} k{k} T{T}")


def test_decode_argument_errors():
    moe = lib()
    from synth.layers import bf16_tensor
    L = layer_of(0)
    s = L.shape
    shape = moe_shape(s)
    x = bf16_tensor(gapped_rows(L, 4), DEV)
    ids, w = moe.route_topk(shape, L.router_w, L.bias, x)
    ws = moe.workspace(shape, 4, moe.DECODE, DEV)
    wts = weights_of(L)
    with pytest.raises(moe.MoeError) as e:       # workspace too small
        moe.iq4nl_decode(shape, wts, x, ids, w, ws[:1024])
    assert e.value.status == moe.MOE_ERR_WORKSPACE
    with pytest.raises(moe.MoeError) as e:       # misaligned activations
        xb = torch.empty(4 * s.H + 1, dtype=torch.bfloat16, device=DEV)[1:].view(4, s.H)
        moe.iq4nl_decode(shape, wts, xb, ids, w, ws)
    assert e.value.status == moe.MOE_ERR_MISALIGNED
    big = torch.zeros((17, s.H), dtype=torch.bfloat16, device=DEV)
    ids17 = torch.zeros((17, s.k), dtype=torch.int32, device=DEV)
    w17 = torch.zeros((17, s.k), dtype=torch.float32, device=DEV)
    with pytest.raises(moe.MoeError) as e:       # more than 16 decode tokens
        moe.iq4nl_decode(shape, wts, big, ids17, w17, ws)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    bad_shape = moe.make_shape(s.H, s.F, s.E, s.E + 1)
    with pytest.raises(moe.MoeError) as e:
        moe.iq4nl_decode(bad_shape, wts, x, ids, w, ws)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    empty = torch.zeros((0, s.H), dtype=torch.bfloat16, device=DEV)
    y0 = moe.iq4nl_decode(shape, wts, empty, ids[:0], w[:0], ws)   # T == 0: nothing to do
    assert y0.shape == (0, s.H)


def test_fused_and_two_kernel_paths_agree_bitwise():
    # 1..4 tokens run the fused single-launch kernel, 5..16 the two-kernel
    # path; per token both do the same arithmetic in the same order.
    s = synth.Shape("paths", 512, 256, 16, 4, 6, 1)
    L = layer_of(s, 0, seed=7)
    rng = np.random.default_rng(3)
    x_host = synth.to_bf16_bits(rng.standard_normal((6, s.H)))
    ids = np.stack([rng.choice(s.E, s.k, replace=False) for _ in range(6)]).astype(np.int32)
    w = rng.random((6, s.k)).astype(np.float32)
    _, _, y6 = run_decode(L, x_host, ids, w)
    for t in range(6):
        _, _, y1 = run_decode(L, x_host[t:t + 1], ids[t:t + 1], w[t:t + 1])
        assert np.array_equal(y1[0].view(np.uint32), y6[t].view(np.uint32)), t
    check_close(y6, oracle_layer(L, x_host, ids, w.astype(np.float64)), "paths shape")


@pytest.mark.parametrize("cfg,T,layer", [(1, 1, 3), (2, 2, 7), (3, 1, 2), (3, 4, 0), (0, 4, 0)])
def test_decode_routed_matches_route_then_decode(cfg, T, layer):
    # one call (fused routing where the shape allows) == moe_route_topk + moe_iq4nl_decode
    moe = lib()
    from synth.layers import bf16_tensor
    L = layer_of(cfg, layer)
    s = L.shape
    shape = moe_shape(s)
    x_host = gapped_rows(L, T)
    x = bf16_tensor(x_host, DEV)
    ws = moe.workspace(shape, T, moe.DECODE, DEV)
    ids, w, y = moe.iq4nl_decode_routed(shape, L.router_w, L.bias, weights_of(L), x, ws)
    torch.cuda.synchronize()
    ids, w, y = ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()
    check_route(ids, w, L, x_host)
    ids2, _, _ = run_decode(L, x_host)            # moe_route_topk + moe_iq4nl_decode
    assert np.array_equal(np.sort(ids, 1), np.sort(ids2, 1))
    check_close(y, oracle_layer(L, x_host, ids, w), f"decode_routed cfg{cfg} T{T}")
    # a second call on the same workspace (barrier counters reset) gives the same bits
    ids3, w3, y3 = moe.iq4nl_decode_routed(shape, L.router_w, L.bias, weights_of(L), x, ws)
    torch.cuda.synchronize()
    assert np.array_equal(y3.cpu().numpy().view(np.uint32), y.view(np.uint32))
    n = moe.launches_per_call(shape, T, moe.CALL_DECODE_ROUTED)
    assert n >= 1

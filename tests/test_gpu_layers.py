"""moe_iq4nl_decode_layers: several MoE layers of one shape in one call.

Independent inputs: each layer must give exactly (bit for bit) what
moe_iq4nl_decode_routed gives for that layer, and match the oracle. Chained
inputs (layer l + 1 takes bf16(y_l)): each layer is checked against the oracle
applied to the input the GPU fed it, layer by layer.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV, check_close, gapped_rows, lib, moe_shape, oracle_layer, weights_of

pytestmark = pytest.mark.gpu

_layers = {}


def layers_of(cfg_or_shape, n, seed=None):
    from synth.layers import Layer
    s = synth.SHAPES[cfg_or_shape] if isinstance(cfg_or_shape, int) else cfg_or_shape
    seed = synth.seed_of(cfg_or_shape) if seed is None else seed
    key = (s.name, s.H, s.F, s.E, s.k, s.n_shared, seed, n)
    if key not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        _layers[key] = [Layer(s, seed, l, device=DEV) for l in range(n)]
    return _layers[key]


def spec(Ls):
    return [(weights_of(L), L.router_w, L.bias) for L in Ls]


def routed_one(L, x_host, ws):
    from synth.layers import bf16_tensor
    moe = lib()
    ids, w, y = moe.iq4nl_decode_routed(moe_shape(L.shape), L.router_w, L.bias, weights_of(L),
                                        bf16_tensor(x_host, DEV), ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()


# (config, tokens, layers, one launch for all layers?) The tiny shape's widths
# (ffn 128) are not multiples of 256: it runs layer by layer.
@pytest.mark.parametrize("cfg,T,n,single", [(1, 1, 4, True), (2, 2, 3, True), (0, 4, 2, False),
                                            (3, 1, 2, True)])
def test_layers_independent_match_single_layer_calls(cfg, T, n, single):
    from synth.layers import bf16_tensor
    moe = lib()
    Ls = layers_of(cfg, n)
    s = Ls[0].shape
    shape = moe_shape(s)
    nl = moe.launches_per_call(shape, T, moe.call_decode_layers(n, False))
    assert (nl == 1) == single, nl
    xs = np.stack([gapped_rows(L, T) for L in Ls])
    ws = moe.workspace(shape, T, moe.DECODE, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, w, y = moe.iq4nl_decode_layers(shape, spec(Ls), bf16_tensor(xs, DEV), ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ids, w, y = ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()
    ws1 = moe.workspace(shape, T, moe.DECODE, DEV)
    for l, L in enumerate(Ls):
        i1, w1, y1 = routed_one(L, xs[l], ws1)
        assert np.array_equal(ids[l], i1), l                  # order included
        assert np.array_equal(w[l].view(np.uint32), w1.view(np.uint32)), l
        assert np.array_equal(y[l].view(np.uint32), y1.view(np.uint32)), l
        check_close(y[l], oracle_layer(L, xs[l], ids[l], w[l]), f"layers cfg{cfg} layer {l}")


def _check_chained(Ls, x0, ids, w, y, what):
    """Layer by layer against the oracle, on the input the GPU fed each layer."""
    s = Ls[0].shape
    x_l = x0
    for l, L in enumerate(Ls):
        ids_ref, _, gap, scores = oracle.route(L.router_w_host, L.bias_host, x_l, s.k)
        for t in range(x_l.shape[0]):
            if gap[t] > 1e-4:                   # a clear decision: the same experts
                assert sorted(ids[l, t]) == sorted(ids_ref[t]), (what, l, t)
        # the GPU's own choice is valid: distinct ids, weights p / sum p
        p = 1.0 / (1.0 + np.exp(-scores))
        for t in range(x_l.shape[0]):
            assert len(set(ids[l, t].tolist())) == s.k
            pw = p[t, ids[l, t]]
            assert np.allclose(w[l, t], pw / pw.sum(), rtol=2e-6, atol=1e-7)
        check_close(y[l], oracle_layer(L, x_l, ids[l], w[l]), f"{what} layer {l}")
        x_l = synth.to_bf16_bits(y[l])          # round to nearest even, as the kernel


@pytest.mark.parametrize("cfg,T,n", [(1, 1, 4), (1, 2, 3), (2, 2, 3), (0, 4, 3)])
def test_layers_chained_layer_by_layer(cfg, T, n):
    from synth.layers import bf16_tensor
    moe = lib()
    Ls = layers_of(cfg, n)
    shape = moe_shape(Ls[0].shape)
    x0 = gapped_rows(Ls[0], T)
    ws = moe.workspace(shape, T, moe.DECODE, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, w, y = moe.iq4nl_decode_layers(shape, spec(Ls), bf16_tensor(x0, DEV), ws, chained=True,
                                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ids, w, y = ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()
    _check_chained(Ls, x0, ids, w, y, f"chained cfg{cfg}")
    # the same call again on the same workspace (new score tags): the same bits
    ids2, w2, y2 = moe.iq4nl_decode_layers(shape, spec(Ls), bf16_tensor(x0, DEV), ws,
                                           chained=True)
    torch.cuda.synchronize()
    assert np.array_equal(ids2.cpu().numpy(), ids)
    assert np.array_equal(y2.cpu().numpy().view(np.uint32), y.view(np.uint32))


@pytest.mark.parametrize("chained", [False, True])
def test_layers_launch_per_layer_path(chained):
    # 16 tokens (beyond the single launch's 4): router + layer per layer, with
    # the bf16 rounding kernel between chained layers; the same results
    from synth.layers import bf16_tensor
    moe = lib()
    s = synth.Shape("layers T16", 512, 256, 16, 4, 16, 3)
    Ls = layers_of(s, 3, seed=31)
    shape = moe_shape(s)
    assert moe.launches_per_call(shape, 16, moe.call_decode_layers(3, chained)) > 3
    ws = moe.workspace(shape, 16, moe.DECODE, DEV)
    if chained:
        x0 = gapped_rows(Ls[0], 16)
        ids, w, y = moe.iq4nl_decode_layers(shape, spec(Ls), bf16_tensor(x0, DEV), ws,
                                            chained=True)
        torch.cuda.synchronize()
        _check_chained(Ls, x0, ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy(),
                       "per-layer chained")
    else:
        xs = np.stack([gapped_rows(L, 16) for L in Ls])
        ids, w, y = moe.iq4nl_decode_layers(shape, spec(Ls), bf16_tensor(xs, DEV), ws)
        torch.cuda.synchronize()
        ids, w, y = ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()
        for l, L in enumerate(Ls):
            check_close(y[l], oracle_layer(L, xs[l], ids[l], w[l]), f"per-layer {l}")


@pytest.mark.parametrize("chained", [False, True])
def test_layers_barrier_timeout_is_reported_and_recovers(chained):
    # every grid-wide wait of the kernel (score tags, h counter, y counter)
    # gives up at once with the limit at 0
    from synth.layers import bf16_tensor
    moe = lib()
    Ls = layers_of(1, 3)
    shape = moe_shape(Ls[0].shape)
    xs = bf16_tensor(np.stack([gapped_rows(L, 1) for L in Ls]), DEV)
    xin = xs[0] if chained else xs
    ws = moe.workspace(shape, 1, moe.DECODE, DEV)
    _, _, y0 = moe.iq4nl_decode_layers(shape, spec(Ls), xin, ws, chained=chained)
    torch.cuda.synchronize()
    y0 = y0.cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    old = moe.set_barrier_wait_ns(0)
    try:
        moe.iq4nl_decode_layers(shape, spec(Ls), xin, ws, chained=chained, status=status)
        torch.cuda.synchronize()
    finally:
        moe.set_barrier_wait_ns(old)
    assert int(status.item()) & 0xFFFFFFFF & moe.STATUS_TIMEOUT
    status.zero_()
    _, _, y1 = moe.iq4nl_decode_layers(shape, spec(Ls), xin, ws, chained=chained, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(y1.cpu().numpy().view(np.uint32), y0.view(np.uint32))


def test_layers_argument_errors():
    from synth.layers import bf16_tensor
    moe = lib()
    Ls = layers_of(0, 2)
    shape = moe_shape(Ls[0].shape)
    ws = moe.workspace(shape, 4, moe.DECODE, DEV)
    xs = bf16_tensor(np.stack([gapped_rows(L, 4) for L in Ls]), DEV)
    with pytest.raises(ValueError):                       # one input per layer
        moe.iq4nl_decode_layers(shape, spec(Ls), xs[:1], ws)
    with pytest.raises(moe.MoeError) as e:                # workspace too small
        moe.iq4nl_decode_layers(shape, spec(Ls), xs, ws[:256])
    assert e.value.status == moe.MOE_ERR_WORKSPACE
    big = torch.zeros((2, 17, Ls[0].shape.H), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(moe.MoeError) as e:                # more than 16 tokens
        moe.iq4nl_decode_layers(shape, spec(Ls), big, ws)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG


# (experts, k, tokens): the one-warp selection (64 experts) and the selection
# spread over the warps (1, 2, 3 and 4 tokens; a warp range with no expert)
@pytest.mark.parametrize("E,k,T", [(64, 4, 1), (512, 10, 1), (512, 10, 2), (384, 6, 3),
                                   (100, 16, 4), (512, 16, 4)])
def test_layers_exact_ties(E, k, T):
    # keys with exact ties (zero router rows, biases on a 1/64 grid): every
    # layer's ordered ids equal the oracle's, ties to the lower index
    from synth.layers import bf16_tensor
    moe = lib()
    s = synth.Shape(f"layer ties E{E}", 256, 256, E, k, T, 2)
    Ls = layers_of(s, 2, seed=17)
    shape = moe_shape(s)
    assert moe.launches_per_call(shape, T, moe.call_decode_layers(2, False)) == 1
    rng = np.random.default_rng(E * 7 + T)
    spec_t, routers = [], []
    for L in Ls:
        wr_host = np.zeros((E, s.H), np.uint16)
        bias = (rng.integers(0, 6, E) / 64.0).astype(np.float32)
        routers.append((wr_host, bias))
        spec_t.append((weights_of(L), bf16_tensor(wr_host, DEV), torch.from_numpy(bias).to(DEV)))
    xs = np.stack([synth.x_rows(9, l, s.H, T) for l in range(2)])
    ws = moe.workspace(shape, T, moe.DECODE, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, w, y = moe.iq4nl_decode_layers(shape, spec_t, bf16_tensor(xs, DEV), ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ids, w, y = ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()
    for l, (L, (wr_host, bias)) in enumerate(zip(Ls, routers)):
        ids_ref, w_ref, gap, _ = oracle.route(wr_host, bias, xs[l], k)
        assert gap[0] == 0.0                                   # the cut is inside a tie
        assert np.array_equal(ids[l], ids_ref), l              # order included
        assert np.allclose(w[l], w_ref, rtol=2e-6, atol=0)
        check_close(y[l], oracle_layer(L, xs[l], ids_ref, w_ref), f"layer ties E{E} T{T} {l}")

"""Parity of the tensor-core prefill path with the oracle's fp16-operand mode.

The prefill contraction runs on tcgen05 with fp16 operands: each dequantised
weight is the round-to-nearest-even fp16 of d*T[q], x enters as fp16 and h is
rounded to fp16 before the down projection. The oracle's MMA16 mode computes
exactly that in double precision; the exact mode is within a few 1e-4 of it.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import DEV, check_close, gapped_rows, lib, moe_shape, weights_of
from _util import bf16_to_f64

pytestmark = pytest.mark.gpu

_layers = {}


def layer_of(cfg_or_shape, layer=0, seed=None):
    from synth.layers import Layer
    s = synth.SHAPES[cfg_or_shape] if isinstance(cfg_or_shape, int) else cfg_or_shape
    seed = synth.seed_of(cfg_or_shape) if seed is None else seed
    key = (s.name, s.H, s.F, s.E, s.k, s.n_shared, seed, layer)
    if key not in _layers:
        if len(_layers) > 4:
            _layers.clear()
            torch.cuda.empty_cache()
        _layers[key] = Layer(s, seed, layer, device=DEV)
    return _layers[key]


def run_prefill(L, x_host, ids=None, w=None, status=None):
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
    ws = moe.workspace(shape, T, moe.PREFILL, DEV)
    y = moe.iq4nl_prefill_grouped(shape, weights_of(L), x, ids_t, w_t, ws, status=status)
    torch.cuda.synchronize()
    return ids_t.cpu().numpy(), w_t.cpu().numpy(), y.cpu().numpy()


def oracle_rows(L, x_host, ids, w, rows, mode=oracle.MMA16):
    """Oracle output for the given token rows only."""
    s = L.shape
    ids = np.asarray(ids, np.int32)
    used = sorted({int(e) for e in ids[rows].reshape(-1) if 0 <= e < s.E} | {0})
    experts = {e: L.expert_bytes_host(e) for e in used}
    sh = L.shared_bytes_host() if s.n_shared else None
    return oracle.moe_layer(s.H, s.F, s.Fs, s.E, s.k, s.n_shared, experts, sh, x_host[rows],
                            ids[rows], np.asarray(w, np.float64)[rows], mode=mode, threads=16)


def test_prefill_tiny_config():
    L = layer_of(0)
    x_host = gapped_rows(L, 4)
    ids, w, y = run_prefill(L, x_host)
    rows = np.arange(4)
    check_close(y, oracle_rows(L, x_host, ids, w, rows), "prefill tiny vs mma16")
    # informational bound against the exact oracle: fp16 operands
    check_close(y, oracle_rows(L, x_host, ids, w, rows, oracle.EXACT), "prefill tiny vs exact",
                max_rel=5e-3, l2_rel=3e-3)


def test_prefill_ragged_chunk_xing_shape():
    s = synth.SHAPES[4]
    L = layer_of(4, 0)
    rng = np.random.default_rng(11)
    T = 200                                       # not a multiple of the 256-token tile
    x_host = synth.to_bf16_bits(rng.standard_normal((T, s.H)))
    ids, w, y = run_prefill(L, x_host)
    rows = np.arange(T)
    check_close(y, oracle_rows(L, x_host, ids, w, rows), "prefill T=200 vs mma16")


def test_prefill_full_chunk_sampled_tokens():
    # the full 2048-token chunk with the Zipf-skewed router (load imbalance)
    s = synth.SHAPES[4]
    L = layer_of(4, 1)
    T = s.T
    x_host = synth.x_rows(L.seed, 1, s.H, T)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, w, y = run_prefill(L, x_host, status=status)
    assert int(status.item()) == 0
    counts = np.bincount(ids.reshape(-1), minlength=s.E)
    assert counts.max() > 2 * counts.mean()       # the skew is real
    rows = np.random.default_rng(0).choice(T, 12, replace=False)
    rows = np.sort(np.concatenate([rows, [0, T - 1]]))
    check_close(y[rows], oracle_rows(L, x_host, ids, w, rows), "prefill T=2048 sampled")
    # Distance to the exact definition (fp64, unrounded operands) on the same
    # rows, held to the layer's float bar: fp16 operands keep the chunk inside it.
    md, l2 = check_close(y[rows], oracle_rows(L, x_host, ids, w, rows, oracle.EXACT),
                         "prefill T=2048 sampled vs exact")
    print(f"prefill T=2048 vs exact: max|diff|/max|ref| = {md:.3e}, rel-L2 = {l2:.3e}")
    # deterministic: a second run gives the same bits
    _, _, y2 = run_prefill(L, x_host, ids, w)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_prefill_largest_chunk_sampled_tokens():
    # the largest chunk the call takes (16384 tokens), Xing shape: the bucket
    # sort, the tile schedule and the tensor-core router at their maximum
    moe = lib()
    s = synth.SHAPES[4]
    L = layer_of(4, 2)
    T = 16384
    assert moe.workspace_bytes(moe_shape(s), T, moe.PREFILL) > 0
    assert moe.workspace_bytes(moe_shape(s), T + 1, moe.PREFILL) == 0
    x_host = synth.x_rows(L.seed, 2, s.H, T)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, w, y = run_prefill(L, x_host, status=status)
    assert int(status.item()) == 0
    rows = np.random.default_rng(1).choice(T, 10, replace=False)
    rows = np.sort(np.concatenate([rows, [0, T - 1]]))
    check_close(y[rows], oracle_rows(L, x_host, ids, w, rows), "prefill T=16384 sampled")


@pytest.mark.parametrize("H,F,E,k,T,ns", [
    (128, 128, 1, 1, 3, 0),        # one expert, no shared expert: a dense SwiGLU
    (256, 384, 16, 4, 300, 1),     # three 128-row weight tiles, ragged token tiles
    (512, 256, 64, 6, 257, 0),     # many nearly empty buckets, no shared expert
])
def test_prefill_edge_shapes(H, F, E, k, T, ns):
    s = synth.Shape("pf-edge", H, F, E, k, T, 1, n_shared=ns)
    L = layer_of(s, 0, seed=5)
    rng = np.random.default_rng(H + F + T)
    x_host = synth.to_bf16_bits(rng.standard_normal((T, H)))
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    _, _, y = run_prefill(L, x_host, ids, w)
    rows = np.arange(T) if T <= 64 else np.sort(rng.choice(T, 40, replace=False))
    check_close(y[rows], oracle_rows(L, x_host, ids, w, rows), f"prefill edge H{H} F{F} E{E}")


def test_prefill_invalid_and_duplicate_routes():
    L = layer_of(0)
    s = L.shape
    x_host = gapped_rows(L, 4)
    rng = np.random.default_rng(2)
    ids = np.stack([rng.choice(s.E, s.k, replace=False) for _ in range(4)]).astype(np.int32)
    w = rng.random((4, s.k)).astype(np.float32)
    ids[0, 1] = -3
    ids[2, 0] = s.E
    ids[3, 1] = ids[3, 0]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _, _, y = run_prefill(L, x_host, ids, w, status=status)
    assert int(status.item()) & 0xFFFF == 2
    check_close(y, oracle_rows(L, x_host, ids, w, np.arange(4)), "prefill invalid routes")


def test_prefill_argument_errors():
    moe = lib()
    from synth.layers import bf16_tensor
    L = layer_of(0)
    s = L.shape
    shape = moe_shape(s)
    x = bf16_tensor(gapped_rows(L, 4), DEV)
    ids, w = moe.route_topk(shape, L.router_w, L.bias, x)
    with pytest.raises(moe.MoeError) as e:
        moe.iq4nl_prefill_grouped(shape, weights_of(L), x, ids, w,
                                  moe.workspace(shape, 2, moe.PREFILL, DEV))
    assert e.value.status == moe.MOE_ERR_WORKSPACE
    odd = moe.make_shape(192, 128, 4, 2)        # hidden not a multiple of 128
    z = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoeError) as e:
        moe.iq4nl_prefill_grouped(odd, weights_of(L), x[:, :192].contiguous(), ids, w, z)
    assert e.value.status in (moe.MOE_ERR_UNSUPPORTED, moe.MOE_ERR_WORKSPACE)

"""The Python binding refuses mis-shaped, mistyped or misplaced tensors before
it calls libmoe, so that a wrong tensor never reaches a kernel. Runs on the
CPU: shapes and dtypes are checked before devices, so CPU tensors of the wrong
shape are refused for their shape, and CPU tensors of the right shape for not
being on a CUDA device. No compute call is made."""
import pytest
import torch


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__._moe_build_module().build()
    import quantized_routed_expert_gb300 as m
    return m


def _weights(moe, s, short=None):
    H, F, E, Fs = s.hidden, s.ffn, s.n_experts, s.ffn_shared
    sizes = {"gate": E * F * H // 32 * 18, "up": E * F * H // 32 * 18,
             "down": E * H * F // 32 * 18, "sh_gate": Fs * H // 32 * 18,
             "sh_up": Fs * H // 32 * 18, "sh_down": H * Fs // 32 * 18}
    if short:
        sizes[short] -= 18
    return {k: torch.zeros(v, dtype=torch.uint8) for k, v in sizes.items()}


def _args(moe, T=2):
    s = moe.make_shape(256, 128, 8, 2)
    x = torch.zeros((T, 256), dtype=torch.bfloat16)
    ids = torch.zeros((T, 2), dtype=torch.int32)
    w = torch.zeros((T, 2), dtype=torch.float32)
    y = torch.zeros((T, 256), dtype=torch.float32)
    return s, x, ids, w, y


def test_layer_shapes_are_checked(moe):
    s, x, ids, w, y = _args(moe)
    wt = moe.ExpertWeights(**_weights(moe, s))
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    cases = [
        ("x", dict(x=torch.zeros((2, 255), dtype=torch.bfloat16))),
        ("ids", dict(ids=torch.zeros((2, 3), dtype=torch.int32))),
        ("ids", dict(ids=torch.zeros((3, 2), dtype=torch.int32))),
        ("weights", dict(weights=torch.zeros((2, 1), dtype=torch.float32))),
        ("y", dict(y=torch.zeros((2, 128), dtype=torch.float32))),
    ]
    for name, over in cases:
        a = dict(x=x, ids=ids, weights=w, y=y)
        a.update(over)
        with pytest.raises(ValueError, match=name):
            moe.iq4nl_decode(s, wt, a["x"], a["ids"], a["weights"], ws, y=a["y"])
        with pytest.raises(ValueError, match=name):
            moe.iq4nl_decode_static(s, wt, a["x"], a["ids"], a["weights"], y=a["y"])
        with pytest.raises(ValueError, match=name):
            moe.iq4nl_prefill_grouped(s, wt, a["x"], a["ids"], a["weights"], ws, y=a["y"])


def test_layer_dtypes_are_checked(moe):
    s, x, ids, w, y = _args(moe)
    wt = moe.ExpertWeights(**_weights(moe, s))
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    with pytest.raises(TypeError, match="x"):
        moe.iq4nl_decode(s, wt, x.float(), ids, w, ws, y=y)
    with pytest.raises(TypeError, match="ids"):
        moe.iq4nl_decode(s, wt, x, ids.long(), w, ws, y=y)
    with pytest.raises(TypeError, match="status"):
        moe.iq4nl_decode(s, wt, x, ids, w, ws, y=y, status=torch.zeros(1))


def test_right_shapes_on_the_cpu_are_refused_for_the_device(moe):
    s, x, ids, w, y = _args(moe)
    wt = moe.ExpertWeights(**_weights(moe, s))
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA device"):
        moe.iq4nl_decode(s, wt, x, ids, w, ws, y=y)


@pytest.mark.parametrize("short", ["gate", "up", "down", "sh_gate", "sh_up", "sh_down"])
def test_short_weight_tensors_are_refused(moe, short):
    # byte sizes are checked before anything else about the call
    s, x, ids, w, y = _args(moe)
    wt = moe.ExpertWeights(**_weights(moe, s, short=short))
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    with pytest.raises(ValueError, match=f"{short} holds"):
        moe.iq4nl_decode(s, wt, x, ids, w, ws, y=y)


def test_missing_shared_weights_are_refused(moe):
    s, x, ids, w, y = _args(moe)
    d = _weights(moe, s)
    d["sh_down"] = None
    with pytest.raises(ValueError, match="sh_down is missing"):
        moe.iq4nl_decode(s, moe.ExpertWeights(**d), x, ids, w, None, y=y)


def test_router_shapes_are_checked(moe):
    s = moe.make_shape(256, 128, 8, 2)
    wr = torch.zeros((8, 256), dtype=torch.bfloat16)
    x = torch.zeros((3, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="router_w"):
        moe.route_topk(s, torch.zeros((7, 256), dtype=torch.bfloat16), None, x)
    with pytest.raises(ValueError, match="router_bias"):
        moe.route_topk(s, wr, torch.zeros(9), x)
    with pytest.raises(ValueError, match="x"):
        moe.route_topk(s, wr, None, torch.zeros((3, 128), dtype=torch.bfloat16))


def test_dequantize_arguments_are_checked(moe):
    with pytest.raises(ValueError, match="mode"):
        moe.iq4nl_dequantize(torch.zeros(36, dtype=torch.uint8), mode=7)
    with pytest.raises(ValueError, match="18-byte"):
        moe.iq4nl_dequantize(torch.zeros(35, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA device"):
        moe.iq4nl_dequantize(torch.zeros(36, dtype=torch.uint8))


def test_fp8_prefill_arguments_are_checked(moe):
    s, x, ids, w, y = _args(moe)
    wt = moe.ExpertWeights(**_weights(moe, s))
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    n = 2 * 8 * 128 + 8 * 256 + 2 * 128 + 256       # gate, up, down rows; shared ones
    good = torch.zeros(n, dtype=torch.int8)
    with pytest.raises(TypeError, match="row_exp"):
        moe.iq4nl_prefill_grouped_fp8(s, wt, good.float(), x, ids, w, ws, y=y)
    with pytest.raises(ValueError, match="row_exp"):
        moe.iq4nl_prefill_grouped_fp8(s, wt, good[:-1], x, ids, w, ws, y=y)
    with pytest.raises(ValueError, match="x"):
        moe.iq4nl_prefill_grouped_fp8(s, wt, good, torch.zeros((2, 255), dtype=torch.bfloat16),
                                      ids, w, ws, y=y)
    with pytest.raises(ValueError, match="CUDA device"):
        moe.iq4nl_prefill_grouped_fp8(s, wt, good, x, ids, w, ws, y=y)
    with pytest.raises(ValueError, match="CUDA device"):
        moe.fp8_row_exponents(s, wt)
    with pytest.raises(ValueError, match="18 bytes"):
        moe.iq4nl_dequantize_e4m3(torch.zeros(36, dtype=torch.uint8), 1, 48)
    with pytest.raises(ValueError, match="18 bytes"):
        moe.iq4nl_dequantize_e4m3(torch.zeros(35, dtype=torch.uint8), 1, 64)
    with pytest.raises(ValueError, match="CUDA device"):
        moe.iq4nl_dequantize_e4m3(torch.zeros(36, dtype=torch.uint8), 1, 64)

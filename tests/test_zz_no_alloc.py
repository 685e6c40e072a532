"""moe_iq4nl_decode_static: decode on the library's own fixed scratch.

It must give what moe_iq4nl_decode gives with a caller workspace, call after
call: the scratch keeps whatever the previous call (of any token count, so of
any scratch layout) left in it, and the entry point clears its counters
itself. This file is collected last so that it also runs after every other
GPU test in the same process.
"""
import numpy as np
import pytest
import torch

import synth
from _gpu import DEV, check_close, gapped_rows, lib, moe_shape, weights_of

pytestmark = pytest.mark.gpu

_layers = {}


def layer_of(cfg):
    from synth.layers import Layer
    if cfg not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        _layers[cfg] = Layer(synth.SHAPES[cfg], synth.seed_of(cfg), 0, device=DEV)
    return _layers[cfg]


def inputs(L, T):
    from synth.layers import bf16_tensor
    moe = lib()
    shape = moe_shape(L.shape)
    x = bf16_tensor(gapped_rows(L, T), DEV)
    ids, w = moe.route_topk(shape, L.router_w, L.bias, x)
    return shape, x, ids, w


def with_workspace(L, shape, x, ids, w):
    moe = lib()
    ws = moe.workspace(shape, x.shape[0], moe.DECODE, DEV)
    y = moe.iq4nl_decode(shape, weights_of(L), x, ids, w, ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("cfg,T", [(1, 1), (1, 4), (3, 16), (2, 2)])
def test_static_matches_workspace_decode_twice(cfg, T):
    moe = lib()
    L = layer_of(cfg)
    shape, x, ids, w = inputs(L, T)
    assert moe.workspace_bytes(shape, T, moe.DECODE) <= moe.STATIC_SCRATCH_BYTES
    ref = with_workspace(L, shape, x, ids, w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = torch.empty((T, shape.hidden), dtype=torch.float32, device=DEV)
    for call in range(2):
        y.fill_(float("nan"))
        moe.iq4nl_decode_static(shape, weights_of(L), x, ids, w, y=y, status=status)
        torch.cuda.synchronize()
        check_close(y.cpu().numpy(), ref, f"static decode cfg {cfg} T={T} call {call}")
    assert int(status.item()) == 0


def test_static_after_a_different_token_count():
    # A 16-token call fills the scratch with h and records at offsets where a
    # 1-token call keeps its counters; the next call must not see them.
    moe = lib()
    L = layer_of(1)
    shape, x16, ids16, w16 = inputs(L, 16)
    ref16 = with_workspace(L, shape, x16, ids16, w16)
    x1, ids1, w1 = x16[:1].contiguous(), ids16[:1].contiguous(), w16[:1].contiguous()
    ref1 = with_workspace(L, shape, x1, ids1, w1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        y16 = moe.iq4nl_decode_static(shape, weights_of(L), x16, ids16, w16, status=status)
        y1 = moe.iq4nl_decode_static(shape, weights_of(L), x1, ids1, w1, status=status)
        torch.cuda.synchronize()
        check_close(y16.cpu().numpy(), ref16, "static decode T=16")
        check_close(y1.cpu().numpy(), ref1, "static decode T=1 after T=16")
    assert int(status.item()) == 0


def test_static_call_allocates_no_device_memory():
    # The raw C call, with every buffer made beforehand: the device's free
    # memory (cudaMemGetInfo, which sees every allocation in the process, the
    # caching allocator's included) and torch's own counters are the same
    # before and after a call. The first call on the device is made before
    # measuring, since loading the library's kernels may map their code and
    # the fixed scratch itself.
    import ctypes
    moe = lib()
    L = layer_of(1)
    shape, x, ids, w = inputs(L, 4)
    y = torch.empty((4, shape.hidden), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    wts = weights_of(L)
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        st = moe._lib.moe_iq4nl_decode_static(ctypes.byref(shape), ctypes.byref(wts.c),
                                              x.data_ptr(), 4, ids.data_ptr(), w.data_ptr(),
                                              y.data_ptr(), status.data_ptr(), stream)
        assert st == moe.MOE_OK
        torch.cuda.synchronize()

    call()
    free0, _ = torch.cuda.mem_get_info()
    alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    for _ in range(3):
        call()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.memory_reserved() == reserved0
    assert int(status.item()) == 0


def test_static_refuses_a_layout_beyond_the_scratch():
    # The C entry point itself refuses a shape whose decode workspace exceeds
    # the fixed scratch, before it launches anything (called directly: the
    # Python wrapper would already refuse these tensors as too small).
    import ctypes
    moe = lib()
    L = layer_of(1)
    big = moe.make_shape(8192, 8192, 64, 16)
    assert moe.workspace_bytes(big, 16, moe.DECODE) > moe.STATIC_SCRATCH_BYTES
    x = torch.zeros((16, 8192), dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros((16, 16), dtype=torch.int32, device=DEV)
    w = torch.zeros((16, 16), dtype=torch.float32, device=DEV)
    y = torch.zeros((16, 8192), dtype=torch.float32, device=DEV)
    st = moe._lib.moe_iq4nl_decode_static(ctypes.byref(big), ctypes.byref(weights_of(L).c),
                                          x.data_ptr(), 16, ids.data_ptr(), w.data_ptr(),
                                          y.data_ptr(), None,
                                          torch.cuda.current_stream().cuda_stream)
    assert st == moe.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool(torch.all(y == 0))                    # nothing ran

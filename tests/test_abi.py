"""The C ABI library loads and exports every function include/moe.h declares;
host-only calls (workspace sizing, status strings, version) answer without a
GPU. No compute call is made here."""
import ctypes
import os
import re

import pytest

from _util import ROOT


def _header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._moe_build_module().build()
    return ctypes.CDLL(path)


def test_header_declares_the_three_calls():
    fns = _header_functions()
    for name in ("moe_route_topk", "moe_iq4nl_decode", "moe_iq4nl_prefill_grouped",
                 "moe_workspace_bytes", "moe_iq4nl_dequantize", "moe_sanitize_routes"):
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name


def test_binding_names_match_header(lib):
    import quantized_routed_expert_gb300 as moe
    assert sorted(moe.EXPORTS) == _header_functions()


def test_status_strings_and_version(lib):
    import quantized_routed_expert_gb300 as moe
    assert moe.status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5):
        assert moe.status_string(code) != "unknown status"
    assert "sm_103a" in moe.version()


def test_workspace_bytes_rules(lib):
    import quantized_routed_expert_gb300 as moe
    s = moe.make_shape(3584, 1024, 64, 4)
    assert moe.workspace_bytes(s, 1, moe.DECODE) > 0
    assert moe.workspace_bytes(s, 16, moe.DECODE) > moe.workspace_bytes(s, 1, moe.DECODE)
    assert moe.workspace_bytes(s, 17, moe.DECODE) == 0          # decode is 1..16 tokens
    assert moe.workspace_bytes(s, 0, moe.DECODE) == 0
    assert moe.workspace_bytes(s, 2048, moe.PREFILL) > 0
    assert moe.workspace_bytes(s, 2, 7) == 0                    # unknown mode
    bad = moe.make_shape(3584, 1024, 64, 65)                     # k > E
    assert moe.workspace_bytes(bad, 1, moe.DECODE) == 0
    odd = moe.make_shape(96, 1024, 64, 4)                        # valid IQ4_NL, not built
    assert moe.workspace_bytes(odd, 1, moe.DECODE) == 0
    # 256-byte aligned regions: size is a multiple of 256
    assert moe.workspace_bytes(s, 3, moe.DECODE) % 256 == 0
    # the 8-bit prefill keeps the fp16 layout's regions and adds its own
    assert moe.workspace_bytes(s, 2048, moe.PREFILL_FP8) > moe.workspace_bytes(s, 2048, moe.PREFILL)
    assert moe.workspace_bytes(s, 16385, moe.PREFILL_FP8) == 0


def test_fp8_row_exponent_count(lib):
    import quantized_routed_expert_gb300 as moe
    s = moe.make_shape(3584, 1024, 64, 4)
    n = lib.moe_fp8_row_exponent_count
    n.restype = ctypes.c_int64
    assert n(ctypes.byref(s)) == 2 * 64 * 1024 + 64 * 3584 + 2 * 1024 + 3584
    bad = moe.make_shape(3584, 1024, 64, 65)
    assert n(ctypes.byref(bad)) == 0


def test_pdl_switch_round_trips(lib):
    import quantized_routed_expert_gb300 as moe
    prev = moe.set_pdl(False)
    assert moe.set_pdl(prev) is False


def test_static_decode_checks_on_the_host(lib):
    # Refusals happen before any CUDA call, so they answer without a GPU.
    import quantized_routed_expert_gb300 as moe
    P = ctypes.c_void_p
    fn = lib.moe_iq4nl_decode_static
    fn.argtypes = [ctypes.POINTER(moe.Shape), P, P, ctypes.c_int32, P, P, P, P, P]
    fn.restype = ctypes.c_int
    big = moe.make_shape(8192, 8192, 64, 16)                     # 16 tokens need > 8 MiB
    assert moe.workspace_bytes(big, 16, moe.DECODE) > moe.STATIC_SCRATCH_BYTES
    assert fn(ctypes.byref(big), None, None, 16, None, None, None, None, None) == \
        moe.MOE_ERR_UNSUPPORTED
    small = moe.make_shape(3584, 1024, 64, 4)
    assert fn(ctypes.byref(small), None, None, 1, None, None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert fn(ctypes.byref(small), None, None, 17, None, None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert fn(ctypes.byref(small), None, None, 0, None, None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG                                  # T == 0 still wants weights

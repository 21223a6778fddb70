"""The C-ABI library loads and exports every symbol the header declares (no GPU calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "include", "moe_verify.h")
LIB = os.path.join(ROOT, "serving_router_softmax_gb300", "libmoeverify.so")


def declared_functions():
    src = open(HDR).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__ as g
        g.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["moe_router_logits", "moe_route", "moe_union_permute", "moe_verify_ffn", "moe_verify_ffn_workspace",
              "eco_select", "moe_verify_step", "moe_verify_step_workspace"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_host_only_calls(lib):
    lib.moe_version.restype = ctypes.c_int
    assert lib.moe_version() >= 100
    lib.moe_status_str.restype = ctypes.c_char_p
    assert lib.moe_status_str(0) == b"ok"
    # argument validation happens before any CUDA call
    from serving_router_softmax_gb300 import _lib as L
    cfg = L.RouteCfg(4, 8, 9, 0, 0, 0.0)  # k > E
    lib.moe_route.argtypes = [ctypes.c_void_p] * 2 + [ctypes.POINTER(L.RouteCfg)] + [ctypes.c_void_p] * 4
    assert lib.moe_route(None, None, ctypes.byref(cfg), None, None, None, None) == L.MOE_ERR_UNSUPPORTED
    ecfg = L.EcoCfg(14, 4, 4, 0, 0.3)  # eps not a power of two
    lib.eco_select.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int32, ctypes.c_void_p,
                                                       ctypes.POINTER(L.EcoCfg)] + [ctypes.c_void_p] * 4
    assert lib.eco_select(None, None, None, 1, None, ctypes.byref(ecfg), None, None, None,
                          None) == L.MOE_ERR_UNSUPPORTED
    rcfg = L.RouterCfg(2, 12, 4, L.DTYPE_BF16, L.DTYPE_BF16)  # H not a multiple of 8
    lib.moe_router_logits.argtypes = [ctypes.c_void_p] * 2 + [ctypes.POINTER(L.RouterCfg)] + [ctypes.c_void_p] * 2
    assert lib.moe_router_logits(None, None, ctypes.byref(rcfg), None, None) == L.MOE_ERR_UNSUPPORTED
    rcfg = L.RouterCfg(0, 64, 4, L.DTYPE_BF16, L.DTYPE_F32)  # T = 0: nothing to do, no pointers needed
    assert lib.moe_router_logits(None, None, ctypes.byref(rcfg), None, None) == L.MOE_OK
    rcfg = L.RouterCfg(2, 64, 4, L.DTYPE_E4M3_B128, L.DTYPE_BF16)  # FP8 activations not accepted
    assert lib.moe_router_logits(None, None, ctypes.byref(rcfg), None, None) == L.MOE_ERR_UNSUPPORTED
    lw = L.LayerWeights(100, 64, 8, 1, 0, None, None, None, None)  # H not a multiple of 64
    lib.moe_verify_ffn_workspace.argtypes = [ctypes.POINTER(L.LayerWeights), ctypes.c_int32, ctypes.c_int32]
    lib.moe_verify_ffn_workspace.restype = ctypes.c_size_t
    assert lib.moe_verify_ffn_workspace(ctypes.byref(lw), 4, 2) == 0

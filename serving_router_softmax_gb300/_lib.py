"""ctypes view of libmoeverify.so (include/moe_verify.h).

Loading fails loudly: there is no fallback implementation of any call.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoeverify.so")

MOE_OK, MOE_ERR_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_WORKSPACE = 0, 1, 2, 3, 4
DEV_NAN_LOGIT, DEV_BAD_ID, DEV_DUP_ID, DEV_BAD_TREE, DEV_BAD_PROB, DEV_TIMEOUT, DEV_CAPACITY = (
    0x01, 0x02, 0x04, 0x08, 0x10, 0x20, 0x40)
DTYPE_F32, DTYPE_BF16, DTYPE_E4M3_B128 = 0, 1, 2
LAYOUT_ROWMAJOR, LAYOUT_TILED = 0, 1
TEST_STALL_GATE_UP, TEST_STALL_READY_FLAG = 1, 2
PROF_CLASSES = ["eco_select", "route", "union_permute", "ffn_prep", "ffn_gate_up", "ffn_down",
                "combine", "router_logits", "s2_expand", "stage_experts", "hot_list", "depth_policy"]

EXPORTED = ["s2_expand", "moe_router_logits", "moe_route", "moe_union_permute", "moe_verify_ffn_workspace", "moe_verify_ffn",
            "eco_select", "moe_verify_step_workspace", "moe_verify_step", "moe_verify_plan", "moe_profile_begin",
            "moe_profile_end", "moe_status_str", "moe_launch_count", "moe_version", "moe_expert_bytes",
            "moe_stage_experts", "moe_test_set_stall", "moe_hot_list", "moe_depth_policy", "moe_set_nvtx"]


class S2Cfg(C.Structure):
    _fields_ = [("N", C.c_int32), ("W", C.c_int32), ("T_AR", C.c_float), ("T_exp", C.c_float),
                ("C_draft", C.c_float), ("T_cold", C.c_float), ("cold_fp", C.c_void_p)]


class DepthCfg(C.Structure):
    _fields_ = [("nseq", C.c_int32), ("D", C.c_int32), ("W", C.c_int32), ("C0", C.c_float),
                ("T_exp", C.c_float)]


class RouterCfg(C.Structure):
    _fields_ = [("T", C.c_int32), ("H", C.c_int32), ("E", C.c_int32), ("x_dtype", C.c_int32),
                ("w_dtype", C.c_int32)]


class RouteCfg(C.Structure):
    _fields_ = [("T", C.c_int32), ("E", C.c_int32), ("k", C.c_int32), ("use_bias", C.c_int32),
                ("cap", C.c_int32), ("alpha", C.c_float)]


class ExpertPool(C.Structure):
    _fields_ = [("n_slots", C.c_int32), ("stage_first", C.c_int32), ("n_stage", C.c_int32),
                ("home_slot", C.c_void_p), ("host_gate_up", C.c_void_p), ("host_down", C.c_void_p),
                ("slot_of", C.c_void_p)]


class LayerWeights(C.Structure):
    _fields_ = [("H", C.c_int32), ("I", C.c_int32), ("E", C.c_int32), ("dtype", C.c_int32),
                ("layout", C.c_int32), ("w_gate_up", C.c_void_p), ("w_down", C.c_void_p),
                ("scales_gate_up", C.c_void_p), ("scales_down", C.c_void_p),
                ("pool", C.POINTER(ExpertPool))]


class EcoCfg(C.Structure):
    _fields_ = [("N", C.c_int32), ("W", C.c_int32), ("gamma_max", C.c_int32), ("mode", C.c_int32),
                ("eps", C.c_float)]


class StepCfg(C.Structure):
    _fields_ = [("L", C.c_int32), ("nseq", C.c_int32), ("N", C.c_int32), ("W", C.c_int32),
                ("E", C.c_int32), ("k", C.c_int32), ("H", C.c_int32), ("I", C.c_int32),
                ("dtype", C.c_int32), ("layout", C.c_int32), ("T", C.c_int32), ("gamma_max", C.c_int32),
                ("mode", C.c_int32), ("eps", C.c_float), ("use_bias", C.c_int32),
                ("cap", C.c_int32), ("alpha", C.c_float)]


_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load the library once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"libmoeverify.so not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = C.CDLL(path)
    vp, i32, sz = C.c_void_p, C.c_int32, C.c_size_t
    P = C.POINTER
    lib.s2_expand.argtypes = [vp, vp, vp, i32, P(S2Cfg), vp, vp, vp, vp, vp]
    lib.s2_expand.restype = C.c_int
    lib.moe_router_logits.argtypes = [vp, vp, P(RouterCfg), vp, vp]
    lib.moe_router_logits.restype = C.c_int
    lib.moe_route.argtypes = [vp, vp, P(RouteCfg), vp, vp, vp, vp]
    lib.moe_route.restype = C.c_int
    lib.moe_union_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.moe_union_permute.restype = C.c_int
    lib.moe_tiled_bytes.argtypes = [P(LayerWeights), P(sz), P(sz)]
    lib.moe_tiled_bytes.restype = sz
    lib.moe_pack_tiled.argtypes = [P(LayerWeights), vp, vp, vp]
    lib.moe_pack_tiled.restype = C.c_int
    lib.moe_expert_bytes.argtypes = [P(LayerWeights), P(sz), P(sz)]
    lib.moe_expert_bytes.restype = sz
    lib.moe_stage_experts.argtypes = [P(LayerWeights), vp, vp, vp, vp, vp]
    lib.moe_stage_experts.restype = C.c_int
    lib.moe_hot_list.argtypes = [vp, C.c_int64, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.moe_hot_list.restype = C.c_int
    lib.moe_depth_policy.argtypes = [vp, vp, vp, P(DepthCfg), vp, vp, vp, vp, vp]
    lib.moe_depth_policy.restype = C.c_int
    lib.moe_verify_ffn_workspace.argtypes = [P(LayerWeights), i32, i32]
    lib.moe_verify_ffn_workspace.restype = sz
    lib.moe_verify_ffn.argtypes = [vp, i32, i32, P(LayerWeights), vp, vp, vp, vp, vp, vp, vp, vp,
                                   sz, vp, vp]
    lib.moe_verify_ffn.restype = C.c_int
    lib.eco_select.argtypes = [vp, vp, vp, i32, vp, P(EcoCfg), vp, vp, vp, vp]
    lib.eco_select.restype = C.c_int
    lib.moe_verify_step_workspace.argtypes = [P(StepCfg)]
    lib.moe_verify_step_workspace.restype = sz
    lib.moe_verify_step.argtypes = [P(StepCfg), vp, vp, vp, vp, vp, vp, P(LayerWeights), vp, vp,
                                    vp, vp, vp, sz, vp, vp]
    lib.moe_verify_step.restype = C.c_int
    lib.moe_verify_plan.argtypes = [P(StepCfg)] + [vp] * 19
    lib.moe_verify_plan.restype = C.c_int
    lib.moe_profile_begin.argtypes = [i32, i32]
    lib.moe_profile_begin.restype = C.c_int
    lib.moe_profile_end.argtypes = [vp, vp, i32]
    lib.moe_profile_end.restype = C.c_int
    lib.moe_status_str.argtypes = [C.c_int]
    lib.moe_status_str.restype = C.c_char_p
    lib.moe_launch_count.argtypes = []
    lib.moe_launch_count.restype = C.c_uint64
    lib.moe_version.argtypes = []
    lib.moe_version.restype = C.c_int
    lib.moe_test_set_stall.argtypes = [i32]
    lib.moe_test_set_stall.restype = C.c_int
    lib.moe_set_nvtx.argtypes = [i32]
    lib.moe_set_nvtx.restype = C.c_int
    _lib = lib
    return lib

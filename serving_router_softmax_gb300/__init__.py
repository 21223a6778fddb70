"""GB300-native MoE speculative-verify hot path (router, reuse bias, expert
union, grouped SwiGLU expert FFN, EcoSpec draft selection, S2-MoE expansion,
expert residency with on-demand staging from host memory).

The computation lives in ``libmoeverify.so`` (hand-written CUDA for sm_103a,
C ABI in ``include/moe_verify.h``); this package only marshals arguments.
Importing it loads the library and raises if it has not been built.
"""
from . import _lib
from .api import (ExpertLayer, ExpertPool, MoEError, StepSpec, VerifyPlan, VerifyStep, depth_policy,  # noqa: F401
                  eco_select,
                  expert_bytes, ffn_workspace_bytes, hot_list, HostExperts, launch_count, new_dev_err, pack_tiled,
                  profile_begin, profile_end, route, router_logits, s2_expand, set_nvtx, stage_experts,
                  step_workspace_bytes, union_permute, verify_ffn)

_lib.load()

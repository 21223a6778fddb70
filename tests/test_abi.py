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


def test_nvtx_switch_is_host_only(lib):
    """moe_set_nvtx accepts 0 and 1 and rejects anything else, with no GPU call."""
    lib.moe_set_nvtx.argtypes = [ctypes.c_int32]
    lib.moe_set_nvtx.restype = ctypes.c_int
    from serving_router_softmax_gb300 import _lib as L
    assert lib.moe_set_nvtx(1) == L.MOE_OK
    assert lib.moe_set_nvtx(0) == L.MOE_OK
    assert lib.moe_set_nvtx(2) == L.MOE_ERR_ARG
    assert lib.moe_set_nvtx(-1) == L.MOE_ERR_ARG


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


def test_ctypes_structs_match_the_header(tmp_path):
    """Field offsets and sizes of every struct the binding mirrors, as the C compiler lays them out."""
    import shutil
    import subprocess
    from serving_router_softmax_gb300 import _lib as L
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    pairs = {"moe_router_cfg": L.RouterCfg, "moe_route_cfg": L.RouteCfg, "moe_expert_pool": L.ExpertPool,
             "moe_layer_weights": L.LayerWeights, "eco_cfg": L.EcoCfg, "moe_step_cfg": L.StepCfg,
             "s2_cfg": L.S2Cfg}
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HDR}"', "int main(void) {"]
    for cname, py in pairs.items():
        lines.append(f'  printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'  printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {(a, b): int(c) for a, b, c in (l.split() for l in out if l)}
    for cname, py in pairs.items():
        assert got[(cname, "sizeof")] == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


def test_expert_pool_validation(lib):
    from serving_router_softmax_gb300 import _lib as L
    L.load()  # sets argtypes on its own handle
    h = L.load()
    fake = 1 << 20  # aligned non-NULL placeholders: validation fails before any use
    lw = L.LayerWeights(128, 256, 8, L.DTYPE_BF16, L.LAYOUT_ROWMAJOR, fake, fake, None, None, None)
    gu, dn = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert h.moe_expert_bytes(ctypes.byref(lw), ctypes.byref(gu), ctypes.byref(dn)) == 3 * 128 * 256 * 2
    assert (gu.value, dn.value) == (2 * 256 * 128 * 2, 128 * 256 * 2)
    lt = L.LayerWeights(128, 192, 8, L.DTYPE_BF16, L.LAYOUT_TILED, fake, fake, None, None, None)
    assert h.moe_expert_bytes(ctypes.byref(lt), ctypes.byref(gu), ctypes.byref(dn)) > 0
    # I = 192: two gate/up row tiles of 128 (the second zero-padded), one down row tile
    assert (gu.value, dn.value) == (2 * 256 * 128 * 2, 1 * 128 * 192 * 2)
    lt = L.LayerWeights(128, 384, 8, L.DTYPE_E4M3_B128, L.LAYOUT_TILED, fake, fake, fake, fake, None)
    assert h.moe_expert_bytes(ctypes.byref(lt), ctypes.byref(gu), ctypes.byref(dn)) > 0
    assert (gu.value, dn.value) == (3 * 256 * 128, 1 * 128 * 384)
    # staging needs a pool
    assert h.moe_stage_experts(ctypes.byref(lw), fake, fake, None, None, None) == L.MOE_ERR_ARG
    bad_pools = [L.ExpertPool(4, 3, 2, fake, fake, fake, fake),   # staging range past n_slots
                 L.ExpertPool(0, 0, 0, fake, fake, fake, fake),   # no slots
                 L.ExpertPool(4, 2, 2, fake, None, fake, fake),   # staging without a host copy
                 L.ExpertPool(4, 2, 2, fake, fake + 8, fake, fake),  # host copy not 16-byte aligned
                 L.ExpertPool(4, 2, 2, None, fake, fake, fake),   # no home-slot table
                 L.ExpertPool(4, 2, 2, fake, fake, fake, None)]   # no slot table
    for pool in bad_pools:
        lw.pool = ctypes.pointer(pool)
        assert h.moe_stage_experts(ctypes.byref(lw), fake, fake, None, None, None) == L.MOE_ERR_ARG
        assert h.moe_verify_ffn_workspace(ctypes.byref(lw), 4, 2) in (0, h.moe_verify_ffn_workspace(
            ctypes.byref(L.LayerWeights(128, 256, 8, L.DTYPE_BF16, L.LAYOUT_ROWMAJOR, fake, fake, None, None,
                                        None)), 4, 2))
    lw.pool = ctypes.pointer(L.ExpertPool(4, 2, 2, fake, fake, fake, fake))
    assert h.moe_stage_experts(ctypes.byref(lw), None, fake, None, None, None) == L.MOE_ERR_ARG
    # a pool cannot be packed
    assert h.moe_pack_tiled(ctypes.byref(lw), fake, fake, None) == L.MOE_ERR_ARG

"""The no-allocation FFN entry point agrees with moe_verify_ffn.

moe_verify_ffn_noalloc exists for callers that cannot allocate device memory
(graph capture, plugin hosts that own the allocator, serving loops that must
not synchronise): it takes inputs and outputs only and keeps its scratch in a
static device array.  This test calls it through the C ABI twice in a row
(the second call runs on the array as the first left it) and compares each
result with the workspace-taking call, within the FFN tolerance the other
tests use.  The file name makes pytest collect it last.
"""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2, "e4m3": 2e-2}


@pytest.fixture(scope="module")
def mv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import serving_router_softmax_gb300 as m
    return m


def rowwise_err(y, ref):
    den = np.max(np.abs(ref), axis=1)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.max(np.abs(y - ref), axis=1) / den))


@pytest.mark.parametrize("dtype,H,I,E,k,T,layout", [
    ("bf16", 576, 320, 16, 4, 5, "rowmajor"), ("f32", 256, 512, 16, 2, 5, "rowmajor"),
    ("bf16", 4096, 1536, 128, 8, 20, "rowmajor"), ("bf16", 4096, 1536, 128, 8, 5, "tiled"),
    ("e4m3", 7168, 2048, 64, 8, 5, "rowmajor"), ("e4m3", 7168, 2048, 64, 8, 5, "tiled")])
def test_noalloc_matches_workspace_call(mv, dtype, H, I, E, k, T, layout):
    from serving_router_softmax_gb300 import _lib as L
    from workload import device as wdev
    from workload import gen

    lib = L.load()
    fn = lib.moe_verify_ffn_noalloc
    fn.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.POINTER(L.LayerWeights)] + [C.c_void_p] * 9
    fn.restype = C.c_int
    lib.moe_verify_ffn_workspace.argtypes = [C.POINTER(L.LayerWeights), C.c_int32, C.c_int32]
    lib.moe_verify_ffn_workspace.restype = C.c_size_t

    cfg = gen.MoEConfig("noalloc", L=1, H=H, E=E, k=k, I=I, dtype=dtype, seed=H + T)
    gu, dn, sgu, sdn = wdev.make_layer_tensors(cfg, 0)
    layer = mv.ExpertLayer(gu, dn, dtype, sgu, sdn)
    if layout == "tiled":
        layer = mv.pack_tiled(layer)
    lw = layer.struct()
    need = lib.moe_verify_ffn_workspace(C.byref(lw), T, k)
    assert 0 < need <= 64 << 20, need
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        rng = np.random.default_rng(100 * call + T)
        lg = (rng.standard_normal((T, E)) - 0.05 * rng.permutation(E)).astype(np.float32)
        xs = rng.standard_normal((T, H)).astype(np.float32)
        x = torch.from_numpy(xs if dtype == "f32" else gen.bf16_bits_rne(xs).view(np.int16)).cuda()
        dev_err = mv.new_dev_err()
        ids, w = mv.route(torch.from_numpy(lg).cuda(), k, dev_err=dev_err)
        up = mv.union_permute(ids, E, dev_err=dev_err)
        ref = mv.verify_ffn(x, k, layer, up, w, dev_err=dev_err)
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        st = fn(x.data_ptr(), T, k, C.byref(lw), up["n_unique"].data_ptr(), up["unique"].data_ptr(),
                up["offsets"].data_ptr(), up["perm_token"].data_ptr(), up["inv"].data_ptr(),
                w.data_ptr(), y.data_ptr(), dev_err.data_ptr(), stream)
        assert st == L.MOE_OK, lib.moe_status_str(st)
        torch.cuda.synchronize()
        assert dev_err.item() == 0
        err = rowwise_err(y.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64))
        assert err < TOL[dtype], (call, err)


def test_noalloc_rejects_sizes_beyond_its_scratch(mv):
    from serving_router_softmax_gb300 import _lib as L
    lib = L.load()
    fn = lib.moe_verify_ffn_noalloc
    fn.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.POINTER(L.LayerWeights)] + [C.c_void_p] * 9
    fn.restype = C.c_int
    # T = 256, k = 16, E = 1024 at H = I = 8192 needs far more than 64 MiB of scratch.
    lw = L.LayerWeights(8192, 8192, 1024, L.DTYPE_BF16, L.LAYOUT_ROWMAJOR, 256, 256, None, None)
    dummy = 256
    st = fn(dummy, 256, 16, C.byref(lw), *([dummy] * 7), None, None)
    assert st == L.MOE_ERR_UNSUPPORTED


def _workspace_need(lib, L, H, I, E, k, T):
    lw = L.LayerWeights(H, I, E, L.DTYPE_BF16, L.LAYOUT_ROWMAJOR, 256, 256, None, None)
    return lib.moe_verify_ffn_workspace(C.byref(lw), T, k)


def test_noalloc_at_the_edge_of_its_scratch(mv):
    """The largest hidden size whose workspace still fits the 64 MiB array
    runs and agrees with the workspace call; the next one is rejected."""
    from serving_router_softmax_gb300 import _lib as L
    from workload import device as wdev
    from workload import gen

    lib = L.load()
    fn = lib.moe_verify_ffn_noalloc
    fn.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.POINTER(L.LayerWeights)] + [C.c_void_p] * 9
    fn.restype = C.c_int
    lib.moe_verify_ffn_workspace.argtypes = [C.POINTER(L.LayerWeights), C.c_int32, C.c_int32]
    lib.moe_verify_ffn_workspace.restype = C.c_size_t
    limit = 64 << 20
    I, E, k, T = 256, 8, 4, 32
    H = 64
    while _workspace_need(lib, L, H + 64, I, E, k, T) <= limit:
        H += 64
    need_in, need_out = _workspace_need(lib, L, H, I, E, k, T), _workspace_need(lib, L, H + 64, I, E, k, T)
    assert need_in <= limit < need_out and need_in > limit - (2 << 20), (H, need_in, need_out)

    # just past the limit: rejected before anything runs
    lw_out = L.LayerWeights(H + 64, I, E, L.DTYPE_BF16, L.LAYOUT_ROWMAJOR, 256, 256, None, None)
    assert fn(256, T, k, C.byref(lw_out), *([256] * 7), None, None) == L.MOE_ERR_UNSUPPORTED

    # at the limit: runs, twice in a row, like the workspace call
    cfg = gen.MoEConfig("noalloc_edge", L=1, H=H, E=E, k=k, I=I, dtype="bf16", seed=7)
    gu, dn, sgu, sdn = wdev.make_layer_tensors(cfg, 0)
    layer = mv.ExpertLayer(gu, dn, "bf16", sgu, sdn)
    lw = layer.struct()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        rng = np.random.default_rng(900 + call)
        lg = (rng.standard_normal((T, E)) - 0.05 * rng.permutation(E)).astype(np.float32)
        x = torch.from_numpy(gen.bf16_bits_rne(rng.standard_normal((T, H)).astype(np.float32)).view(np.int16)).cuda()
        dev_err = mv.new_dev_err()
        ids, w = mv.route(torch.from_numpy(lg).cuda(), k, dev_err=dev_err)
        up = mv.union_permute(ids, E, dev_err=dev_err)
        ref = mv.verify_ffn(x, k, layer, up, w, dev_err=dev_err)
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        st = fn(x.data_ptr(), T, k, C.byref(lw), up["n_unique"].data_ptr(), up["unique"].data_ptr(),
                up["offsets"].data_ptr(), up["perm_token"].data_ptr(), up["inv"].data_ptr(),
                w.data_ptr(), y.data_ptr(), dev_err.data_ptr(), stream)
        assert st == L.MOE_OK, lib.moe_status_str(st)
        torch.cuda.synchronize()
        assert dev_err.item() == 0
        err = rowwise_err(y.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64))
        assert err < TOL["bf16"], (call, err)

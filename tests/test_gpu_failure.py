"""Failure path of the expert FFN without any GPU fault: with the test hook
moe_test_set_stall(MOE_TEST_STALL_GATE_UP) the gate/up producer issues no
copies, so every bounded
wait of that launch runs out after its budget (2 s).  The launch must report
MOE_DEV_TIMEOUT, release its resources and leave the context usable: the next
call gives the oracle's result."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import serving_router_softmax_gb300 as m
    return m


def test_stalled_gate_up_reports_timeout_and_recovers(mv):
    from test_gpu_ffn_step import host_experts, make_layer, rowwise_err, x_decode
    from oracle import moe_layer as ml
    from workload import gen
    import serving_router_softmax_gb300._lib as L
    cfg = gen.MoEConfig("stall_case", L=1, H=576, E=16, k=4, I=320, dtype="bf16", seed=9)
    layer = make_layer(mv, cfg, 0, "tiled")
    rng = np.random.default_rng(4)
    T = 5
    lg = (rng.standard_normal((T, cfg.E)) - 0.1 * rng.permutation(cfg.E)).astype(np.float32)
    x_host = gen.bf16_bits_rne(rng.standard_normal((T, cfg.H)).astype(np.float32))
    x = torch.from_numpy(x_host.view(np.int16).copy()).cuda()
    dev_err = mv.new_dev_err()
    ids, w = mv.route(torch.from_numpy(lg).cuda(), cfg.k, dev_err=dev_err)
    up = mv.union_permute(ids, cfg.E, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0

    lib = L.load()
    assert lib.moe_test_set_stall(L.TEST_STALL_GATE_UP) == L.MOE_OK
    try:
        t0 = time.time()
        mv.verify_ffn(x, cfg.k, layer, up, w, dev_err=dev_err)
        torch.cuda.synchronize()
        waited = time.time() - t0
    finally:
        lib.moe_test_set_stall(0)
    assert dev_err.item() & L.DEV_TIMEOUT
    assert 1.5 < waited < 30.0, waited  # the 2 s budget ran out, nothing hung

    dev_err.zero_()
    y = mv.verify_ffn(x, cfg.k, layer, up, w, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    ref = ml.layer_forward(lg, x_decode(cfg)(x_host), cfg.k, cfg.E, host_experts(cfg, 0))
    assert rowwise_err(y.cpu().numpy().astype(np.float64), ref["y"]) < 2e-2

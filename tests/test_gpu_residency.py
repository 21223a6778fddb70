"""GPU parity of expert residency: the staging kernel against the oracle's plan,
and the FFN / whole step on a pooled layer against the fully resident run
(bit for bit: same kernels, same arithmetic, only the weight addresses differ)
and against the oracle (the tolerances of the FFN tests)."""
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


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def rowwise_err(y, ref):
    den = np.max(np.abs(ref), axis=1)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.max(np.abs(y - ref), axis=1) / den))


def make_layer(mv, cfg, l, layout):
    from workload import device as wdev
    gu, dn, sgu, sdn = wdev.make_layer_tensors(cfg, l)
    layer = mv.ExpertLayer(gu, dn, cfg.dtype, sgu, sdn)
    return mv.pack_tiled(layer) if layout == "tiled" else layer


def routed_inputs(mv, cfg, T, seed):
    from workload import gen
    rng = np.random.default_rng(seed)
    lg = (rng.standard_normal((T, cfg.E)) - 0.1 * rng.permutation(cfg.E)).astype(np.float32)
    xs = rng.standard_normal((T, cfg.H)).astype(np.float32)
    x_host = xs if cfg.dtype == "f32" else gen.bf16_bits_rne(xs)
    x_dev = cuda(xs) if cfg.dtype == "f32" else cuda(x_host.view(np.int16))
    return lg, x_host, x_dev


CASES = [
    # dtype, H, I, E, k, T, layout, hot fraction
    ("bf16", 576, 320, 16, 4, 5, "rowmajor", 0.5),
    ("bf16", 576, 320, 16, 4, 5, "tiled", 0.25),
    ("bf16", 256, 192, 32, 8, 24, "tiled", 0.0),     # nothing resident: every union expert staged
    ("bf16", 256, 192, 8, 8, 3, "tiled", 1.0),       # everything resident: nothing to copy
    ("f32", 256, 512, 16, 2, 5, "rowmajor", 0.5),    # CUDA-core path
    ("e4m3", 640, 384, 16, 4, 5, "rowmajor", 0.5),
    ("e4m3", 256, 256, 32, 8, 28, "tiled", 0.5),
    ("e4m3", 384, 256, 16, 2, 40, "rowmajor", 0.5),  # T > 32: CUDA-core FP8 path
]


@pytest.mark.parametrize("dtype,H,I,E,k,T,layout,frac", CASES)
def test_staged_ffn_matches_resident_and_oracle(mv, dtype, H, I, E, k, T, layout, frac):
    from oracle import moe_layer as ml
    from oracle import residency as R
    from workload import gen
    cfg = gen.MoEConfig("residency_case", L=1, H=H, E=E, k=k, I=I, dtype=dtype, seed=H + 3 * I + T)
    layer = make_layer(mv, cfg, 0, layout)
    lg, x_host, x_dev = routed_inputs(mv, cfg, T, seed=T * 7 + k)
    dev_err = mv.new_dev_err()
    ids, w = mv.route(cuda(lg), k, dev_err=dev_err)
    up = mv.union_permute(ids, E, dev_err=dev_err)
    y_res = mv.verify_ffn(x_dev, k, layer, up, w, dev_err=dev_err).clone()
    torch.cuda.synchronize()
    assert dev_err.item() == 0

    # Hot list from a profiled routing of other tokens (the oracle's rule).
    lg_prof, _, _ = routed_inputs(mv, cfg, 64, seed=991)
    ids_prof, _ = ml.route(lg_prof, k)
    n_hot = int(round(frac * E))
    hot = R.hot_experts(R.activation_counts(ids_prof, E), n_hot)
    hot_dev, counts_dev, home_dev = mv.hot_list(cuda(ids_prof.astype(np.int32).reshape(-1)), E, n_hot)
    assert hot_dev.cpu().tolist() == hot
    assert counts_dev.cpu().tolist() == R.activation_counts(ids_prof, E).tolist()
    assert home_dev.cpu().tolist() == R.home_slots(hot, E).tolist()
    pool = mv.ExpertPool([layer], [hot], n_stage=E - n_hot)
    # The pooled FFN must not read the original device copy.
    layer.gate_up.zero_()
    layer.down.zero_()
    pl = pool.layers[0]
    n_staged = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    mv.stage_experts(pl, up, n_staged=n_staged, dev_err=dev_err)
    y_pool = mv.verify_ffn(x_dev, k, pl, up, w, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0

    U = int(up["n_unique"].item())
    unique = up["unique"][:U].cpu().numpy()
    home = pool.home_slot[0].cpu().numpy()
    slot_ref, staged_ref, errors = R.stage_plan(unique, home, pool.n_slots, pool.stage_first, pool.n_stage)
    assert errors == []
    slot_of = pool.slot_of[0].cpu().numpy()
    assert {int(e): int(slot_of[e]) for e in unique} == slot_ref
    assert int(n_staged.item()) == len(staged_ref)
    gu_host, dn_host = pool.host_gate_up[0].numpy(), pool.host_down[0].numpy()
    for c, e in enumerate(staged_ref):
        s = pool.stage_first + c
        assert np.array_equal(pool.pool_gate_up[s].cpu().numpy(), gu_host[e])
        assert np.array_equal(pool.pool_down[s].cpu().numpy(), dn_host[e])

    assert torch.equal(y_pool, y_res)
    x64 = np.asarray(x_host, np.float64) if dtype == "f32" else ml.decode_bf16(x_host)
    ref = ml.layer_forward(lg, x64, k, E, lambda e: ml.expert_matrices(gen.expert_weights_host(cfg, 0, e), dtype))
    assert rowwise_err(y_pool.cpu().numpy().astype(np.float64), ref["y"]) < TOL[dtype]


def test_stage_capacity_and_bad_home(mv):
    from oracle import residency as R
    from workload import gen
    cfg = gen.MoEConfig("residency_err", L=1, H=256, E=16, k=4, I=128, dtype="bf16", seed=5)
    layer = make_layer(mv, cfg, 0, "rowmajor")
    lg, _, _ = routed_inputs(mv, cfg, 6, seed=3)
    dev_err = mv.new_dev_err()
    ids, w = mv.route(cuda(lg), 4, dev_err=dev_err)
    up = mv.union_permute(ids, 16, dev_err=dev_err)
    torch.cuda.synchronize()
    U = int(up["n_unique"].item())
    unique = up["unique"][:U].cpu().numpy()
    assert U >= 6
    hot = [int(unique[0]), int(unique[1])]
    # Two staging slots for at least four cold experts: the excess get no slot.
    pool = mv.ExpertPool([layer], [hot], n_stage=2)
    n_staged = torch.zeros(1, dtype=torch.int32, device="cuda")
    mv.stage_experts(pool.layers[0], up, n_staged=n_staged, dev_err=dev_err)
    torch.cuda.synchronize()
    import serving_router_softmax_gb300._lib as L
    assert dev_err.item() == L.DEV_CAPACITY
    slot_ref, staged_ref, errors = R.stage_plan(unique, pool.home_slot[0].cpu().numpy(), pool.n_slots,
                                                pool.stage_first, pool.n_stage)
    assert errors == ["capacity"]
    slot_of = pool.slot_of[0].cpu().numpy()
    assert {int(e): int(slot_of[e]) for e in unique} == slot_ref
    assert int(n_staged.item()) == 2
    # The FFN reports the experts left without a slot and reads nothing for them.
    dev_err.zero_()
    mv.verify_ffn(torch.zeros((6, 256), dtype=torch.int16, device="cuda"), 4, pool.layers[0], up, w,
                  dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == L.DEV_BAD_ID

    # A home slot inside the staging range is rejected for that expert.
    pool.home_slot[0][int(unique[0])] = pool.stage_first
    dev_err.zero_()
    mv.stage_experts(pool.layers[0], up, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() & L.DEV_BAD_ID
    assert int(pool.slot_of[0][int(unique[0])].item()) == -1


def test_step_with_pools_matches_resident_step(mv):
    """A whole multi-layer step with every layer pooled (one shared staging range) equals the resident step."""
    from oracle import residency as R
    from workload import device as wdev
    from workload import gen
    from workload import CONFIGS
    cfg = CONFIGS["batched_qwen_like"].replace(L=3, H=256, I=192, E=32, k=4)
    wl = gen.make_workload(cfg)
    t = wdev.workload_tensors(wl)
    layers = [make_layer(mv, cfg, l, "tiled") for l in range(cfg.L)]
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), layout="tiled")
    step = mv.VerifyStep(spec, layers)
    args = (t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    y_res = step(*args).clone()
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    nu_res = step.n_unique.clone()
    # Hot lists: the first 8 experts by a fixed profile; staging holds a whole union.
    hot = [R.hot_experts((np.arange(32) * (l + 3)) % 32, 8) for l in range(cfg.L)]
    pool = mv.ExpertPool(layers, hot, n_stage=32 - 8)
    for ly in layers:
        ly.gate_up.zero_()
        ly.down.zero_()
    pstep = mv.VerifyStep(spec, pool.layers)
    y_pool = pstep(*args)
    torch.cuda.synchronize()
    assert pstep.dev_err.item() == 0
    assert torch.equal(pstep.n_unique, nu_res)
    assert torch.equal(y_pool, y_res)


def _host_mem_available():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def test_step_with_pool_full_size_layer(mv):
    """One Qwen3-235B-like layer at full size (128 experts of 37.7 MB, tiled), half resident by a
    calibration profile: the pooled step equals the resident step bit for bit, and the staged
    bytes of the union's cold experts equal the host copy."""
    from oracle import residency as R
    from workload import CONFIGS, gen
    from workload import device as wdev
    cfg = CONFIGS["qwen3_235b_like"].replace(L=1)
    need = cfg.E * 3 * cfg.H * cfg.I * 2
    if _host_mem_available() < 3 * need:
        pytest.skip("not enough free host memory for the page-locked expert copy")
    free, _ = torch.cuda.mem_get_info()
    if free < 3 * need:
        pytest.skip("not enough free device memory")
    layers = [make_layer(mv, cfg, 0, "tiled")]
    wl = gen.make_workload(cfg)
    t = wdev.workload_tensors(wl)
    spec = mv.StepSpec(L=1, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H, I=cfg.I,
                       dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=cfg.mode, eps=cfg.eps,
                       layout="tiled")
    args = (t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    step = mv.VerifyStep(spec, layers)
    y_res = step(*args).clone()
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    # calibration profile: routing of another seed's workload
    cal = cfg.replace(seed=cfg.seed + 1000)
    wl_cal = gen.make_workload(cal)
    plan = mv.VerifyPlan(mv.StepSpec(L=1, nseq=cal.nseq, N=wl_cal.parent.shape[0], W=cal.W, E=cal.E, k=cal.k,
                                     H=cal.H, I=cal.I, dtype=cal.dtype, T=wl_cal.T,
                                     gamma_max=int(wl_cal.gamma.max()), mode=cal.mode, eps=cal.eps,
                                     layout="tiled"))
    tc = wdev.workload_tensors(wl_cal)
    plan(tc["P"], tc["parent"], tc["own_fp"], tc["gamma"], tc["logits"])
    torch.cuda.synchronize()
    hot = [R.hot_experts(R.activation_counts(plan.ids[0].cpu().numpy(), cfg.E), cfg.E // 2)]
    pool = mv.ExpertPool(layers, hot, n_stage=min(cfg.E // 2, wl.T * cfg.k))
    pstep = mv.VerifyStep(spec, pool.layers)
    y_pool = pstep(*args)
    torch.cuda.synchronize()
    assert pstep.dev_err.item() == 0
    assert torch.equal(y_pool, y_res)
    U = int(pstep.n_unique[0].item())
    plan2 = mv.VerifyPlan(spec)
    plan2(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"])
    torch.cuda.synchronize()
    unique = plan2.unique[0][:U].cpu().numpy()
    slot_ref, staged, errors = R.stage_plan(unique, pool.home_slot[0].cpu().numpy(), pool.n_slots,
                                            pool.stage_first, pool.n_stage)
    assert errors == [] and len(staged) > 0
    slot_of = pool.slot_of[0].cpu().numpy()
    assert {int(e): int(slot_of[e]) for e in unique} == slot_ref
    for c, e in enumerate(staged[:3]):
        s = pool.stage_first + c
        assert torch.equal(pool.pool_gate_up[s].cpu(), pool.host_gate_up[0][e])
        assert torch.equal(pool.pool_down[s].cpu(), pool.host_down[0][e])


def test_pooled_step_in_a_cuda_graph(mv):
    """Staging runs inside a captured step: replays equal the eager pooled step."""
    from oracle import residency as R
    from workload import CONFIGS, gen
    from workload import device as wdev
    cfg = CONFIGS["qwen3_235b_like"].replace(L=2, H=256, I=192, E=32, k=4)
    wl = gen.make_workload(cfg)
    t = wdev.workload_tensors(wl)
    layers = [make_layer(mv, cfg, l, "tiled") for l in range(cfg.L)]
    hot = [R.hot_experts(np.arange(32)[::-1].copy(), 8) for _ in range(cfg.L)]
    pool = mv.ExpertPool(layers, hot, n_stage=24)
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), layout="tiled")
    args = (t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    eager = mv.VerifyStep(spec, pool.layers)
    y0 = eager(*args).clone()
    torch.cuda.synchronize()
    assert eager.dev_err.item() == 0
    step = mv.VerifyStep(spec, pool.layers)
    g = step.capture(*args)
    step.y.zero_()
    pool.pool_gate_up[pool.stage_first:].zero_()  # the replay must stage the cold experts again
    g.replay()
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    assert torch.equal(step.y, y0)


def test_step_mixing_pooled_and_resident_layers(mv):
    """Resident layers hand their union straight from the head to gate/up
    (no prep kernel); pooled layers stage their cold experts and keep the
    prep kernel.  A step that alternates the two equals the all-resident step
    bit for bit."""
    from oracle import residency as R
    from workload import device as wdev
    from workload import gen
    from workload import CONFIGS
    cfg = CONFIGS["qwen3_235b_like"].replace(L=4, H=256, I=192, E=32, k=4)
    wl = gen.make_workload(cfg)
    t = wdev.workload_tensors(wl)
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), layout="tiled")
    args = (t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    resident = [make_layer(mv, cfg, l, "tiled") for l in range(cfg.L)]
    step = mv.VerifyStep(spec, resident)
    y_res = step(*args).clone()
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    hot = [R.hot_experts((np.arange(32) * (l + 5)) % 32, 8) for l in range(cfg.L)]
    pool = mv.ExpertPool([make_layer(mv, cfg, l, "tiled") for l in range(cfg.L)], hot, n_stage=32 - 8)
    mixed = [resident[0], pool.layers[1], resident[2], pool.layers[3]]
    mstep = mv.VerifyStep(spec, mixed)
    for _ in range(2):
        y_mix = mstep(*args)
        torch.cuda.synchronize()
        assert mstep.dev_err.item() == 0
        assert torch.equal(y_mix, y_res)

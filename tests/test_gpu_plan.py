"""GPU parity of moe_verify_plan (the step's selection and per-layer routing
and union, written out) against the oracle, at small and full sizes."""
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


def plan_for(mv, cfg):
    from workload import device as wdev
    from workload import gen
    wl = gen.make_workload(cfg)
    t = wdev.workload_tensors(wl, "cuda")
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=cfg.mode,
                       eps=cfg.eps, use_bias=cfg.use_bias, cap=cfg.cap, alpha=cfg.alpha)
    plan = mv.VerifyPlan(spec)
    plan(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"])
    torch.cuda.synchronize()
    return wl, plan


def check_against_oracle(wl, plan):
    from oracle import moe_layer as ml
    from oracle import verify_step as vs
    cfg = wl.cfg
    assert int(plan.dev_err.item()) == 0
    sels, sizes = vs.run_selection(wl)
    sel = plan.selected.cpu().numpy()
    for s in range(cfg.nseq):
        assert sel[s, : len(sels[s])].tolist() == sels[s]
        assert (sel[s, len(sels[s]):] == -1).all()
    assert plan.union_size.cpu().tolist() == sizes
    rows = vs.verify_rows(wl.parent.shape[0], sels)
    conf = vs.token_conf(wl.P, sels)
    assert plan.verify_rows.cpu().tolist() == list(rows)
    assert np.array_equal(plan.verify_conf.cpu().numpy(), conf)
    ids, w = plan.ids.cpu().numpy(), plan.w.cpu().numpy()
    cap = min(cfg.E, wl.T * cfg.k)
    for l in range(cfg.L):
        lg = wl.logits[l].reshape(-1, cfg.E)[rows]
        if cfg.use_bias:
            lg = ml.reuse_bias(lg, conf, cfg.k, cfg.cap, cfg.alpha)
        rid, rw = ml.route(lg, cfg.k)
        assert np.array_equal(ids[l], rid), f"layer {l} ids"
        np.testing.assert_allclose(w[l], rw, rtol=2e-6, atol=1e-7)
        up = ml.union_permute(rid, cfg.E)
        U = up["n_unique"]
        assert int(plan.n_unique[l]) == U
        assert plan.unique[l, :U].cpu().tolist() == up["unique"].tolist()
        assert plan.offsets[l, : U + 1].cpu().tolist() == up["offsets"].tolist()
        assert plan.perm_token[l].cpu().tolist() == up["perm_token"].tolist()
        assert plan.perm_slot[l].cpu().tolist() == up["perm_slot"].tolist()
        assert plan.inv[l].cpu().tolist() == up["inv"].tolist()
        assert float(plan.reuse_ratio[l]) == float(np.float32(up["reuse_ratio"]))
        assert U <= cap


SMALL = [dict(name="plan_bf16"), dict(name="plan_bias", use_bias=True, cap=8, alpha=0.25),
         dict(name="plan_batched", nseq=4, ragged=True, tau=0.1),
         dict(name="plan_batched_bias", nseq=4, ragged=True, tau=0.1, use_bias=True, cap=6, alpha=0.5),
         dict(name="plan_static", mode=1),
         dict(name="plan_batch_global", nseq=4, ragged=True, tau=0.1, mode=2),
         dict(name="plan_batch_global_bias", nseq=3, mode=2, use_bias=True, cap=6, alpha=0.5),
         # negative and zero lam_b: the biased pass may lower the preferred experts
         dict(name="plan_bias_neg_alpha", use_bias=True, cap=8, alpha=-0.5),
         dict(name="plan_bias_zero_alpha", use_bias=True, cap=8, alpha=0.0),
         dict(name="plan_bias_big_cap", E=64, k=6, use_bias=True, cap=40, alpha=0.25),
         dict(name="plan_bias_wide", E=256, k=8, use_bias=True, cap=16, alpha=1.0)]


@pytest.mark.parametrize("kw", SMALL, ids=[d["name"] for d in SMALL])
def test_plan_small_matches_oracle(mv, kw):
    from workload import gen
    kw = dict(kw)
    cfg = gen.small_case(kw.pop("name"), L=3, **kw)
    wl, plan = plan_for(mv, cfg)
    check_against_oracle(wl, plan)


@pytest.mark.parametrize("name", ["qwen3_235b_like", "gpt_oss_120b_like", "deepseek_v3_like",
                                  "batched_qwen_like"])
def test_plan_full_size_matches_oracle(mv, name):
    from workload import CONFIGS
    wl, plan = plan_for(mv, CONFIGS[name])
    check_against_oracle(wl, plan)


def test_plan_matches_the_step_unions(mv):
    """The plan's per-layer union sizes are the ones the whole step reports."""
    from workload import device as wdev
    from workload import gen
    cfg = gen.small_case("plan_vs_step", L=2, use_bias=True, cap=8, alpha=0.25)
    wl, plan = plan_for(mv, cfg)
    t = wdev.workload_tensors(wl, "cuda")
    layers = []
    for l in range(cfg.L):
        gu, dn, sgu, sdn = wdev.make_layer_tensors(cfg, l, "cuda")
        layers.append(mv.ExpertLayer(gu, dn, cfg.dtype, sgu, sdn))
    step = mv.VerifyStep(plan.spec, layers)
    step(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    torch.cuda.synchronize()
    assert step.n_unique.cpu().tolist() == plan.n_unique.cpu().tolist()


@pytest.mark.parametrize("alpha", [0.25, 2.0])
def test_plan_bias_with_tied_logits(mv, alpha):
    """Logits on a coarse grid: many equal values, so the lower-id rule decides
    in both the unbiased and the biased top-k."""
    from workload import gen
    cfg = gen.small_case("plan_bias_ties", L=3, E=32, k=4, use_bias=True, cap=6, alpha=alpha)
    wl = gen.make_workload(cfg)
    wl.logits = (np.round(wl.logits * 2.0) / 2.0).astype(np.float32)
    from workload import device as wdev
    t = wdev.workload_tensors(wl, "cuda")
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=cfg.mode,
                       eps=cfg.eps, use_bias=True, cap=cfg.cap, alpha=cfg.alpha)
    plan = mv.VerifyPlan(spec)
    plan(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"])
    torch.cuda.synchronize()
    check_against_oracle(wl, plan)


@pytest.mark.parametrize("E,k,use_bias", [(128, 16, True), (256, 16, True), (1024, 16, False), (128, 8, False)])
def test_plan_crowded_and_tied_rows(mv, E, k, use_bias):
    """The layer head's top-k on rows whose winners crowd into a few lanes of
    its warp layout, and on all-equal and coarse-grid rows (test_gpu_kernels'
    crowded_rows), with and without the reuse bias."""
    from test_gpu_kernels import crowded_rows
    from workload import device as wdev
    from workload import gen
    kw = dict(use_bias=True, cap=8, alpha=0.5) if use_bias else {}
    cfg = gen.small_case(f"plan_crowded_{E}_{k}", L=2, E=E, k=k, **kw)
    wl = gen.make_workload(cfg)
    shape = wl.logits.shape
    flat = wl.logits.reshape(-1, E)
    wl.logits = crowded_rows(np.random.default_rng(E + k), flat.shape[0], E, k).reshape(shape)
    t = wdev.workload_tensors(wl, "cuda")
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=cfg.mode,
                       eps=cfg.eps, use_bias=cfg.use_bias, cap=cfg.cap, alpha=cfg.alpha)
    plan = mv.VerifyPlan(spec)
    plan(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"])
    torch.cuda.synchronize()
    check_against_oracle(wl, plan)


def test_plan_fuzz_small_configs(mv):
    """Randomised control-path configurations (experts, top-k, batch, selection
    mode, bias settings) against the oracle: selection, routing and unions."""
    from workload import gen
    rng = np.random.default_rng(2024)
    for trial in range(24):
        E = int(rng.choice([8, 16, 40, 64, 128, 200, 256, 300]))
        k = int(rng.integers(1, min(8, E - 1) + 1))
        L = int(rng.integers(1, 4))
        nseq = int(rng.integers(1, 4))
        mode = int(rng.choice([0, 1, 2])) if nseq > 1 else int(rng.choice([0, 1]))
        use_bias = bool(rng.integers(0, 2))
        kw = dict(L=L, E=E, k=k, nseq=nseq, mode=mode, c=float(rng.uniform(0.0, 0.1)),
                  rho=float(rng.uniform(0.2, 0.9)), seed=int(rng.integers(0, 1 << 20)))
        if nseq > 1:
            kw.update(ragged=bool(rng.integers(0, 2)), tau=0.1)
        if use_bias:
            kw.update(use_bias=True, cap=int(rng.integers(1, min(E, 24) + 1)),
                      alpha=float(rng.choice([-0.5, 0.0, 0.1, 0.25, 1.0, 3.0])))
        cfg = gen.small_case(f"fuzz{trial}", **kw)
        wl, plan = plan_for(mv, cfg)
        check_against_oracle(wl, plan)


def test_plan_in_a_cuda_graph(mv):
    """The control path alone is capturable: replaying a CUDA graph of it gives
    the eager plan's outputs bit for bit."""
    from workload import CONFIGS, gen
    from workload import device as wdev
    cfg = CONFIGS["gpt_oss_120b_like"].replace(L=3)
    wl = gen.make_workload(cfg)
    t = wdev.workload_tensors(wl, "cuda")
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=cfg.mode,
                       eps=cfg.eps, use_bias=cfg.use_bias, cap=cfg.cap, alpha=cfg.alpha)
    args = (t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"])
    eager = mv.VerifyPlan(spec)
    eager(*args)
    plan = mv.VerifyPlan(spec)
    g = plan.capture(*args)
    for x in (plan.ids, plan.unique, plan.perm_token, plan.n_unique):
        x.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert plan.dev_err.item() == 0 and eager.dev_err.item() == 0
    for name in ("selected", "verify_rows", "verify_conf", "ids", "w", "n_unique", "unique", "offsets",
                 "perm_token", "perm_slot", "inv", "reuse_ratio"):
        a, b = getattr(plan, name), getattr(eager, name)
        if name in ("unique", "offsets"):
            for l in range(cfg.L):
                U = int(eager.n_unique[l])
                n = U + 1 if name == "offsets" else U
                assert torch.equal(a[l, :n], b[l, :n]), name
        else:
            assert torch.equal(a, b), name

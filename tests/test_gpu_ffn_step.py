"""GPU parity of the expert FFN and of the whole verify step against the oracle.

Tolerance (written from the arithmetic): the oracle is exact fp64 on the
stored weights; the GPU accumulates in fp32 and, for bf16/FP8 weights, rounds
the SwiGLU intermediate to bf16 (relative error <= 2^-9 per element), so the
row-wise normwise error max_t |y_t - ref_t|_inf / |ref_t|_inf is bounded by
2e-2 for bf16/FP8 and 1e-4 for fp32 weights, the bounds the workloads state.
"""
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
    """The bound the tests hold: max over tokens of |y_t - ref_t|_inf / |ref_t|_inf."""
    den = np.max(np.abs(ref), axis=1)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.max(np.abs(y - ref), axis=1) / den))


def elementwise_err(y, ref):
    """Reported beside the bound: max |y - ref| / max(|ref|, rms(ref)), each
    element against its own size, floored at the output's rms."""
    rms = float(np.sqrt(np.mean(ref * ref))) or 1.0
    return float(np.max(np.abs(y - ref) / np.maximum(np.abs(ref), rms)))


def make_layer(mv, cfg, l, layout="rowmajor"):
    from workload import device as wdev
    gu, dn, sgu, sdn = wdev.make_layer_tensors(cfg, l)
    layer = mv.ExpertLayer(gu, dn, cfg.dtype, sgu, sdn)
    if layout == "tiled":
        layer = mv.pack_tiled(layer)
    return layer


def host_experts(cfg, l):
    from oracle import moe_layer as ml
    from workload import gen
    return lambda e: ml.expert_matrices(gen.expert_weights_host(cfg, l, e), cfg.dtype)


def x_decode(cfg):
    from oracle import moe_layer as ml
    if cfg.dtype == "f32":
        return lambda a: np.asarray(a, np.float32).astype(np.float64)
    return ml.decode_bf16


FFN_CASES = [
    # dtype, H, I, E, k, T
    ("bf16", 576, 320, 16, 4, 5),
    ("bf16", 576, 320, 16, 4, 1),
    ("bf16", 256, 192, 8, 8, 19),      # E == k: every expert used
    ("bf16", 128, 64, 32, 2, 256),     # maximum T
    ("bf16", 640, 384, 64, 16, 9),     # maximum k
    ("f32", 256, 512, 16, 2, 5),       # the fp32 toy shape
    ("f32", 320, 192, 12, 3, 17),
    ("e4m3", 640, 384, 16, 4, 5),
    ("e4m3", 256, 256, 32, 8, 28),
    ("e4m3", 256, 256, 8, 8, 32),      # every expert, maximum T of the FP8 tensor-core path
    ("e4m3", 384, 256, 16, 2, 40),     # T > 32: CUDA-core FP8 path
    ("bf16", 256, 192, 32, 4, 32),     # largest T of the token-dense gate/up (N = 32)
    ("bf16", 256, 192, 32, 4, 33),     # smallest T of the padded-group gate/up
    ("bf16", 128, 64, 1024, 4, 9),     # maximum E
    ("e4m3", 128, 128, 1024, 2, 5),    # maximum E, FP8
]


FFN_CASES_ALL = [c + ("rowmajor",) for c in FFN_CASES] + [
    c + ("tiled",) for c in FFN_CASES if c[0] == "bf16" or (c[0] == "e4m3" and c[5] <= 32)]


@pytest.mark.parametrize("dtype,H,I,E,k,T,layout", FFN_CASES_ALL)
def test_ffn_matches_oracle(mv, dtype, H, I, E, k, T, layout):
    from oracle import moe_layer as ml
    from workload import gen
    cfg = gen.MoEConfig("ffn_case", L=1, H=H, E=E, k=k, I=I, dtype=dtype, seed=H + I + T)
    layer = make_layer(mv, cfg, 0, layout)
    rng = np.random.default_rng(T * 31 + k)
    lg = (rng.standard_normal((T, E)) - 0.1 * rng.permutation(E)).astype(np.float32)
    xs = rng.standard_normal((T, H)).astype(np.float32)
    if dtype == "f32":
        x_host = xs
        x_dev = cuda(xs)
    else:
        x_host = gen.bf16_bits_rne(xs)
        x_dev = cuda(x_host.view(np.int16))
    dev_err = mv.new_dev_err()
    ids, w = mv.route(cuda(lg), k, dev_err=dev_err)
    up = mv.union_permute(ids, E, dev_err=dev_err)
    y = mv.verify_ffn(x_dev, k, layer, up, w, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    ref = ml.layer_forward(lg, x_decode(cfg)(x_host), k, E, host_experts(cfg, 0))
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    yh = y.cpu().numpy().astype(np.float64)
    err = rowwise_err(yh, ref["y"])
    assert err < TOL[dtype], (err, elementwise_err(yh, ref["y"]))


@pytest.mark.parametrize("dtype,layout", [("bf16", "tiled"), ("bf16", "rowmajor"), ("e4m3", "tiled"),
                                          ("f32", "rowmajor")])
def test_ffn_empty_verify_set(mv, dtype, layout):
    """T = 0, the empty verify set: the union is empty, and the FFN call succeeds
    without launching anything or writing a flag."""
    from workload import gen
    cfg = gen.MoEConfig("ffn_empty", L=1, H=256, E=16, k=4, I=256, dtype=dtype, seed=5)
    layer = make_layer(mv, cfg, 0, layout)
    xdt = torch.float32 if dtype == "f32" else torch.int16
    x = torch.zeros((0, cfg.H), dtype=xdt, device="cuda")
    dev_err = mv.new_dev_err()
    up = mv.union_permute(torch.zeros((0, cfg.k), dtype=torch.int32, device="cuda"), cfg.E, dev_err=dev_err)
    w = torch.zeros((0, cfg.k), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    n0 = mv.launch_count()
    y = mv.verify_ffn(x, cfg.k, layer, up, w, dev_err=dev_err)
    torch.cuda.synchronize()
    assert mv.launch_count() == n0
    assert y.shape == (0, cfg.H) and dev_err.item() == 0 and up["n_unique"].item() == 0


def test_ffn_device_fill_matches_host_generator(mv):
    """The device weight fill and the host regeneration agree bit for bit."""
    from workload import gen
    for dtype in ("bf16", "f32", "e4m3"):
        cfg = gen.MoEConfig("fillcheck", L=1, H=256, E=4, k=2, I=128, dtype=dtype, seed=77)
        layer = make_layer(mv, cfg, 0)
        for e in (0, 3):
            hw = gen.expert_weights_host(cfg, 0, e)
            gu = layer.gate_up[e].cpu().numpy()
            dn = layer.down[e].cpu().numpy()
            if dtype == "bf16":
                gu, dn = gu.view(np.uint16), dn.view(np.uint16)
            assert np.array_equal(gu, hw["gate_up"]) and np.array_equal(dn, hw["down"])
            if dtype == "e4m3":
                assert np.array_equal(layer.scales_gate_up[e].cpu().numpy(), hw["scale_gate_up"])
                assert np.array_equal(layer.scales_down[e].cpu().numpy(), hw["scale_down"])


@pytest.mark.parametrize("dtype,H,I", [("bf16", 256, 192), ("bf16", 192, 320), ("e4m3", 256, 384)])
def test_pack_tiled_layout(mv, dtype, H, I):
    """The tiled copy holds exactly the documented block arrangement."""
    from workload import gen
    cfg = gen.MoEConfig("packcheck", L=1, H=H, E=3, k=2, I=I, dtype=dtype, seed=H * I)
    layer = make_layer(mv, cfg, 0)
    tl = mv.pack_tiled(layer)
    torch.cuda.synchronize()
    nt = np.uint16 if dtype == "bf16" else np.uint8
    C = 64 if dtype == "bf16" else 128  # reduction elements per 128-byte block
    gu = tl.gate_up.cpu().numpy().view(nt)
    dn = tl.down.cpu().numpy().view(nt)
    MTg, MTd, KBg, KBd = -(-I // 128), -(-H // 128), H // C, I // C
    gu = gu.reshape(3, MTg, KBg, 256, C)
    dn = dn.reshape(3, MTd, KBd, 128, C)
    for e in range(3):
        w = gen.expert_weights_host(cfg, 0, e)
        g, u, d = w["gate_up"][:I], w["gate_up"][I:], w["down"]
        ref_g = np.zeros((MTg * 128, H), nt)
        ref_u = np.zeros((MTg * 128, H), nt)
        ref_d = np.zeros((MTd * 128, I), nt)
        ref_g[:I], ref_u[:I], ref_d[:H] = g, u, d
        for m in range(MTg):
            for kb in range(KBg):
                blk = gu[e, m, kb]
                assert np.array_equal(blk[:128], ref_g[m * 128:(m + 1) * 128, kb * C:(kb + 1) * C])
                assert np.array_equal(blk[128:], ref_u[m * 128:(m + 1) * 128, kb * C:(kb + 1) * C])
        for m in range(MTd):
            for kb in range(KBd):
                assert np.array_equal(dn[e, m, kb], ref_d[m * 128:(m + 1) * 128, kb * C:(kb + 1) * C])


# ------------------------------------------------------------------ whole step
def run_step(mv, cfg, sample_tokens=None, sample_layers=None, layout="rowmajor"):
    """Runs the GPU step and the oracle; returns (gpu dict, oracle dict)."""
    from oracle import verify_step as ovs
    from workload import device as wdev
    from workload import gen
    wl = gen.make_workload(cfg)
    layers = []
    for l in range(cfg.L):
        layers.append(make_layer(mv, cfg, l, layout))
        torch.cuda.empty_cache()
    t = wdev.workload_tensors(wl)
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k,
                       H=cfg.H, I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()),
                       mode=cfg.mode, eps=cfg.eps, use_bias=cfg.use_bias, cap=cfg.cap,
                       alpha=cfg.alpha, layout=layout)
    step = mv.VerifyStep(spec, layers)
    step(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    torch.cuda.synchronize()
    got = {"selected": step.selected.cpu().numpy(), "union_size": step.union_size.cpu().tolist(),
           "n_unique": step.n_unique.cpu().tolist(), "y": step.y.cpu().numpy(),
           "dev_err": int(step.dev_err.item())}
    del step, layers
    torch.cuda.empty_cache()
    ref = ovs.run_step(wl, lambda l: host_experts(cfg, l), layers=sample_layers,
                       tokens=sample_tokens, x_decode=x_decode(cfg))
    return wl, got, ref


def check_step(wl, got, ref, tol, sample_tokens=None):
    from oracle import moe_layer as ml
    cfg = wl.cfg
    assert got["dev_err"] == 0
    for s in range(cfg.nseq):
        n = len(ref["selected"][s])  # gamma_s, or what the batch-global greedy gave it
        assert got["selected"][s, :n].tolist() == ref["selected"][s]
        assert (got["selected"][s, n:] == -1).all()
    assert got["union_size"] == ref["union_size"]
    # union size of every layer, from oracle routing on all layers
    from oracle import verify_step as ovs
    for l in range(cfg.L):
        lg = wl.logits[l].reshape(-1, cfg.E)[ref["rows"]]
        if cfg.use_bias:
            lg = ml.reuse_bias(lg, ref["conf"], cfg.k, cfg.cap, cfg.alpha)
        ids, _ = ml.route(lg, cfg.k)
        assert got["n_unique"][l] == ml.union_permute(ids, cfg.E)["n_unique"], l
    for l, r in ref["layers"].items():
        toks = list(range(wl.T)) if sample_tokens is None else sample_tokens
        yl = got["y"][l][toks].astype(np.float64)
        err = rowwise_err(yl, r["y"])
        assert err < tol, (l, err, elementwise_err(yl, r["y"]))


SMALL = {
    "toy": {},
    "qwen3_235b_like": dict(L=3, H=512, I=256),
    "gpt_oss_120b_like": dict(L=3, H=576, I=320),
    "deepseek_v3_like": dict(L=2, H=512, I=256),
    "batched_qwen_like": dict(L=2, H=512, I=256),
}


SMALL_CASES = [(n, "rowmajor") for n in SMALL] + [(n, "tiled") for n in SMALL if n != "toy"]


@pytest.mark.parametrize("name,layout", SMALL_CASES)
def test_step_small_shapes_full_compare(mv, name, layout):
    """Every workload's routing/selection structure at reduced H/I: all outputs compared."""
    from workload import CONFIGS
    cfg = CONFIGS[name].replace(**SMALL[name])
    wl, got, ref = run_step(mv, cfg, layout=layout)
    check_step(wl, got, ref, TOL[cfg.dtype])


@pytest.mark.parametrize("layout", ["rowmajor", "tiled"])
@pytest.mark.parametrize("bias", [False, True])
def test_step_batch_global_selection(mv, layout, bias):
    """Batch-global selection (one buffer over the batch, per-sequence depth
    decided by the greedy) through the whole step."""
    from workload import CONFIGS
    kw = dict(L=2, H=512, I=256, mode=2)
    if bias:
        kw.update(use_bias=True, cap=8, alpha=0.25)
    cfg = CONFIGS["batched_qwen_like"].replace(**kw)
    wl, got, ref = run_step(mv, cfg, layout=layout)
    check_step(wl, got, ref, TOL[cfg.dtype])


@pytest.mark.parametrize("name", ["toy", "qwen3_235b_like", "gpt_oss_120b_like", "deepseek_v3_like",
                                  "batched_qwen_like"])
def test_step_full_size_sampled(mv, name):
    """Full-size workloads as the bench runs them: exact selection and unions on
    every layer; FFN outputs on a sample of (layer, token) pairs."""
    from workload import CONFIGS
    cfg = CONFIGS[name]
    free, _ = torch.cuda.mem_get_info()
    from workload import gen
    need = cfg.L * sum(int(np.prod(s)) for s in gen.weight_shapes(cfg).values()) * gen.ELEM_BYTES[cfg.dtype]
    if need > free * 0.9:
        pytest.skip(f"needs {need / 2**30:.1f} GiB of device memory")
    layers = [0, cfg.L - 1] if cfg.L > 1 else [0]
    wl_T = gen.make_workload(cfg).T
    tokens = sorted({0, wl_T // 2, wl_T - 1})
    layout = "tiled" if cfg.dtype in ("bf16", "e4m3") else "rowmajor"  # as the bench runs it
    wl, got, ref = run_step(mv, cfg, sample_tokens=tokens, sample_layers=layers, layout=layout)
    check_step(wl, got, ref, TOL[cfg.dtype], sample_tokens=tokens)


def test_step_in_a_cuda_graph(mv):
    """The whole step is capturable: replaying a CUDA graph of it gives the eager
    step's outputs bit for bit, also after new inputs are copied into the captured
    tensors."""
    from workload import CONFIGS, gen
    from workload import device as wdev
    cfg = CONFIGS["batched_qwen_like"].replace(L=2, H=512, I=256, use_bias=True, cap=8, alpha=0.25)
    wl = gen.make_workload(cfg)
    layers = [make_layer(mv, cfg, l, "tiled") for l in range(cfg.L)]
    t = wdev.workload_tensors(wl)
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=cfg.mode,
                       eps=cfg.eps, use_bias=True, cap=cfg.cap, alpha=cfg.alpha, layout="tiled")
    args = (t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    eager = mv.VerifyStep(spec, layers)
    y0 = eager(*args).clone()
    sel0 = eager.selected.clone()
    torch.cuda.synchronize()
    assert eager.dev_err.item() == 0
    step = mv.VerifyStep(spec, layers)
    g = step.capture(*args)
    step.y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    assert torch.equal(step.y, y0) and torch.equal(step.selected, sel0)
    # new inputs of the same shape: logits and hidden states of another seed
    wl2 = gen.make_workload(cfg.replace(seed=cfg.seed + 7))
    t2 = wdev.workload_tensors(wl2)
    for k_ in ("P", "own_fp", "logits", "x"):
        t[k_].copy_(t2[k_])
    g.replay()
    y_eager = eager(*args)
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0 and eager.dev_err.item() == 0
    assert torch.equal(step.y, y_eager) and torch.equal(step.selected, eager.selected)
    assert not torch.equal(y_eager, y0)


def test_step_with_nvtx_ranges(mv):
    """moe_set_nvtx(1) only adds host-side trace ranges: the step's and the
    plan's outputs are bit-identical to a run without them, and switching the
    ranges off again leaves the library in its default state."""
    from workload import CONFIGS, gen
    from workload import device as wdev
    cfg = CONFIGS["batched_qwen_like"].replace(L=2, H=512, I=256)
    wl = gen.make_workload(cfg)
    layers = [make_layer(mv, cfg, l, "tiled") for l in range(cfg.L)]
    t = wdev.workload_tensors(wl)
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=cfg.mode,
                       eps=cfg.eps, layout="tiled")
    args = (t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    step = mv.VerifyStep(spec, layers)
    plan = mv.VerifyPlan(spec)
    y0 = step(*args).clone()
    plan(*args[:5])
    ids0 = plan.ids.clone()
    try:
        mv.set_nvtx(True)
        y1 = step(*args).clone()
        plan(*args[:5])
        ids1 = plan.ids.clone()
    finally:
        mv.set_nvtx(False)
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0 and plan.dev_err.item() == 0
    assert torch.equal(y0, y1) and torch.equal(ids0, ids1)


def test_ffn_fuzz_shapes(mv):
    """Random FFN shapes, dtypes and layouts against the oracle: ragged tiles
    (H, I not multiples of 128), token groups of every size, all kernel paths."""
    from oracle import moe_layer as ml
    from workload import gen
    rng = np.random.default_rng(77)
    for trial in range(16):
        dtype = str(rng.choice(["bf16", "bf16", "e4m3", "f32"]))
        mult = 128 if dtype == "e4m3" else 64
        H = mult * int(rng.integers(1, 7))
        I = mult * int(rng.integers(1, 6))
        E = int(rng.choice([4, 9, 16, 33, 64]))
        k = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.choice([1, 2, 5, 13, 24, 40])) if dtype != "e4m3" else int(rng.choice([1, 3, 5, 17, 32, 40]))
        layout = "tiled" if dtype != "f32" and rng.integers(0, 2) else "rowmajor"
        if dtype == "e4m3" and T > 32:
            layout = "rowmajor"  # the CUDA-core FP8 path reads row-major weights
        cfg = gen.MoEConfig(f"ffnfuzz{trial}", L=1, H=H, E=E, k=k, I=I, dtype=dtype, seed=1000 + trial)
        layer = make_layer(mv, cfg, 0, layout)
        lg = (rng.standard_normal((T, E)) - 0.2 * rng.permutation(E)).astype(np.float32)
        xs = rng.standard_normal((T, H)).astype(np.float32)
        x_host = xs if dtype == "f32" else gen.bf16_bits_rne(xs)
        x_dev = cuda(xs) if dtype == "f32" else cuda(x_host.view(np.int16))
        dev_err = mv.new_dev_err()
        ids, w = mv.route(cuda(lg), k, dev_err=dev_err)
        up = mv.union_permute(ids, E, dev_err=dev_err)
        y = mv.verify_ffn(x_dev, k, layer, up, w, dev_err=dev_err)
        torch.cuda.synchronize()
        assert dev_err.item() == 0, (trial, dtype, H, I, E, k, T, layout)
        ref = ml.layer_forward(lg, x_decode(cfg)(x_host), k, E, host_experts(cfg, 0))
        yh = y.cpu().numpy().astype(np.float64)
        err = rowwise_err(yh, ref["y"])
        assert err < TOL[dtype], (trial, dtype, H, I, E, k, T, layout, err, elementwise_err(yh, ref["y"]))


@pytest.mark.parametrize("T", [5, 24, 40])
def test_ffn_group_order_checked(mv, T):
    """A union whose token group does not ascend (the union's layout) is
    flagged, not silently mis-scattered.  T <= 32 runs the token-dense
    gate/up, which places each token by its rank in the group; T = 40 runs
    the padded-group path, which reads the group in stored order and so
    needs no order (it must stay clean)."""
    from workload import gen
    H, I, E, k = 256, 192, 8, 4
    cfg = gen.MoEConfig("order", L=1, H=H, E=E, k=k, I=I, dtype="bf16", seed=3)
    layer = make_layer(mv, cfg, 0, "tiled")
    rng = np.random.default_rng(T)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    x_dev = cuda(gen.bf16_bits_rne(rng.standard_normal((T, H)).astype(np.float32)).view(np.int16))
    dev_err = mv.new_dev_err()
    ids, w = mv.route(cuda(lg), k, dev_err=dev_err)
    up = mv.union_permute(ids, E, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    off = up["offsets"].cpu().numpy()
    U = int(up["n_unique"].item())
    g = next(u for u in range(U) if off[u + 1] - off[u] >= 2)
    pt = up["perm_token"].clone()
    a, b = int(off[g]), int(off[g]) + 1
    pt[a], pt[b] = up["perm_token"][b].item(), up["perm_token"][a].item()
    inv = up["inv"].clone()
    for p in (a, b):  # keep inv consistent with the swapped positions
        t = int(pt[p].item())
        for j in range(k):
            if int(ids[t, j].item()) == int(up["unique"][g].item()):
                inv[t * k + j] = p
    bad = dict(up, perm_token=pt, inv=inv)
    mv.verify_ffn(x_dev, k, layer, bad, w, dev_err=dev_err)
    torch.cuda.synchronize()
    if T <= 32:
        assert dev_err.item() & mv._lib.DEV_BAD_ID
    else:
        assert dev_err.item() == 0


@pytest.mark.parametrize("name", ["qwen3_235b_like", "gpt_oss_120b_like", "batched_qwen_like"])
def test_step_union_handshake_fallback(mv, name):
    """bf16 layers with T <= 32 hand each layer's union from the head kernel
    to the gate/up kernel through a release/acquire word, so gate/up can read
    it before its dependency wait.  With the test hook the heads never
    publish: every gate/up waits out its bounded handshake (100 us) and reads
    the union after its dependency wait.  The step must give the same
    outputs bit for bit, with no error flagged."""
    from workload import CONFIGS, gen
    from workload import device as wdev
    cfg = CONFIGS[name].replace(**SMALL[name])
    wl = gen.make_workload(cfg)
    layers = [make_layer(mv, cfg, l, "tiled") for l in range(cfg.L)]
    t = wdev.workload_tensors(wl)
    spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                       I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=cfg.mode,
                       eps=cfg.eps, use_bias=cfg.use_bias, cap=cfg.cap, alpha=cfg.alpha, layout="tiled")
    args = (t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    step = mv.VerifyStep(spec, layers)
    y0 = step(*args).clone()
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    L = mv._lib
    lib = L.load()
    assert lib.moe_test_set_stall(L.TEST_STALL_READY_FLAG) == L.MOE_OK
    try:
        y1 = step(*args).clone()
        torch.cuda.synchronize()
    finally:
        lib.moe_test_set_stall(0)
    assert step.dev_err.item() == 0
    assert torch.equal(y0, y1)
    y2 = step(*args)
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0 and torch.equal(y0, y2)

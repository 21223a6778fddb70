"""moe_depth_policy against the oracle (width-vs-depth note, section 2): the
depth vector, the common depth and both throughputs must be bit-exact; and
the width-vs-depth unions (section 1) of the plan on chain workloads equal
the oracle's."""
import numpy as np
import pytest

from oracle import width_depth as wd

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import serving_router_softmax_gb300 as m
    return m


def run(mv, conf, fp, C0, T_exp, max_depth=None):
    dev_err = mv.new_dev_err()
    md = None if max_depth is None else torch.tensor(max_depth, dtype=torch.int32, device="cuda")
    d, common, thr = mv.depth_policy(torch.from_numpy(conf).cuda(),
                                     torch.from_numpy(fp.view(np.int32)).cuda(), C0, T_exp,
                                     max_depth=md, dev_err=dev_err)
    torch.cuda.synchronize()
    return d.cpu().tolist(), int(common.item()), thr.cpu().tolist(), int(dev_err.item())


def check(mv, conf, fp, C0, T_exp, max_depth=None):
    d, common, thr, err = run(mv, conf, fp, C0, T_exp, max_depth)
    ref = wd.depth_policy(conf, fp, C0, T_exp, max_depth)
    assert err == 0
    assert d == ref["depth"] and common == ref["common"]
    assert thr == [ref["thr_common"], ref["thr"]]  # bit-exact fp64
    return ref


def test_hand_batch(mv):
    conf = np.array([[0.875, 0.75], [0.125, 0.0625]], np.float32)
    fp = np.zeros((2, 3, 1), np.uint32)
    for i, row in enumerate([[{0}, {0}, {1}], [{2}, {3, 4}, {5, 6}]]):
        for j, bits in enumerate(row):
            for b in bits:
                fp[i, j, 0] |= np.uint32(1 << b)
    ref = check(mv, conf, fp, 8.0, 1.0)
    assert ref["depth"] == [2, 0]
    check(mv, conf, fp, 8.0, 1.0, max_depth=[1, 2])


def rand_case(rng, nseq, D, W, density):
    q = rng.uniform(0.0, 1.0, size=(nseq, D))
    if rng.random() < 0.3:
        q[rng.random(nseq) < 0.5] = 0.0  # hopeless drafts
    conf = np.cumprod(q, axis=1).astype(np.float32)
    fp = np.zeros((nseq, D + 1, W), np.uint32)
    mask = rng.random((nseq, D + 1, W, 32)) < density
    for b in range(32):
        fp |= (mask[..., b].astype(np.uint32) << np.uint32(b))
    if rng.random() < 0.3:
        fp[1:] = fp[:1]  # identical footprints across sequences (many equal unions)
    return conf, fp


CASES = [(1, 6, 1), (2, 2, 1), (4, 6, 64), (4, 6, 96), (8, 8, 64), (16, 4, 8), (3, 32, 2), (64, 6, 16),
         (256, 3, 2), (5, 1, 7), (7, 12, 33)]


@pytest.mark.parametrize("nseq,D,W", CASES)
@pytest.mark.parametrize("seed", range(3))
def test_matches_oracle_random(mv, nseq, D, W, seed):
    rng = np.random.default_rng(1000 * seed + nseq * 37 + D * 5 + W)
    conf, fp = rand_case(rng, nseq, D, W, density=float(rng.choice([0.01, 0.05, 0.2])))
    C0 = float(np.float32(rng.uniform(0.5, 50.0)))
    T_exp = float(np.float32(rng.choice([0.0, rng.uniform(0.01, 3.0)])))
    lim = None if seed == 0 else rng.integers(-1, D + 2, size=nseq).tolist()
    check(mv, conf, fp, C0, T_exp, lim)


def test_chain_workload(mv):
    from workload import CONFIGS, gen
    for nseq in (1, 4, 8):
        cfg = gen.chain_config(CONFIGS["qwen3_235b_like"], nseq)
        wl = gen.make_workload(cfg)
        fp = np.concatenate([wl.root_fp[:, None, :], wl.own_fp], axis=1)
        for C0, T_exp in ((1000.0, 6.0), (300.0, 6.0), (1000.0, 0.5)):
            check(mv, wl.P.copy(), fp, C0, T_exp)


def test_bad_confidence_flags_and_verifies_nothing(mv):
    conf = np.array([[0.5, 1.5], [0.25, 0.125]], np.float32)
    fp = np.ones((2, 3, 1), np.uint32)
    d, common, _, err = run(mv, conf, fp, 4.0, 1.0)
    assert err & mv._lib.DEV_BAD_PROB and d == [0, 0] and common == 0
    conf[0, 1] = np.nan
    d, _, _, err = run(mv, conf, fp, 4.0, 1.0)
    assert err & mv._lib.DEV_BAD_PROB and d == [0, 0]


def test_host_validation(mv):
    conf = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    fp = torch.zeros((2, 3, 1), dtype=torch.int32, device="cuda")
    for C0, T_exp in ((0.0, 1.0), (1.0, -1.0), (float("inf"), 1.0)):
        with pytest.raises(mv.MoEError):
            mv.depth_policy(conf, fp, C0, T_exp)
    with pytest.raises(mv.MoEError):  # D = 33 > 32
        mv.depth_policy(torch.zeros((1, 33), dtype=torch.float32, device="cuda"),
                        torch.zeros((1, 34, 1), dtype=torch.int32, device="cuda"), 1.0, 1.0)


@pytest.mark.parametrize("d", [2, 4, 7])
def test_width_and_depth_unions_match_oracle(mv, d):
    """Section 1: d consecutive positions of one sequence (root + d-1 chain
    drafts) against the roots of d independent sequences; the plan's per-layer
    unions equal the oracle's top-k unions of the same rows."""
    from workload import CONFIGS, gen
    from workload import device as wdev
    base = CONFIGS["qwen3_235b_like"]
    for kind in ("depth", "width"):
        if kind == "depth":
            cfg = gen.chain_config(base, 1, depth=6, seed=200 + d, gamma=d - 1)
        else:
            cfg = gen.chain_config(base, d, depth=6, seed=300 + d, gamma=0)
        wl = gen.make_workload(cfg)
        t = wdev.workload_tensors(wl)
        spec = mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k, H=cfg.H,
                           I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=0, eps=cfg.eps,
                           use_bias=False, cap=0, alpha=0.0)
        plan = mv.VerifyPlan(spec)
        plan(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"])
        torch.cuda.synchronize()
        assert plan.dev_err.item() == 0
        if kind == "depth":
            rows = list(range(d))  # root, then chain positions 1..d-1
            lg = wl.logits[:, 0, rows, :]
        else:
            lg = wl.logits[:, :, 0, :]
        assert plan.n_unique.cpu().tolist() == wd.layer_unions(lg, cfg.k)

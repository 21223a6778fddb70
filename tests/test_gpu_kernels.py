"""GPU parity of each C-ABI call against the CPU oracle (same seeded inputs)."""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def mv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import serving_router_softmax_gb300 as m
    return m


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ------------------------------------------------------------------ routing
ROUTE_CASES = [(1, 16, 2), (5, 16, 2), (5, 128, 8), (28, 128, 8), (5, 256, 8), (7, 1000, 16),
               (100, 64, 4), (3, 8, 8), (33, 33, 1), (256, 128, 8)]


@pytest.mark.parametrize("T,E,k", ROUTE_CASES)
def test_route_matches_oracle(mv, T, E, k):
    from oracle import moe_layer as ml
    rng = np.random.default_rng(T * 1000 + E + k)
    lg = (rng.standard_normal((T, E)) - 0.02 * rng.permutation(E)).astype(np.float32)
    if T > 1:
        lg[1, : E // 2] = lg[1, E // 2: 2 * (E // 2)]  # exact ties
        lg[0, 0] = -0.0
        lg[0, 1] = 0.0
    dev_err = mv.new_dev_err()
    ids, w = mv.route(cuda(lg), k, dev_err=dev_err)
    torch.cuda.synchronize()
    rid, rw = ml.route(lg, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)
    assert dev_err.item() == 0


def test_route_empty_and_nan(mv):
    ids, w = mv.route(torch.zeros((0, 16), dtype=torch.float32, device="cuda"), 2)
    assert ids.shape == (0, 2)
    lg = np.zeros((3, 16), dtype=np.float32)
    lg[1, 5] = np.nan
    dev_err = mv.new_dev_err()
    ids, w = mv.route(cuda(lg), 2, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() & 0x01
    assert ids[1].tolist() == [-1, -1] and w[1].tolist() == [0.0, 0.0]
    assert ids[0].tolist() == [0, 1]


@pytest.mark.parametrize("name", ["reuse_bias_fig5.json", "reuse_bias_weighting.json"])
def test_route_bias_golden(mv, name):
    from oracle import moe_layer as ml
    g = json.load(open(os.path.join(GOLD, name)))
    lg = np.array(g["logits"], dtype=np.float32)
    wc = np.array(g["w_conf"], dtype=np.float32)
    ids, w = mv.route(cuda(lg), g["k"], w_conf=cuda(wc), cap=g["cap"], alpha=g["alpha"])
    rid, rw = ml.route(ml.reuse_bias(lg, wc, g["k"], g["cap"], g["alpha"]), g["k"])
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)
    if "ids_after" in g["expected"]:
        assert ids.cpu().tolist() == g["expected"]["ids_after"]


@pytest.mark.parametrize("T,E,k,cap,alpha", [(5, 128, 4, 8, 0.25), (5, 128, 4, 8, 1.0),
                                             (20, 128, 8, 16, 0.5), (28, 256, 8, 12, 0.1),
                                             (3, 9, 8, 8, 2.0), (64, 64, 2, 3, 4.0),
                                             (256, 32, 4, 8, 0.25)])
def test_route_bias_matches_oracle(mv, T, E, k, cap, alpha):
    from oracle import moe_layer as ml
    rng = np.random.default_rng(T + E * 7 + k)
    lg = (rng.standard_normal((T, E)) - 0.07 * rng.permutation(E)).astype(np.float32)
    wc = rng.uniform(0, 1, T).astype(np.float32)
    wc[0] = 1.0
    ids, w = mv.route(cuda(lg), k, w_conf=cuda(wc), cap=cap, alpha=alpha)
    rid, rw = ml.route(ml.reuse_bias(lg, wc, k, cap, alpha), k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)


def crowded_rows(rng, T, E, k):
    """Rows that load the top-k's warp layout (expert e sits in lane e mod 32)
    unevenly.  Kind 0: the winners crowd into k + 1 lanes, each of which holds
    only winners, in an order that interleaves the lanes' values; kind 1: one
    value everywhere (the lower id decides every slot); kind 2: values on a
    coarse grid (many ties); kind 3: plain normal rows."""
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lanes = min(32, E)
    K = min(k + 1, lanes)
    for t in range(T):
        kind = t % 4
        if kind == 0:
            npl = -(-E // 32)
            for r, lane in enumerate(rng.choice(lanes, size=K, replace=False)):
                ex = np.arange(lane, E, 32)
                lg[t, ex] = 10.0 + r * npl + np.arange(len(ex))
        elif kind == 1:
            lg[t] = 0.5
        elif kind == 2:
            lg[t] = np.round(lg[t] * 2.0) / 2.0
    return lg


@pytest.mark.parametrize("T,E,k", [(8, 128, 8), (8, 128, 16), (8, 256, 8), (8, 300, 16), (8, 1024, 16),
                                   (8, 40, 4), (8, 17, 16)])
def test_route_crowded_and_tied_rows(mv, T, E, k):
    from oracle import moe_layer as ml
    lg = crowded_rows(np.random.default_rng(E * 31 + k), T, E, k)
    dev_err = mv.new_dev_err()
    ids, w = mv.route(cuda(lg), k, dev_err=dev_err)
    torch.cuda.synchronize()
    rid, rw = ml.route(lg, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)
    assert dev_err.item() == 0


@pytest.mark.parametrize("T,E,k,cap", [(8, 128, 16, 8), (8, 256, 8, 12), (9, 1024, 16, 12), (8, 20, 16, 3)])
def test_route_bias_crowded_and_tied_rows(mv, T, E, k, cap):
    from oracle import moe_layer as ml
    rng = np.random.default_rng(E * 17 + k)
    lg = crowded_rows(rng, T, E, k)
    wc = rng.uniform(0, 1, T).astype(np.float32)
    ids, w = mv.route(cuda(lg), k, w_conf=cuda(wc), cap=cap, alpha=0.5)
    rid, rw = ml.route(ml.reuse_bias(lg, wc, k, cap, 0.5), k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)


# ------------------------------------------------------------------ union
@pytest.mark.parametrize("T,E,k", [(1, 16, 2), (5, 128, 8), (20, 128, 8), (28, 256, 8),
                                   (256, 1024, 16), (7, 8, 8), (4096, 16, 2)])
def test_union_matches_oracle(mv, T, E, k):
    from oracle import moe_layer as ml
    rng = np.random.default_rng(T * 3 + E)
    pop = np.exp(-0.05 * np.arange(E))
    pop /= pop.sum()
    ids = np.stack([rng.choice(E, size=k, replace=False, p=pop) for _ in range(T)]).astype(np.int32)
    up = mv.union_permute(cuda(ids), E)
    torch.cuda.synchronize()
    ref = ml.union_permute(ids, E)
    U = int(up["n_unique"].item())
    assert U == ref["n_unique"]
    assert np.array_equal(up["unique"][:U].cpu().numpy(), ref["unique"])
    assert np.array_equal(up["offsets"][: U + 1].cpu().numpy(), ref["offsets"])
    for key in ("perm_token", "perm_slot", "inv"):
        assert np.array_equal(up[key][: T * k].cpu().numpy(), ref[key]), key
    assert up["reuse_ratio"].cpu().numpy()[0] == ref["reuse_ratio"]


def test_union_errors(mv):
    dev_err = mv.new_dev_err()
    up = mv.union_permute(cuda(np.array([[1, 1], [0, 2]], np.int32)), 4, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() & 0x04 and up["n_unique"].item() == 0
    dev_err = mv.new_dev_err()
    up = mv.union_permute(cuda(np.array([[1, 7]], np.int32)), 4, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() & 0x02 and up["n_unique"].item() == 0
    up = mv.union_permute(torch.zeros((0, 2), dtype=torch.int32, device="cuda"), 4)
    torch.cuda.synchronize()
    assert up["n_unique"].item() == 0 and up["reuse_ratio"].item() == 0.0


# ------------------------------------------------------------------ selection
def _bits(own_lists, L, E):
    W = (L * E + 31) // 32
    out = np.zeros((len(own_lists), W), dtype=np.uint32)
    for t, pairs in enumerate(own_lists):
        for l, e in pairs:
            b = l * E + e
            out[t, b // 32] |= np.uint32(1 << (b % 32))
    return out


def test_eco_golden_trees(mv):
    g = json.load(open(os.path.join(GOLD, "ecospec_trees.json")))
    for tree in g["trees"]:
        fp = _bits(tree["own"], tree["L"], tree["E"])[None]
        P = np.array([tree["P"]], dtype=np.float32)
        par = np.array([tree["parent"]], dtype=np.int32)
        for ex in tree["expect"]:
            sel, usz = mv.eco_select(cuda(P), cuda(par), cuda(fp.view(np.int32)), ex["gamma"],
                                     eps=g["eps"], mode=ex["mode"])
            got = [v for v in sel[0].cpu().tolist() if v >= 0]
            assert got == ex["selected"], (tree["name"], ex)
            assert usz.item() == ex["union"]


def test_eco_rounded_scores_tie_but_exact_scores_do_not(mv):
    """The selection kernel compares scores P / (c + eps) through the correctly
    rounded fp32 quotient P / X, X = c * 2^s + 1 (eps = 2^-s), and falls back to
    the exact comparison only on equal quotients.  With eps = 1/2: node 0 has
    P = 1 and one new expert (X = 3), node 1 has P = fl32(1/3) > 1/3 and none
    (X = 1).  Both quotients round to fl32(1/3), but exactly
    P_1 * X_0 = 3 * fl32(1/3) > 1 = P_0 * X_1, so node 1 wins, not the lower
    index."""
    from oracle import eco_select as oeco
    p1 = float(np.float32(1.0 / 3.0))
    P = np.array([[1.0, p1]], dtype=np.float32)
    par = np.array([[-1, -1]], dtype=np.int32)
    fp = _bits([[(0, 3)], []], 1, 16)[None]
    # the quotients the kernel's key uses round to the same value
    assert np.float32(np.float32(1.0) / np.float32(3.0)) == np.float32(np.float32(p1) / np.float32(1.0))
    sel, usz = mv.eco_select(cuda(P), cuda(par), cuda(fp.view(np.int32)), 1, eps=0.5)
    torch.cuda.synchronize()
    rsel, _ = oeco.select_batch(P, np.array([-1, -1]), fp, 16, np.array([1]), 0.5, 0)
    assert rsel[0] == [1]
    assert sel[0].cpu().tolist() == [1] and usz.item() == 0


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("cfgname", ["toy", "qwen3_235b_like", "deepseek_v3_like", "batched_qwen_like"])
def test_eco_matches_oracle_on_workload_trees(mv, mode, cfgname):
    from oracle import eco_select as oeco
    from workload import CONFIGS, make_workload
    cfg = CONFIGS[cfgname].replace(mode=mode)
    for seed in range(3):
        wl = make_workload(cfg.replace(seed=100 + seed, L=min(cfg.L, 4)))
        nseq, N = wl.P.shape
        gmax = int(wl.gamma.max())
        par = np.tile(wl.parent, (nseq, 1)).astype(np.int32)
        sel, usz = mv.eco_select(cuda(wl.P), cuda(par), cuda(wl.own_fp.view(np.int32)), gmax,
                                 gamma_per_seq=cuda(wl.gamma), eps=cfg.eps, mode=mode)
        rsel, rsz = oeco.select_batch(wl.P, wl.parent, wl.own_fp, cfg.E, wl.gamma, cfg.eps, mode)
        s_np = sel.cpu().numpy()
        for s in range(nseq):
            assert s_np[s, : wl.gamma[s]].tolist() == rsel[s]
            assert np.all(s_np[s, wl.gamma[s]:] == -1)
        assert usz.cpu().tolist() == rsz


def test_eco_random_large_trees(mv):
    """Deeper/wider trees than the workloads (N up to 1022, W up to 256)."""
    from oracle import eco_select as oeco
    rng = np.random.default_rng(9)
    for N, W, gamma in [(30, 4, 8), (126, 64, 20), (1022, 32, 40), (150, 256, 5)]:
        nseq = 2
        par = np.zeros((nseq, N), dtype=np.int32)
        P = np.zeros((nseq, N), dtype=np.float32)
        fp = rng.integers(0, 2 ** 32, size=(nseq, N, W), dtype=np.uint64).astype(np.uint32)
        fp &= rng.integers(0, 2 ** 32, size=(nseq, N, W), dtype=np.uint64).astype(np.uint32)
        fp &= rng.integers(0, 2 ** 32, size=(nseq, N, W), dtype=np.uint64).astype(np.uint32)
        for s in range(nseq):
            for t in range(N):
                par[s, t] = -1 if t < 2 else int(rng.integers(0, t))
                base = np.float32(1) if par[s, t] < 0 else P[s, par[s, t]]
                P[s, t] = np.float32(base * np.float32(rng.uniform(0.05, 1.0)))
        E = 32 * W  # one layer
        gam = np.array([gamma, gamma // 2], dtype=np.int32)
        for mode in (0, 1):
            sel, usz = mv.eco_select(cuda(P), cuda(par), cuda(fp.view(np.int32)), gamma,
                                     gamma_per_seq=cuda(gam), eps=2.0 ** -10, mode=mode)
            for s in range(nseq):
                rsel, rsz = oeco.select_batch(P[s:s + 1], par[s], fp[s:s + 1], E, [gam[s]],
                                              2.0 ** -10, mode)
                assert sel[s, : gam[s]].cpu().tolist() == rsel[0]
                assert usz[s].item() == rsz[0]


def test_eco_bad_tree_flags(mv):
    P = np.array([[0.5, 0.4, 0.3]], dtype=np.float32)
    par = np.array([[-1, 2, 0]], dtype=np.int32)  # parent not before child
    fp = np.ones((1, 3, 1), dtype=np.int32)
    dev_err = mv.new_dev_err()
    sel, usz = mv.eco_select(cuda(P), cuda(par), cuda(fp), 2, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() & 0x08 and sel.cpu().tolist() == [[-1, -1]] and usz.item() == 0
    P[0, 1] = np.nan
    par[0, 1] = 0
    dev_err = mv.new_dev_err()
    mv.eco_select(cuda(P), cuda(par), cuda(fp), 2, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() & 0x10


@pytest.mark.parametrize("cfgname", ["qwen3_235b_like", "batched_qwen_like", "deepseek_v3_like"])
def test_eco_batch_global_matches_oracle(mv, cfgname):
    from oracle import eco_select as oeco
    from workload import CONFIGS, make_workload
    rng = np.random.default_rng(11)
    for seed in range(3):
        cfg = CONFIGS[cfgname].replace(seed=200 + seed, L=min(CONFIGS[cfgname].L, 4))
        wl = make_workload(cfg)
        nseq, N = wl.P.shape
        for cap in [int(wl.gamma.max()), N]:
            gam = wl.gamma.copy()
            par = np.tile(wl.parent, (nseq, 1)).astype(np.int32)
            sel, usz = mv.eco_select(cuda(wl.P), cuda(par), cuda(wl.own_fp.view(np.int32)), cap,
                                     gamma_per_seq=cuda(gam), eps=cfg.eps, mode=2)
            rsel, rsz, _ = oeco.select_batch_global(wl.P, wl.parent, wl.own_fp, cfg.E, gam, cfg.eps, cap)
            s_np = sel.cpu().numpy()
            for s in range(nseq):
                assert s_np[s, : len(rsel[s])].tolist() == rsel[s]
                assert np.all(s_np[s, len(rsel[s]):] == -1)
            assert usz.cpu().tolist() == rsz


def test_eco_batch_global_random_forests(mv):
    from oracle import eco_select as oeco
    rng = np.random.default_rng(12)
    for nseq, N, W, cap in [(4, 14, 8, 6), (8, 30, 4, 10), (16, 60, 2, 20), (2, 500, 16, 40)]:
        parent = np.array([-1 if t < 2 else int(rng.integers(0, t)) for t in range(N)], dtype=np.int32)
        P = np.zeros((nseq, N), dtype=np.float32)
        for s in range(nseq):
            for t in range(N):
                base = np.float32(1) if parent[t] < 0 else P[s, parent[t]]
                P[s, t] = np.float32(base * np.float32(rng.uniform(0.05, 1.0)))
        fp = rng.integers(0, 2 ** 32, size=(nseq, N, W), dtype=np.uint64).astype(np.uint32)
        fp &= rng.integers(0, 2 ** 32, size=(nseq, N, W), dtype=np.uint64).astype(np.uint32)
        gam = rng.integers(0, cap + 1, size=nseq).astype(np.int32)
        par = np.tile(parent, (nseq, 1)).astype(np.int32)
        sel, usz = mv.eco_select(cuda(P), cuda(par), cuda(fp.view(np.int32)), cap, gamma_per_seq=cuda(gam),
                                 eps=2.0 ** -10, mode=2)
        rsel, rsz, _ = oeco.select_batch_global(P, parent, fp, 32 * W, gam, 2.0 ** -10, cap)
        s_np = sel.cpu().numpy()
        for s in range(nseq):
            assert s_np[s, : len(rsel[s])].tolist() == rsel[s]
        assert usz.cpu().tolist() == rsz


def test_eco_batch_global_hand_example(mv):
    # the oracle pin's batch: the greedy gives sequence A nothing and B two nodes
    E = 16
    parent = np.array([[-1, 0], [-1, 0]], dtype=np.int32)
    P = np.array([[0.9, 0.8], [0.6, 0.5]], dtype=np.float32)
    fp = np.zeros((2, 2, 1), dtype=np.uint32)
    for t, bits in enumerate([[1, 2, 3], [4, 5]]):
        for b in bits:
            fp[0, t, 0] |= np.uint32(1 << b)
    fp[1, 0, 0] = np.uint32(1 << 6)
    fp[1, 1, 0] = np.uint32(1 << 7)
    sel, usz = mv.eco_select(cuda(P), cuda(parent), cuda(fp.view(np.int32)), 2,
                             gamma_per_seq=cuda(np.array([1, 1], dtype=np.int32)), eps=2.0 ** -10, mode=2)
    assert sel.cpu().tolist() == [[-1, -1], [0, 1]] and usz.cpu().tolist() == [0, 2]

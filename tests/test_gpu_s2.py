"""GPU parity of s2_expand (S2-MoE utility expansion) against the oracle."""
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


def run(mv, P, parent, own_fp, T_AR, T_exp, C, dev_err=None, T_cold=0.0, cold_bits=None):
    Pt = torch.from_numpy(np.ascontiguousarray(P, dtype=np.float32)).cuda()
    par = torch.from_numpy(np.ascontiguousarray(np.tile(parent, (P.shape[0], 1)), dtype=np.int32)).cuda()
    fp = torch.from_numpy(np.ascontiguousarray(own_fp).view(np.int32)).cuda()
    cold = None
    if cold_bits is not None:
        cold = torch.from_numpy(np.ascontiguousarray(cold_bits, dtype=np.uint32).view(np.int32)).cuda()
    sel, n, u = mv.s2_expand(Pt, par, fp, T_AR, T_exp, C, dev_err=dev_err, T_cold=T_cold, cold_fp=cold)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), n.cpu().tolist(), u.cpu().tolist()


def check(mv, P, parent, own_fp, E, T_AR, T_exp, C, T_cold=0.0, cold_bits=None):
    from oracle import s2_expand as s2
    from oracle.eco_select import footprint_set
    sel, n, u = run(mv, P, parent, own_fp, T_AR, T_exp, C, T_cold=T_cold, cold_bits=cold_bits)
    cold = None if cold_bits is None else footprint_set(cold_bits, E)
    want, sizes = s2.s2_expand_batch(P, parent, own_fp, E, T_AR, T_exp, C, T_cold, cold)
    for s in range(P.shape[0]):
        assert n[s] == len(want[s])
        assert sel[s, : n[s]].tolist() == want[s]
        assert (sel[s, n[s]:] == -1).all()
    assert u == sizes


@pytest.mark.parametrize("name", ["toy", "qwen3_235b_like", "gpt_oss_120b_like", "deepseek_v3_like",
                                  "batched_qwen_like"])
def test_s2_workload_trees(mv, name):
    from workload import CONFIGS, gen
    cfg = CONFIGS[name]
    wl = gen.make_workload(cfg)
    rng = np.random.default_rng(len(name))
    T_exp = 1.0
    for T_AR in [float(cfg.L * cfg.k), 16.0, 400.0]:
        for C in [0.0, 0.5, 3.0]:
            check(mv, wl.P, wl.parent, wl.own_fp, cfg.E, T_AR, T_exp, C)
    for _ in range(6):
        check(mv, wl.P, wl.parent, wl.own_fp, cfg.E, float(rng.uniform(1, 500)), float(rng.uniform(0, 4)),
              float(rng.uniform(0, 4)))
    # zero cost (every node), zero gain (nothing unless free)
    check(mv, wl.P, wl.parent, wl.own_fp, cfg.E, 1.0, 0.0, 0.0)
    check(mv, wl.P, wl.parent, wl.own_fp, cfg.E, 0.0, 1.0, 0.5)


def test_s2_hand_example(mv):
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "s2_expand_hand.json")))
    fp = np.zeros((1, len(g["own"]), 1), dtype=np.uint32)
    for t, s in enumerate(g["own"]):
        for b in s:
            fp[0, t, 0] |= np.uint32(1 << b)
    P = np.array([g["P"]], dtype=np.float32)
    sel, n, u = run(mv, P, np.array(g["parent"]), fp, g["T_AR"], g["T_exp"], g["C_draft"])
    assert sel[0, : n[0]].tolist() == g["selected"] and u[0] == g["union_size"]
    c2 = g["second_case"]
    sel, n, u = run(mv, P, np.array(g["parent"]), fp, g["T_AR"], c2["T_exp"], c2["C_draft"])
    assert sel[0, : n[0]].tolist() == c2["selected"] and u[0] == c2["union_size"]


def test_s2_large_random_tree(mv):
    # N = 1024 nodes (the maximum), W = 40 words, random parents and footprints
    rng = np.random.default_rng(3)
    N, W, E = 1024, 40, 64
    parent = np.array([-1] + [int(rng.integers(-1, t)) for t in range(1, N)], dtype=np.int32)
    P = np.zeros((2, N), dtype=np.float32)
    for s in range(2):
        for t in range(N):
            q = np.float32(rng.uniform(0.3, 1.0))
            P[s, t] = q if parent[t] < 0 else np.float32(P[s, parent[t]] * q)
    own = rng.integers(0, 2 ** 32, size=(2, N, W), dtype=np.uint64).astype(np.uint32)
    for _ in range(5):  # about 20 of the 1280 bits per node
        own &= rng.integers(0, 2 ** 32, size=(2, N, W), dtype=np.uint64).astype(np.uint32)
    check(mv, P, parent, own, E, 100.0, 1.0, 0.25)
    check(mv, P, parent, own, E, 25.0, 1.0, 0.1)
    check(mv, P, parent, own, E, 3000.0, 2.0, 0.0)


def test_s2_errors(mv):
    from serving_router_softmax_gb300 import _lib as L
    P = np.array([[0.5, np.nan, 0.2]], dtype=np.float32)
    fp = np.zeros((1, 3, 1), dtype=np.uint32)
    dev_err = mv.new_dev_err()
    sel, n, u = run(mv, P, np.array([-1, 0, 0]), fp, 1.0, 1.0, 0.0, dev_err=dev_err)
    assert dev_err.item() & L.DEV_BAD_PROB and n == [0] and (sel == -1).all()
    dev_err = mv.new_dev_err()
    sel, n, u = run(mv, np.array([[0.5, 0.4, 0.2]], dtype=np.float32), np.array([-1, 2, 0]), fp, 1.0, 1.0, 0.0,
                    dev_err=dev_err)
    assert dev_err.item() & L.DEV_BAD_TREE and n == [0]
    with pytest.raises(mv.MoEError):
        run(mv, np.array([[0.5]], dtype=np.float32), np.array([-1]), np.zeros((1, 1, 1), np.uint32), -1.0, 1.0, 0.0)
    with pytest.raises(mv.MoEError):
        run(mv, np.array([[0.5]], dtype=np.float32), np.array([-1]), np.zeros((1, 1, 1), np.uint32), 1.0,
            float("inf"), 0.0)


def test_s2_hand_example_cold(mv):
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "s2_expand_hand.json")))
    fp = np.zeros((1, len(g["own"]), 1), dtype=np.uint32)
    for t, s in enumerate(g["own"]):
        for b in s:
            fp[0, t, 0] |= np.uint32(1 << b)
    P = np.array([g["P"]], dtype=np.float32)
    cc, c2 = g["cold_cases"], g["second_case"]
    cold = np.zeros(1, dtype=np.uint32)
    for b in cc["cold"]:
        cold[0] |= np.uint32(1 << b)
    for case in cc["cases"]:
        sel, n, u = run(mv, P, np.array(g["parent"]), fp, g["T_AR"], c2["T_exp"], c2["C_draft"],
                        T_cold=case["T_cold"], cold_bits=cold)
        assert sel[0, : n[0]].tolist() == case["selected"] and u[0] == case["union_size"]


@pytest.mark.parametrize("name", ["qwen3_235b_like", "deepseek_v3_like", "batched_qwen_like"])
def test_s2_workload_trees_with_cold_experts(mv, name):
    """Residency-aware expansion: a hot list per layer (the most frequent experts of the
    workload's own footprints), every other expert cold at a surcharge T_cold."""
    from workload import CONFIGS, gen
    cfg = CONFIGS[name]
    wl = gen.make_workload(cfg)
    rng = np.random.default_rng(11 + len(name))
    for frac in (0.0, 0.25, 0.5, 0.9):
        cold = (rng.random(cfg.L * cfg.E) >= frac)
        bits = np.zeros(cfg.W, dtype=np.uint32)
        for b in np.nonzero(cold)[0]:
            bits[b // 32] |= np.uint32(1 << (b % 32))
        for T_AR, T_exp, C, T_cold in [(200.0, 1.0, 0.5, 30.0), (2000.0, 1.0, 0.0, 30.0),
                                       (float(rng.uniform(10, 5000)), float(rng.uniform(0, 4)),
                                        float(rng.uniform(0, 4)), float(rng.uniform(0, 100)))]:
            check(mv, wl.P, wl.parent, wl.own_fp, cfg.E, T_AR, T_exp, C, T_cold=T_cold, cold_bits=bits)

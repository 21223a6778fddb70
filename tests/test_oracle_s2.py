"""Pins for the S2-MoE utility-expansion oracle."""
import json
import os

import numpy as np
import pytest

from oracle import s2_expand as s2

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bits_of(sets, W, E=None):
    out = np.zeros((len(sets), W), dtype=np.uint32)
    for t, s in enumerate(sets):
        for b in s:
            out[t, b // 32] |= np.uint32(1 << (b % 32))
    return out


def test_hand_example():
    g = json.load(open(os.path.join(GOLD, "s2_expand_hand.json")))
    fp = bits_of(g["own"], 1)
    sel, size = s2.s2_expand(g["P"], g["parent"], fp, g["E"], g["T_AR"], g["T_exp"], g["C_draft"])
    assert sel == g["selected"] and size == g["union_size"]
    c2 = g["second_case"]
    sel, size = s2.s2_expand(g["P"], g["parent"], fp, g["E"], g["T_AR"], c2["T_exp"], c2["C_draft"])
    assert sel == c2["selected"] and size == c2["union_size"]


def test_later_pass_takes_a_node_made_cheap_by_a_later_one():
    # node 1 is too expensive in the first pass; node 2 (later in draft order)
    # brings its experts, so the second pass takes node 1 at the draft cost only
    P = [0.5, 0.2, 0.5]
    parent = [-1, -1, 0]
    fp = bits_of([{0}, {1, 2}, {1, 2}], 1)
    sel, size = s2.s2_expand(P, parent, fp, 8, 1.0, 0.125, 0.0625)
    assert sel == [0, 1, 2] and size == 3


def jacobi(P, parent, own, T_AR, T_exp, C):
    """Simultaneous-update iteration: all candidates against the same union."""
    N = len(parent)
    gain = [float(np.float64(np.float32(P[t])) * np.float64(np.float32(T_AR))) for t in range(N)]
    chosen = [False] * N
    B = set()
    while True:
        take = []
        for i in range(N):
            if chosen[i] or (parent[i] >= 0 and not chosen[parent[i]]):
                continue
            cost = np.float64(len(own[i] - B)) * np.float64(np.float32(T_exp)) + np.float64(np.float32(C))
            if gain[i] >= cost:
                take.append(i)
        if not take:
            return [t for t in range(N) if chosen[t]], len(B)
        for i in take:
            chosen[i] = True
            B |= own[i]


def random_trees(n, seed):
    from workload import gen
    cfg = gen.small_case("s2_pins", L=2, E=16, k=4, seed=seed)
    wl = gen.make_workload(cfg)
    return cfg, wl


@pytest.mark.parametrize("seed", range(6))
def test_order_independent_prefix_closed_and_union(seed):
    cfg, wl = random_trees(1, seed)
    from oracle.eco_select import footprint_set
    rng = np.random.default_rng(seed)
    for _ in range(20):
        T_AR = float(rng.uniform(1, 200))
        T_exp = float(rng.uniform(0, 3))
        C = float(rng.uniform(0, 2))
        sel, size = s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, T_AR, T_exp, C)
        own = [footprint_set(wl.own_fp[0][t], cfg.E) for t in range(len(wl.parent))]
        assert (sel, size) == jacobi(wl.P[0], wl.parent, own, T_AR, T_exp, C)
        for t in sel:
            assert wl.parent[t] < 0 or wl.parent[t] in sel
        U = set()
        for t in sel:
            U |= own[t]
        assert len(U) == size


@pytest.mark.parametrize("seed", range(4))
def test_zero_expert_cost_is_a_confidence_threshold(seed):
    # with T_exp = 0 the utility is p_i T_AR / C_draft: a plain threshold on P,
    # prefix-closed because P never grows along a path
    cfg, wl = random_trees(1, seed)
    for thr in [0.05, 0.1, 0.3, 0.6]:
        T_AR, C = 1.0, thr
        sel, _ = s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, T_AR, 0.0, C)
        want = [t for t in range(len(wl.parent)) if np.float64(np.float32(wl.P[0][t])) >= np.float64(np.float32(C))]
        assert sel == want


@pytest.mark.parametrize("seed", range(3))
def test_monotone_in_costs_and_gain(seed):
    cfg, wl = random_trees(1, seed)
    prev = None
    for T_exp in [0.0, 0.25, 0.5, 1.0, 2.0, 4.0, 1e9]:
        sel, _ = s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, 50.0, T_exp, 0.5)
        if prev is not None:
            assert set(sel) <= set(prev)
        prev = sel
    assert prev == []
    prev = None
    for T_AR in [1.0, 10.0, 100.0, 1e6]:
        sel, _ = s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, T_AR, 1.0, 0.5)
        if prev is not None:
            assert set(prev) <= set(sel)
        prev = sel
    # zero cost: every node is worth its draft (utility +inf), down every path
    sel, size = s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, 1.0, 0.0, 0.0)
    assert sel == list(range(len(wl.parent)))


def test_errors():
    fp = bits_of([{0}, {1}], 1)
    with pytest.raises(s2.S2Error):
        s2.s2_expand([0.5, float("nan")], [-1, 0], fp, 8, 1.0, 1.0, 0.0)
    with pytest.raises(s2.S2Error):
        s2.s2_expand([0.5, 0.25], [-1, 1], fp, 8, 1.0, 1.0, 0.0)
    with pytest.raises(s2.S2Error):
        s2.s2_expand([-0.5, 0.25], [-1, 0], fp, 8, 1.0, 1.0, 0.0)


def test_utility_exactly_one_is_taken():
    # U_i >= 1 includes equality: gain 0.5 * 4 = 2, cost 2 new * 0.5 + 1 = 2
    fp = bits_of([{1, 2}], 1)
    sel, size = s2.s2_expand([0.5], [-1], fp, 8, 4.0, 0.5, 1.0)
    assert sel == [0] and size == 2
    sel, _ = s2.s2_expand([0.5], [-1], fp, 8, 4.0, 0.5, 1.0 + 2.0 ** -20)
    assert sel == []


# ---------------------------------------------------------------- cold experts (residency)
def cold_set(bits, E):
    return {(b // E, b % E) for b in bits}


def test_hand_example_with_cold_experts():
    g = json.load(open(os.path.join(GOLD, "s2_expand_hand.json")))
    fp = bits_of(g["own"], 1)
    cc = g["cold_cases"]
    c2 = g["second_case"]
    for case in cc["cases"]:
        sel, size = s2.s2_expand(g["P"], g["parent"], fp, g["E"], g["T_AR"], c2["T_exp"], c2["C_draft"],
                                 case["T_cold"], cold_set(cc["cold"], g["E"]))
        assert sel == case["selected"] and size == case["union_size"], case["T_cold"]


@pytest.mark.parametrize("seed", range(4))
def test_all_cold_equals_a_dearer_expert(seed):
    # every expert cold: n_new * T_exp + n_new * T_cold == n_new * (T_exp + T_cold)
    # exactly for dyadic costs, so the selection is the plain one at T_exp + T_cold
    cfg, wl = random_trees(1, seed)
    every = {(l, e) for l in range(cfg.L) for e in range(cfg.E)}
    rng = np.random.default_rng(seed)
    for _ in range(10):
        T_exp = float(rng.integers(0, 32)) / 16
        T_cold = float(rng.integers(0, 64)) / 16
        C = float(rng.integers(0, 16)) / 16
        T_AR = float(rng.integers(1, 200))
        got = s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, T_AR, T_exp, C, T_cold, every)
        assert got == s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, T_AR, T_exp + T_cold, C)
        # nothing cold (or no set): the surcharge never applies
        plain = s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, T_AR, T_exp, C)
        assert s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, T_AR, T_exp, C, T_cold, set()) == plain
        assert s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, T_AR, T_exp, C, T_cold, None) == plain


def jacobi_cold(P, parent, own, T_AR, T_exp, C, T_cold, cold):
    N = len(parent)
    f = lambda v: np.float64(np.float32(v))  # noqa: E731
    gain = [f(P[t]) * f(T_AR) for t in range(N)]
    chosen = [False] * N
    B = set()
    while True:
        take = []
        for i in range(N):
            if chosen[i] or (parent[i] >= 0 and not chosen[parent[i]]):
                continue
            new = own[i] - B
            cost = (np.float64(len(new)) * f(T_exp) + np.float64(len(new & cold)) * f(T_cold)) + f(C)
            if gain[i] >= cost:
                take.append(i)
        if not take:
            return [t for t in range(N) if chosen[t]], len(B)
        for i in take:
            chosen[i] = True
            B |= own[i]


@pytest.mark.parametrize("seed", range(4))
def test_cold_order_independent_and_monotone(seed):
    cfg, wl = random_trees(1, seed)
    from oracle.eco_select import footprint_set
    rng = np.random.default_rng(100 + seed)
    own = [footprint_set(wl.own_fp[0][t], cfg.E) for t in range(len(wl.parent))]
    for _ in range(10):
        cold = {(l, e) for l in range(cfg.L) for e in range(cfg.E) if rng.random() < 0.5}
        T_AR, T_exp, C = float(rng.uniform(1, 200)), float(rng.uniform(0, 3)), float(rng.uniform(0, 2))
        prev = None
        for T_cold in [0.0, 0.5, 1.0, 3.0, 10.0, 1e9]:
            got = s2.s2_expand(wl.P[0], wl.parent, wl.own_fp[0], cfg.E, T_AR, T_exp, C, T_cold, cold)
            assert got == jacobi_cold(wl.P[0], wl.parent, own, T_AR, T_exp, C, T_cold, cold)
            if prev is not None:
                assert set(got[0]) <= set(prev)  # a dearer cold expert never adds nodes
            prev = got[0]
            # selected nodes never bring a cold expert worth more than their gain alone
            for t in got[0]:
                assert np.float64(np.float32(wl.P[0][t])) * np.float64(np.float32(T_AR)) >= np.float64(np.float32(C))

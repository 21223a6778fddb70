"""Pins for the EcoSpec selection oracle."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import eco_select as eco

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bitsets(own_lists, L, E):
    W = (L * E + 31) // 32
    out = np.zeros((len(own_lists), W), dtype=np.uint32)
    for t, pairs in enumerate(own_lists):
        for l, e in pairs:
            bit = l * E + e
            out[t, bit // 32] |= np.uint32(1 << (bit % 32))
    return out


def test_hand_trees():
    g = json.load(open(os.path.join(GOLD, "ecospec_trees.json")))
    for tree in g["trees"]:
        fp = bitsets(tree["own"], tree["L"], tree["E"])[None]
        P = np.array([tree["P"]], dtype=np.float32)
        parent = np.array(tree["parent"], dtype=np.int32)
        for ex in tree["expect"]:
            sels, sizes = eco.select_batch(P, parent, fp, tree["E"], [ex["gamma"]], g["eps"], ex["mode"])
            assert sels[0] == ex["selected"], (tree["name"], ex)
            assert sizes[0] == ex["union"], (tree["name"], ex)


def random_tree(rng, depth=3, branch=2, L=2, E=16, k=2, rho=0.6):
    parent = []
    level = [-1]
    nxt = 0
    for _ in range(depth):
        new = []
        for p in level:
            for _ in range(branch):
                parent.append(p)
                new.append(nxt)
                nxt += 1
        level = new
    N = len(parent)
    P = np.zeros(N, dtype=np.float32)
    for p in [-1] + list(range(N)):
        kids = [t for t in range(N) if parent[t] == p]
        if kids:
            q = np.sort(rng.dirichlet([0.5] * len(kids)))[::-1].astype(np.float32)
            for t, qq in zip(kids, q):
                P[t] = np.float32((np.float32(1) if p < 0 else P[p]) * qq)
    bias = -0.2 * rng.permutation(E)
    z = {-1: rng.standard_normal((L, E))}
    own = []
    for t in range(N):
        z[t] = rho * z[parent[t]] + np.sqrt(1 - rho * rho) * rng.standard_normal((L, E))
        pairs = []
        for l in range(L):
            top = np.argsort(-(bias + z[t][l]))[:k]
            pairs += [(l, int(e)) for e in top]
        own.append(pairs)
    return np.array(parent, dtype=np.int32), P, bitsets(own, L, E)


def popcount_rows(a):
    return np.array([sum(bin(int(v)).count("1") for v in row) for row in a])


def traj_bits(parent, fp):
    out = fp.copy()
    for t in range(len(parent)):
        if parent[t] >= 0:
            out[t] |= out[parent[t]]
    return out


def exact_ratio_key(p, c, eps):
    # P / (c + eps) as an exact (numerator, denominator) integer pair; eps = 2^-s
    pn, pd = float(p).as_integer_ratio()
    en, ed = float(eps).as_integer_ratio()
    return pn * ed, pd * (c * ed + en)


def greater(a, b):
    return a[0] * b[1] > b[0] * a[1]


@pytest.mark.parametrize("mode", [0, 1])
def test_greedy_output_satisfies_argmax_definition(mode):
    """Verify (not recompute) the greedy: with integer cross-multiplication over
    numpy bitsets, each chosen node scores at least as high as every remaining
    node given the buffer at that round, and beats every lower-index one."""
    rng = np.random.default_rng(10 + mode)
    eps = 2.0 ** -10
    for _ in range(60):
        parent, P, fp = random_tree(rng)
        E, gamma = 16, int(rng.integers(1, 9))
        sels, sizes = eco.select_batch(P[None], parent, fp[None], E, [gamma], eps, mode)
        sel = sels[0]
        tb = traj_bits(parent, fp)
        B = np.zeros(fp.shape[1], dtype=np.uint32)
        for r, s in enumerate(sel):
            rem = [t for t in range(len(P)) if t not in sel[:r]]
            cost = lambda t: int(popcount_rows((tb[t] & ~B)[None])[0]) if mode == 0 else int(popcount_rows(tb[t][None])[0])
            ks = exact_ratio_key(P[s], cost(s), eps)
            for t in rem:
                kt = exact_ratio_key(P[t], cost(t), eps)
                assert not greater(kt, ks)
                if t < s:
                    assert greater(ks, kt)
            B |= tb[s]
        assert sizes[0] == int(popcount_rows(B[None])[0])
        assert len(sel) == min(gamma, len(P))


def test_static_mode_equals_sort_by_static_score():
    rng = np.random.default_rng(20)
    eps = 2.0 ** -10
    for _ in range(100):
        parent, P, fp = random_tree(rng)
        gamma = int(rng.integers(1, 15))
        sels, _ = eco.select_batch(P[None], parent, fp[None], 16, [gamma], eps, 1)
        tb = traj_bits(parent, fp)
        c = popcount_rows(tb)
        order = sorted(range(len(P)), key=lambda t: (-Fraction(float(P[t])) / (int(c[t]) + Fraction(eps)), t))
        assert sels[0] == order[:gamma]


def test_prefix_closed():
    """Section 3.3: P(child) <= P(parent) and footprint(parent) subset of
    footprint(child), so the greedy set is closed under taking parents."""
    rng = np.random.default_rng(30)
    for mode in (0, 1):
        for _ in range(200):
            parent, P, fp = random_tree(rng)
            gamma = int(rng.integers(1, 15))
            sels, _ = eco.select_batch(P[None], parent, fp[None], 16, [gamma], 2.0 ** -10, mode)
            seen = set()
            for s in sels[0]:
                assert parent[s] < 0 or parent[s] in seen
                seen.add(s)


def test_marginal_not_worse_than_static_on_aggregate():
    """The write-up's ablation favours marginal cost; per tree it is not a theorem
    (see the hand tree marginal_vs_static), so compare the mean union over 1000
    seeded trees and bound the counterexample rate."""
    rng = np.random.default_rng(40)
    um, us, worse = [], [], 0
    for _ in range(1000):
        parent, P, fp = random_tree(rng, L=2, E=16, k=2)
        _, sm = eco.select_batch(P[None], parent, fp[None], 16, [4], 2.0 ** -10, 0)
        _, ss = eco.select_batch(P[None], parent, fp[None], 16, [4], 2.0 ** -10, 1)
        um.append(sm[0])
        us.append(ss[0])
        worse += sm[0] > ss[0]
    assert np.mean(um) < np.mean(us)
    assert worse / 1000 < 0.05


def test_footprint_set_roundtrip():
    fp = bitsets([[(0, 0), (1, 15), (2, 31), (3, 0)]], 4, 32)[0]
    assert eco.footprint_set(fp, 32) == {(0, 0), (1, 15), (2, 31), (3, 0)}


# ------------------------------------------------------------ batch-global mode
def test_batch_global_one_sequence_is_the_per_sequence_greedy():
    rng = np.random.default_rng(50)
    for _ in range(100):
        parent, P, fp = random_tree(rng)
        g = int(rng.integers(0, 15))
        sels, sizes = eco.select_batch(P[None], parent, fp[None], 16, [g], 2.0 ** -10, 0)
        bs, bsz, bu = eco.select_batch_global(P[None], parent, fp[None], 16, [g], 2.0 ** -10, 14)
        assert bs == sels and bsz == sizes and bu == sizes[0]


def test_batch_global_hand_example():
    # sequence A: a0 (P .9, 3 experts) -> a1 (P .8, 2 more); sequence B: b0 (P .6,
    # 1 expert) -> b1 (P .5, 1 more).  Budget 2 (gamma 1 + 1), cap 2.
    # Per sequence: A takes a0, B takes b0: union {1,2,3,6}.
    # Batch: b0 scores .6/1 > a0 .9/3; then b1 (cost 1, .5) beats a0 (.3):
    # depth vector (0, 2), union {6, 7}.
    E = 16
    parent = np.array([-1, 0])
    P = np.array([[0.9, 0.8], [0.6, 0.5]], dtype=np.float32)
    fp = np.stack([bitsets([[(0, 1), (0, 2), (0, 3)], [(0, 4), (0, 5)]], 1, E),
                   bitsets([[(0, 6)], [(0, 7)]], 1, E)])
    sels, sizes = eco.select_batch(P, parent, fp, E, [1, 1], 2.0 ** -10, 0)
    assert sels == [[0], [0]] and sizes == [3, 1]
    bs, bsz, bu = eco.select_batch_global(P, parent, fp, E, [1, 1], 2.0 ** -10, 2)
    assert bs == [[], [0, 1]] and bsz == [0, 2] and bu == 2
    # a cap of one node per sequence forces the second pick into A
    bs, bsz, bu = eco.select_batch_global(P, parent, fp, E, [1, 1], 2.0 ** -10, 1)
    assert bs == [[0], [0]] and bu == 4


def test_batch_global_budget_cap_prefix_and_unions():
    rng = np.random.default_rng(51)
    for _ in range(60):
        trees = [random_tree(rng) for _ in range(3)]
        parent = trees[0][0]
        P = np.stack([tr[1] for tr in trees])
        fp = np.stack([tr[2] for tr in trees])
        gam = [int(x) for x in rng.integers(0, 7, size=3)]
        cap = int(rng.integers(1, 15))
        bs, bsz, bu = eco.select_batch_global(P, parent, fp, 16, gam, 2.0 ** -10, cap)
        assert sum(len(x) for x in bs) == min(sum(gam), 3 * min(cap, 14))
        U = set()
        for s in range(3):
            assert len(bs[s]) <= cap
            own = [eco.footprint_set(fp[s, t], 16) for t in range(14)]
            traj = eco.trajectory_footprints(list(parent), own)
            seen, Us = set(), set()
            for t in bs[s]:
                assert parent[t] < 0 or parent[t] in seen
                seen.add(t)
                Us |= traj[t]
            assert len(Us) == bsz[s]
            U |= Us
        assert len(U) == bu


def test_batch_global_union_not_larger_on_aggregate():
    """Sharing B across the batch lets the greedy buy experts once for several
    sequences; over seeded batches of four trees with one budget, the batch
    union is smaller on average than the union of per-sequence selections."""
    rng = np.random.default_rng(52)
    ub, up = [], []
    for _ in range(150):
        trees = [random_tree(rng, L=2, E=16, k=2) for _ in range(4)]
        parent = trees[0][0]
        P = np.stack([tr[1] for tr in trees])
        fp = np.stack([tr[2] for tr in trees])
        sels, _ = eco.select_batch(P, parent, fp, 16, [4] * 4, 2.0 ** -10, 0)
        U = set()
        for s in range(4):
            own = [eco.footprint_set(fp[s, t], 16) for t in range(14)]
            traj = eco.trajectory_footprints(list(parent), own)
            for t in sels[s]:
                U |= traj[t]
        up.append(len(U))
        _, _, bu = eco.select_batch_global(P, parent, fp, 16, [4] * 4, 2.0 ** -10, 14)
        ub.append(bu)
    assert np.mean(ub) < np.mean(up)


def test_batch_global_ties_go_to_the_lower_sequence():
    E = 16
    parent = np.array([-1, 0])
    P = np.array([[0.5, 0.25], [0.5, 0.25]], dtype=np.float32)
    one = bitsets([[(0, 1)], [(0, 2)]], 1, E)
    fp = np.stack([one, one])
    bs, bsz, bu = eco.select_batch_global(P, parent, fp, E, [1, 0], 2.0 ** -10, 2)
    assert bs == [[0], []] and bu == 1

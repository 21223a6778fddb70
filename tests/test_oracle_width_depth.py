"""Pins for the width-vs-depth oracle (width-vs-depth note, sections 1 and 2).

Expected values are worked out by hand in the comments, enumerated by brute
force, or closed forms; none comes from the function under test on another
input."""
import itertools

import numpy as np
import pytest

from oracle import width_depth as wd


def _fp(sets, W=1):
    """[nseq, D+1, W] uint32 footprints from lists of bit sets."""
    out = np.zeros((len(sets), len(sets[0]), W), np.uint32)
    for i, row in enumerate(sets):
        for j, bits in enumerate(row):
            for b in bits:
                out[i, j, b // 32] |= np.uint32(1 << (b % 32))
    return out


@pytest.mark.parametrize("q", [[0.5], [0.9, 0.3], [0.25, 0.75, 1.0], [1.0, 0.0, 0.5, 0.5], [0.6] * 5])
def test_expected_accepted_is_the_mean_committed_length(q):
    """Drafts accepted independently with probabilities q_1..q_d; the step
    commits 1 token plus the accepted prefix.  Enumerate every outcome."""
    d = len(q)
    mean = 0.0
    for outcome in itertools.product([0, 1], repeat=d):
        p = 1.0
        for acc, qq in zip(outcome, q):
            p *= qq if acc else 1.0 - qq
        prefix = 0
        while prefix < d and outcome[prefix]:
            prefix += 1
        mean += p * (1 + prefix)
    cum = np.cumprod(np.array(q, np.float64)).astype(np.float32)
    assert abs(wd.expected_accepted(cum, d) - mean) < 1e-6
    assert wd.expected_accepted(cum, 0) == 1.0


# Hand-worked batch (dyadic confidences, every value exact in fp64):
#   seq 0: c = [.875, .75], footprints root {0}, p1 {0}, p2 {1}   (co-activation)
#   seq 1: c = [.125, .0625], footprints root {2}, p1 {3,4}, p2 {5,6}
#   C0 = 8, T_exp = 1.   A_0 = [1, 1.875, 2.625], A_1 = [1, 1.125, 1.1875].
#   common: D'=0 2/10 = .2; D'=1 3/12 = .25; D'=2 3.8125/15 = .2542 -> D* = 2
#   truncation from [2,2]: [1,2] 3.0625/14 = .2188, [2,1] 3.75/13 = .2885 -> [2,1]
#              from [2,1]: [1,1] 3/12 = .25,      [2,0] 3.625/11 = .3295 -> [2,0]
#              from [2,0]: [1,0] 2.875/10 = .2875 < .3295               -> stop
CONF = np.array([[0.875, 0.75], [0.125, 0.0625]], np.float32)
FP = _fp([[{0}, {0}, {1}], [{2}, {3, 4}, {5, 6}]])


def test_hand_batch():
    r = wd.depth_policy(CONF, FP, 8.0, 1.0)
    assert r["common"] == 2
    assert r["depth"] == [2, 0]
    assert r["thr_common"] == 3.8125 / 15
    assert r["thr"] == 3.625 / 11


def test_hand_batch_with_depth_limits():
    # seq 0 limited to depth 1: common D'=0 .2, D'=1 3/12 = .25, D'=2 [1,2]
    # 3.0625/14 = .21875 -> D* = 1, d = [1,1]; truncation: [0,1] 2.125/11 =
    # .1932, [1,0] 2.875/10 = .2875 -> [1,0]; then [0,0] 2/10 = .2 -> stop.
    r = wd.depth_policy(CONF, FP, 8.0, 1.0, max_depth=[1, 2])
    assert (r["common"], r["depth"], r["thr"]) == (1, [1, 0], 2.875 / 10)


def test_common_depth_ties_go_to_the_smaller_depth():
    # seq 0: c = [.75, .5], root {0}, p1 {1}, p2 {2}; seq 1: c = [.25, .125],
    # root {3}, p1 {4,5}, p2 {6,7}; C0 = 4, T_exp = 1:
    # D'=0: 2/6 = 1/3; D'=1: 3/9 = 1/3 (exact tie) -> D* = 0; D'=2: 3.625/12.
    conf = np.array([[0.75, 0.5], [0.25, 0.125]], np.float32)
    fp = _fp([[{0}, {1}, {2}], [{3}, {4, 5}, {6, 7}]])
    r = wd.depth_policy(conf, fp, 4.0, 1.0)
    assert r["common"] == 0 and r["depth"] == [0, 0] and r["thr"] == 2 / 6


def test_union_counts_shared_experts_once_across_sequences():
    fp = _fp([[{0, 1}, {2}], [{1, 33}, {2, 40}]], W=2)
    m = wd.DepthModel(np.zeros((2, 1), np.float32), fp, 1.0, 1.0)
    assert m.union([0, 0]) == 3       # {0,1} | {1,33}
    assert m.union([1, 0]) == 4       # + {2}
    assert m.union([1, 1]) == 5       # + {40} ({2} already counted)


def _rand_batch(rng, nseq, D, W):
    q = rng.uniform(0.0, 1.0, size=(nseq, D))
    conf = np.cumprod(q, axis=1).astype(np.float32)
    fp = rng.integers(0, 2 ** 32, size=(nseq, D + 1, W), dtype=np.uint64)
    fp &= rng.integers(0, 2 ** 32, size=fp.shape, dtype=np.uint64)  # sparser
    return conf, fp.astype(np.uint32)


def _thr_bruteforce(conf, fp, C0, T_exp, d):
    """Throughput of a depth vector written out directly from the definition."""
    nseq = conf.shape[0]
    num = 0.0
    bits = set()
    for i in range(nseq):
        a = 1.0
        for j in range(d[i]):
            a = a + float(conf[i, j])
        num = num + a
        for j in range(d[i] + 1):
            for w, word in enumerate(fp[i, j].tolist()):
                bits |= {32 * w + b for b in range(32) if (word >> b) & 1}
    return num / (float(np.float32(C0)) + float(np.float32(T_exp)) * len(bits))


@pytest.mark.parametrize("seed", range(6))
def test_one_sequence_is_the_exhaustive_optimum(seed):
    rng = np.random.default_rng(seed)
    conf, fp = _rand_batch(rng, 1, 6, 2)
    C0, T_exp = float(rng.uniform(1, 20)), float(rng.uniform(0, 2))
    vals = [_thr_bruteforce(conf, fp, C0, T_exp, [D]) for D in range(7)]
    best = max(vals)
    r = wd.depth_policy(conf, fp, C0, T_exp)
    assert r["depth"] == [vals.index(best)] and r["thr"] == best


@pytest.mark.parametrize("seed", range(8))
def test_gated_never_loses_to_common_and_is_a_local_optimum(seed):
    rng = np.random.default_rng(100 + seed)
    nseq, D = int(rng.integers(2, 5)), int(rng.integers(1, 5))
    conf, fp = _rand_batch(rng, nseq, D, 1)
    C0, T_exp = float(rng.uniform(1, 10)), float(rng.uniform(0.1, 2))
    r = wd.depth_policy(conf, fp, C0, T_exp)
    d = r["depth"]
    assert r["thr"] >= r["thr_common"]
    assert all(0 <= d[i] <= r["common"] for i in range(nseq))
    assert r["thr"] == _thr_bruteforce(conf, fp, C0, T_exp, d)
    for i in range(nseq):
        if d[i] > 0:
            c = list(d)
            c[i] -= 1
            assert _thr_bruteforce(conf, fp, C0, T_exp, c) <= r["thr"]
    best = max(_thr_bruteforce(conf, fp, C0, T_exp, list(v))
               for v in itertools.product(range(D + 1), repeat=nseq))
    assert best >= r["thr"]


def test_free_experts_verify_everything():
    # T_exp = 0: the cost is C0 whatever the union, and every positive
    # confidence adds expected tokens, so the full depth wins for everyone.
    rng = np.random.default_rng(7)
    conf, fp = _rand_batch(rng, 3, 5, 1)
    conf = np.maximum(conf, np.float32(1e-3))
    r = wd.depth_policy(conf, fp, 5.0, 0.0)
    assert r["common"] == 5 and r["depth"] == [5, 5, 5]


def test_hopeless_drafts_verify_nothing():
    rng = np.random.default_rng(8)
    _, fp = _rand_batch(rng, 3, 4, 1)
    r = wd.depth_policy(np.zeros((3, 4), np.float32), fp, 5.0, 1.0)
    assert r["common"] == 0 and r["depth"] == [0, 0, 0]


def test_layer_unions_hand():
    # 2 layers, 3 tokens, E = 5, k = 2.
    lg = np.array([[[5, 4, 0, 0, 0], [0, 5, 4, 0, 0], [5, 0, 0, 0, 4]],
                   [[1, 2, 3, 4, 5], [1, 2, 3, 5, 4], [5, 4, 3, 2, 1]]], np.float32)
    # layer 0: {0,1} | {1,2} | {0,4} = 4;  layer 1: {4,3} | {3,4} | {0,1} = 4
    assert wd.layer_unions(lg, 2) == [4, 4]
    assert wd.layer_unions(lg[:, :1], 2) == [2, 2]

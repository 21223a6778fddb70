"""Pins for the oracle's verify-step glue: which node-table rows a round
verifies, with which bias confidences, in which selection, and how a layer
chains bias -> route -> union -> experts.

EcoSpec write-up, section 2: a round verifies the last accepted token (the
root) followed by the gamma selected draft tokens; section 3.3 (greedy) and
section 4.3 (static ablation).  S2-MoE write-up, component 2: the bias
confidence w_b of a verify token comes from its draft confidence (path
probability; 1 for the root, which is already accepted).

Every expected value below is worked out by hand in the comments; none is
produced by calling the function under test on another input.
"""
import json
import math
import os
from types import SimpleNamespace

import numpy as np
import pytest

from oracle import moe_layer as ml
from oracle import verify_step as vs

GOLD = os.path.join(os.path.dirname(__file__), "golden")
EPS = 2.0 ** -10

# A forest of two sequences over the same 3-node draft tree:
#   root -> node 0 -> node 2,   root -> node 1          (breadth-first)
PARENT = np.array([-1, -1, 0], dtype=np.int32)
N = 3
E = 8
# Path probabilities (child <= parent).
P = np.array([[0.5, 0.25, 0.25],
              [0.75, 0.125, 0.5]], dtype=np.float32)
# Own predicted footprints, one layer of 8 experts (bit e marks expert e):
#   seq 0: node0 {0,1}, node1 {2,3}, node2 {1,4} -> E_traj: {0,1}, {2,3}, {0,1,4}
#   seq 1: node0 {5,6}, node1 {0,7}, node2 {6,7} -> E_traj: {5,6}, {0,7}, {5,6,7}
OWN = np.array([[[0b00000011], [0b00001100], [0b00010010]],
                [[0b01100000], [0b10000001], [0b11000000]]], dtype=np.uint32)
GAMMA = np.array([2, 1], dtype=np.int32)

# Hand-worked selections (eps = 2^-10 never decides an order here):
# marginal, seq 0, gamma 2: round 1 scores .5/2, .25/2, .25/3 -> node 0,
#   B = {0,1}; round 2: node 1 .25/2, node 2 .25/1 -> node 2; |B| = 3.
# marginal, seq 1, gamma 1: .75/2, .125/2, .5/3 -> node 0; |B| = 2.
SEL_MARGINAL = ([[0, 2], [0]], [3, 2])
# static, seq 0: node 0 first (.5/2), then node 1 (.25/2) over node 2 (.25/3);
#   |B| = |{0,1,2,3}| = 4.  seq 1 as marginal.
SEL_STATIC = ([[0, 1], [0]], [4, 2])
# batch-global (one B, budget 2 + 1 = 3, at most 2 nodes per sequence):
#   round 1: s1n0 .75/2 = .375 beats s0n0 .25 -> B = {5,6};
#   round 2: s1n2 .5/|{7}| = .5 beats s0n0 .25 -> B = {5,6,7}, seq 1 full;
#   round 3: s0n0 .25 -> B = {0,1,5,6,7}.
#   Per-sequence unions of their own trajectories: {0,1} and {5,6,7}.
SEL_GLOBAL = ([[0], [0, 2]], [2, 3])


def _wl(mode=0, use_bias=False, cap=0, alpha=0.0, logits=None, x=None, H=4):
    cfg = SimpleNamespace(mode=mode, E=E, eps=EPS, L=1, k=2, H=H, use_bias=use_bias, cap=cap,
                          alpha=alpha)
    if logits is None:
        logits = np.zeros((1, 2, N + 1, E), np.float32)
    if x is None:
        x = np.zeros((1, 2, N + 1, H), np.float32)
    return SimpleNamespace(cfg=cfg, parent=PARENT, P=P, own_fp=OWN, gamma=GAMMA, logits=logits, x=x)


@pytest.mark.parametrize("mode,want", [(0, SEL_MARGINAL), (1, SEL_STATIC), (2, SEL_GLOBAL)])
def test_run_selection_hand_forest(mode, want):
    sels, sizes = vs.run_selection(_wl(mode=mode))
    assert [list(map(int, s)) for s in sels] == want[0]
    assert list(map(int, sizes)) == want[1]


def test_run_selection_mode_argument_overrides_config():
    sels, _ = vs.run_selection(_wl(mode=0), mode=1)
    assert [list(map(int, s)) for s in sels] == SEL_STATIC[0]
    # batch-global with a per-sequence cap of 1: round 1 s1n0, round 2 s0n0,
    # round 3 finds no sequence below its cap -> stops with 2 of 3.
    sels, sizes = vs.run_selection(_wl(mode=2), cap=1)
    assert [list(map(int, s)) for s in sels] == [[0], [0]]
    assert list(map(int, sizes)) == [2, 2]


def test_verify_rows_root_then_selected_in_order():
    # table rows per sequence: N + 1 = 4 (row 0 = root, row 1 + t = node t)
    assert vs.verify_rows(N, [[0, 2], [0]]) == [0, 1, 3, 4, 5]
    assert vs.verify_rows(N, [[2, 0], [1]]) == [0, 3, 1, 4, 6]
    assert vs.verify_rows(N, [[], []]) == [0, 4]
    assert vs.verify_rows(5, [[4], [], [0, 1]]) == [0, 5, 6, 12, 13, 14]


def test_token_conf_root_one_then_path_probabilities():
    c = vs.token_conf(P, [[0, 2], [0]])
    assert c.dtype == np.float32
    assert c.tolist() == [1.0, 0.5, 0.25, 1.0, 0.75]
    assert vs.token_conf(P, [[1], []]).tolist() == [1.0, 0.25, 1.0]


# Node-table logits for the step pin.  Row r of sequence s is s*(N+1) + j.
# Each row has a top-2 pair (4.0, 3.0), a third expert at 2.0 and zeros:
ROW_TOP = {0: (0, 1, 2), 1: (2, 3, 4), 2: (7, 5, 0), 3: (2, 3, 0),
           4: (4, 5, 6), 5: (0, 6, 1), 6: (3, 7, 0), 7: (1, 7, 0)}


def _table_logits():
    lg = np.zeros((1, 2, N + 1, E), np.float32)
    for r, (a, b, c) in ROW_TOP.items():
        s, j = divmod(r, N + 1)
        lg[0, s, j, a], lg[0, s, j, b], lg[0, s, j, c] = 4.0, 3.0, 2.0
    return lg


def _experts(H, I=2):
    """Small distinct expert matrices: W_gate_up [2I, H], W_down [H, I]."""
    def one(e):
        gu = np.array([[((e + 1) * (r + 1) + c) % 5 - 2 for c in range(H)] for r in range(2 * I)],
                      np.float64) / 4.0
        dn = np.array([[((e + 2) * (r + 3) + 2 * c) % 7 - 3 for c in range(I)] for r in range(H)],
                      np.float64) / 8.0
        return gu, dn
    return one


def _swiglu(x, gu, dn):
    I = dn.shape[1]
    a, b = gu[:I] @ x, gu[I:] @ x
    return dn @ ((a / (1.0 + np.exp(-a))) * b)


def test_run_step_verifies_the_selected_rows_unbiased():
    H = 4
    x = np.arange(2 * (N + 1) * H, dtype=np.float32).reshape(1, 2, N + 1, H) / 16.0 - 1.0
    wl = _wl(mode=0, logits=_table_logits(), x=x, H=H)
    ex = _experts(H)
    out = vs.run_step(wl, lambda l: ex, x_decode=lambda a: np.asarray(a, np.float64))
    assert out["rows"] == [0, 1, 3, 4, 5]
    lay = out["layers"][0]
    # verify rows 0, 1, 3, 4, 5 -> their top-2 pairs, in descending logit
    assert lay["ids"].tolist() == [[0, 1], [2, 3], [2, 3], [4, 5], [0, 6]]
    assert lay["n_unique"] == 7 and lay["unique"].tolist() == [0, 1, 2, 3, 4, 5, 6]
    w0 = 1.0 / (1.0 + math.exp(-1.0))  # softmax over (4, 3)
    assert np.allclose(lay["w"], [[w0, 1 - w0]] * 5, rtol=0, atol=1e-15)
    # FFN on the hidden states of the same rows
    xr = x.reshape(-1, H)[[0, 1, 3, 4, 5]].astype(np.float64)
    want = np.stack([w0 * _swiglu(xr[t], *ex(lay["ids"][t, 0])) + (1 - w0) * _swiglu(xr[t], *ex(lay["ids"][t, 1]))
                     for t in range(5)])
    assert np.allclose(lay["y"], want, rtol=1e-14, atol=1e-14)


def test_run_step_bias_uses_root_one_and_path_probability():
    # Verify rows 0,1,3,4,5 with confidences 1, .5, .25, 1, .75 (root 1, node P).
    # g_e over their top-2 sets {0,1},{2,3},{2,3},{4,5},{0,6}:
    #   g = [1.75, 1, .75, .75, 1, 1, .75, 0] -> E* (cap 2) = {0, 1}
    #   (all-ones weights would give {0, 2}; shifted weights {0, 2} too).
    # lambda = alpha * (4 - 2) = 1 for every row, so on E*:
    #   row 0: e0 5, e1 4 -> ids [0, 1]; row 1: e0 1, e1 1 -> ids [2, 3];
    #   row 3: e2 4, e0 3 = e3 3 -> tie to the lower id -> ids [2, 0];
    #   row 4: unchanged [4, 5]; row 5: e0 5, e1 3 = e6 3 -> ids [0, 1].
    H = 4
    x = np.ones((1, 2, N + 1, H), np.float32)
    wl = _wl(mode=0, use_bias=True, cap=2, alpha=0.5, logits=_table_logits(), x=x, H=H)
    out = vs.run_step(wl, lambda l: _experts(H), x_decode=lambda a: np.asarray(a, np.float64))
    assert out["conf"].tolist() == [1.0, 0.5, 0.25, 1.0, 0.75]
    lay = out["layers"][0]
    assert lay["ids"].tolist() == [[0, 1], [2, 3], [2, 0], [4, 5], [0, 1]]
    assert lay["n_unique"] == 6
    used = lay["logits_used"]
    assert used[0].tolist() == [5, 4, 2, 0, 0, 0, 0, 0]
    assert used[4].tolist() == [5, 3, 0, 0, 0, 0, 3, 0]
    w1, w2 = 1.0 / (1.0 + math.exp(-1.0)), 1.0 / (1.0 + math.exp(-2.0))
    assert np.allclose(lay["w"][[0, 2, 4], 0], [w1, w1, w2], rtol=0, atol=1e-15)


def test_run_step_token_subset_changes_only_the_ffn_rows():
    H = 4
    x = np.arange(2 * (N + 1) * H, dtype=np.float32).reshape(1, 2, N + 1, H) / 8.0 - 2.0
    wl = _wl(mode=0, logits=_table_logits(), x=x, H=H)
    dec = lambda a: np.asarray(a, np.float64)  # noqa: E731
    full = vs.run_step(wl, lambda l: _experts(H), x_decode=dec)["layers"][0]
    part = vs.run_step(wl, lambda l: _experts(H), x_decode=dec, tokens=[1, 3])["layers"][0]
    for key in ("ids", "unique", "offsets", "perm_token", "inv"):
        assert np.array_equal(full[key], part[key]), key
    assert np.allclose(full["w"], part["w"], rtol=0, atol=0)
    assert part["tokens"].tolist() == [1, 3]
    assert np.array_equal(part["y"], full["y"][[1, 3]])


def test_run_step_empty_budget_verifies_roots_only():
    wl = _wl(mode=0, logits=_table_logits(), x=np.ones((1, 2, N + 1, 4), np.float32))
    wl.gamma = np.array([0, 0], np.int32)
    out = vs.run_step(wl, lambda l: _experts(4), x_decode=lambda a: np.asarray(a, np.float64))
    assert out["rows"] == [0, 4] and out["selected"] == [[], []]
    assert out["layers"][0]["ids"].tolist() == [[0, 1], [4, 5]]


def test_layer_forward_bias_on_fig5_fixture():
    """S2-MoE Fig. 5 counts through layer_forward: the biased layer routes T4
    onto the preferred set and the union drops from 6 to 4; tokens keep the
    expected top-2 and the FFN rows are those of the biased routing."""
    with open(os.path.join(GOLD, "reuse_bias_fig5.json")) as f:
        g = json.load(f)
    lg = np.array(g["logits"], np.float32)
    H = 4
    x = np.linspace(-1.0, 1.0, lg.shape[0] * H).reshape(lg.shape[0], H)
    ex = _experts(H)
    plain = ml.layer_forward(lg, x, g["k"], g["E"], ex)
    biased = ml.layer_forward(lg, x, g["k"], g["E"], ex, w_conf=np.array(g["w_conf"], np.float32),
                              cap=g["cap"], alpha=g["alpha"])
    assert plain["ids"].tolist() == g["expected"]["ids_before"] and plain["n_unique"] == 6
    assert biased["ids"].tolist() == g["expected"]["ids_after"] and biased["n_unique"] == 4
    assert biased["logits_used"][3].tolist() == g["expected"]["t4_biased_logits"]
    # T1 and T2 route only to preferred experts: both their logits move by the
    # same lambda, so their softmax weights and FFN rows stay as they were.
    # T3 keeps its experts, but one of them (E2) is preferred, so its weights move.
    assert np.array_equal(plain["y"][:2], biased["y"][:2])
    assert biased["ids"][2].tolist() == plain["ids"][2].tolist()
    assert biased["w"][2, 0] > plain["w"][2, 0]
    w = biased["w"][3]
    e0, e1 = g["expected"]["ids_after"][3]
    want = w[0] * _swiglu(x[3], *ex(e0)) + w[1] * _swiglu(x[3], *ex(e1))
    assert np.allclose(biased["y"][3], want, rtol=1e-14, atol=1e-14)
    # T4's weights: softmax over its biased top-2, 1.25 and 1.125
    w_hand = 1.0 / (1.0 + math.exp(-0.125))
    assert abs(w[0] - w_hand) < 1e-15 and abs(w[1] - (1 - w_hand)) < 1e-15

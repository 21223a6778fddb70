"""Pins for the router-logits oracle against a hand example and exact arithmetic."""
import json
import os
from fractions import Fraction

import numpy as np

from oracle import moe_layer as ml
from oracle import router as orr
from workload import counter_hash as ch
from workload import gen

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_example():
    g = json.load(open(os.path.join(GOLD, "router_hand.json")))
    x = np.array(g["x"], dtype=np.float64)
    w = np.array(g["w_r"], dtype=np.float64)
    got = orr.router_logits(x, w)
    assert got.tolist() == g["logits"]
    ids, _ = ml.route(got.astype(np.float32), 2)
    assert ids.tolist() == g["top2_ids"]


def test_hand_example_through_bf16_storage():
    g = json.load(open(os.path.join(GOLD, "router_hand.json")))
    xb = gen.bf16_bits_rne(np.array(g["x"], dtype=np.float32))
    wb = gen.bf16_bits_rne(np.array(g["w_r"], dtype=np.float32))
    got = orr.router_logits(orr.decode(xb, "bf16"), orr.decode(wb, "bf16"))
    assert got.tolist() == g["logits"]


def _exact(xf, wf):
    T, H = len(xf), len(xf[0])
    E = len(wf)
    return [[sum((xf[t][h] * wf[e][h] for h in range(H)), Fraction(0)) for e in range(E)]
            for t in range(T)]


def test_brute_force_rationals():
    # grid values (odd multiples of 2^-13) and bf16 hidden states: every product
    # and every partial sum of <= 64 terms is exact in fp64, so the oracle must
    # equal the rational sum bit for bit
    rng = np.random.default_rng(5)
    for T, H, E in [(1, 8, 1), (3, 16, 5), (4, 64, 7)]:
        key = ch.stream_key(99, T * 1000 + H)
        wbits = ch.fill_host(ch.KIND_GRID8_BF16, key, 0, E * H).reshape(E, H)
        xbits = gen.bf16_bits_rne(rng.standard_normal((T, H)).astype(np.float32))
        x = orr.decode(xbits, "bf16")
        w = orr.decode(wbits, "bf16")
        got = orr.router_logits(x, w)
        want = _exact([[Fraction(v) for v in r] for r in x], [[Fraction(v) for v in r] for r in w])
        assert [[Fraction(v) for v in r] for r in got] == want


def test_basis_rows_select_components():
    rng = np.random.default_rng(6)
    H, E = 32, 6
    x = rng.standard_normal((4, H))
    cols = rng.permutation(H)[:E]
    w = np.zeros((E, H))
    w[np.arange(E), cols] = 1.0
    assert np.array_equal(orr.router_logits(x, w), x[:, cols])
    # a negated, doubled basis row
    w[2] *= -2.0
    assert np.array_equal(orr.router_logits(x, w)[:, 2], -2.0 * x[:, cols[2]])


def test_linearity_in_x():
    rng = np.random.default_rng(7)
    H, E = 48, 5
    grid = lambda *s: rng.integers(-255, 256, size=s) * 2.0 ** -13
    w = grid(E, H)
    x1, x2 = grid(2, H), grid(2, H)
    lhs = orr.router_logits(0.5 * x1 - 4.0 * x2, w)
    rhs = 0.5 * orr.router_logits(x1, w) - 4.0 * orr.router_logits(x2, w)
    assert np.array_equal(lhs, rhs)


def test_fp32_decode_and_shape_checks():
    x = np.array([[1.5, -2.0]], dtype=np.float32)
    assert orr.decode(x, "f32").dtype == np.float64
    try:
        orr.router_logits(np.zeros((2, 3)), np.zeros((4, 5)))
    except ValueError:
        pass
    else:
        raise AssertionError("mismatched H accepted")


def test_router_weights_regenerate():
    cfg = gen.CONFIGS["toy"]
    a = gen.router_weights_host(cfg, 0)
    b = gen.router_weights_host(cfg, 0)
    assert a.shape == (cfg.E, cfg.H) and np.array_equal(a, b)
    assert not np.array_equal(a, gen.router_weights_host(cfg, 1)[: cfg.E])

"""Pins for the MoE-layer oracle against what the pages and mathematics fix."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import moe_layer as ml
from oracle import verify_step as vs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ decoding
def test_bf16_decode_known_values():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x3F00, 0x7F7F, 0x0001], dtype=np.uint16)
    want = [1.0, -2.0, 0.0, -0.0, 0.5, (2 - 2 ** -7) * 2.0 ** 127, 2.0 ** -133]
    got = ml.decode_bf16(bits)
    assert got.tolist() == want
    assert math.copysign(1, got[3]) == -1


def test_e4m3_decode_ocp_values():
    # OCP 8-bit floating point spec, E4M3: max normal 448, min normal 2^-6,
    # min subnormal 2^-9, S.1111.111 is NaN, 0x38 is 1.0.
    codes = np.array([0x7E, 0xFE, 0x08, 0x01, 0x38, 0x00, 0x80, 0x40, 0x07, 0x39], dtype=np.uint8)
    want = [448.0, -448.0, 2.0 ** -6, 2.0 ** -9, 1.0, 0.0, -0.0, 2.0, 7 * 2.0 ** -9, 1.125]
    assert ml.decode_e4m3(codes).tolist() == want
    assert np.isnan(ml.decode_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    # every finite code decodes to a distinct magnitude per sign
    allc = np.arange(256, dtype=np.uint8)
    v = ml.decode_e4m3(allc)
    fin = ~np.isnan(v)
    assert fin.sum() == 254
    pos = v[(allc < 128) & fin]
    assert len(np.unique(pos)) == 127 and pos.max() == 448.0


def test_fp8_block_scale_applies_per_128_block():
    rng = np.random.default_rng(0)
    codes = np.full((256, 256), 0x38, dtype=np.uint8)  # all 1.0
    sc = rng.uniform(0.5, 2.0, size=(2, 2)).astype(np.float32)
    w = {"gate_up": codes, "down": codes[:, :128], "scale_gate_up": sc, "scale_down": sc[:, :1]}
    gu, dn = ml.expert_matrices(w, "e4m3")
    assert gu[0, 0] == sc[0, 0] and gu[127, 127] == sc[0, 0]
    assert gu[128, 0] == sc[1, 0] and gu[0, 128] == sc[0, 1] and gu[255, 255] == sc[1, 1]
    assert dn[200, 100] == sc[1, 0]


# ------------------------------------------------------------------ routing
def test_route_hand_cases():
    g = load("route_hand.json")
    for c in g["cases"]:
        lg = np.array([c["logits"]], dtype=np.float32)
        ids, w = ml.route(lg, c["k"])
        assert ids[0].tolist() == c["ids"]
        np.testing.assert_allclose(w[0], c["weights"], rtol=1e-14)


def test_route_definition_on_random_rows():
    rng = np.random.default_rng(1)
    for _ in range(30):
        E = int(rng.integers(4, 64))
        k = int(rng.integers(1, E + 1))
        lg = rng.standard_normal((3, E)).astype(np.float32)
        # plant exact ties
        lg[0, : E // 2] = lg[0, E // 2: E // 2 * 2]
        ids, w = ml.route(lg, k)
        for t in range(3):
            sel = ids[t].tolist()
            rest = [e for e in range(E) if e not in sel]
            assert len(set(sel)) == k
            # every selected logit >= every unselected; ties among equal values by id
            for a in sel:
                for b in rest:
                    assert lg[t, a] > lg[t, b] or (lg[t, a] == lg[t, b] and a < b)
            # descending order, ties by id
            for a, b in zip(sel, sel[1:]):
                assert lg[t, a] > lg[t, b] or (lg[t, a] == lg[t, b] and a < b)
            # weights = full softmax renormalised over the selected experts
            full = scipy.special.softmax(lg[t].astype(np.float64))
            ref = full[sel] / full[sel].sum()
            np.testing.assert_allclose(w[t], ref, rtol=1e-12)
            assert abs(math.fsum(w[t]) - 1.0) < 1e-14


def test_route_nan_is_error():
    lg = np.array([[0.0, np.nan, 1.0]], dtype=np.float32)
    with pytest.raises(ml.OracleError):
        ml.route(lg, 1)


# ------------------------------------------------------------------ union
def test_union_all_tokens_share_one_set():
    # S2-MoE challenge 2: if all tokens share the same k experts the ratio is 1/s.
    T, k, E = 5, 8, 128
    ids = np.tile(np.array([3, 9, 1, 77, 5, 6, 100, 2], dtype=np.int32), (T, 1))
    up = ml.union_permute(ids, E)
    assert up["n_unique"] == k
    assert up["reuse_ratio"] == np.float32(1.0 / T)


def test_union_disjoint_tokens():
    T, k, E = 4, 3, 12
    ids = np.arange(T * k, dtype=np.int32).reshape(T, k)[:, ::-1].copy()
    up = ml.union_permute(ids, E)
    assert up["n_unique"] == T * k and up["reuse_ratio"] == np.float32(1.0)


def test_union_csr_properties_random():
    rng = np.random.default_rng(2)
    for _ in range(40):
        E = int(rng.integers(2, 40))
        k = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.integers(1, 12))
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        up = ml.union_permute(ids, E)
        U = up["n_unique"]
        # EcoSpec section 1: weights to load = union; bound min(E, T*k)
        assert k <= U <= min(E, T * k)
        assert 1.0 / T - 1e-7 <= up["reuse_ratio"] <= 1.0
        assert up["unique"].tolist() == sorted(set(ids.ravel().tolist()))
        counts = np.bincount(ids.ravel(), minlength=E)
        assert np.diff(up["offsets"]).tolist() == counts[up["unique"]].tolist()
        pt, ps, inv = up["perm_token"], up["perm_slot"], up["inv"]
        for u in range(U):
            seg = range(up["offsets"][u], up["offsets"][u + 1])
            toks = [pt[p] for p in seg]
            assert toks == sorted(toks)
            for p in seg:
                assert ids[pt[p], ps[p]] == up["unique"][u]
        for t in range(T):
            for j in range(k):
                p = inv[t * k + j]
                assert pt[p] == t and ps[p] == j


def test_union_empty_is_zero_ratio():
    up = ml.union_permute(np.zeros((0, 3), dtype=np.int32), 8)
    assert up["n_unique"] == 0 and up["reuse_ratio"] == 0.0 and up["offsets"].tolist() == [0]


def test_union_rejects_duplicates_and_range():
    with pytest.raises(ml.OracleError):
        ml.union_permute(np.array([[1, 1]], dtype=np.int32), 4)
    with pytest.raises(ml.OracleError):
        ml.union_permute(np.array([[1, 4]], dtype=np.int32), 4)


# ------------------------------------------------------------------ reuse bias
def _bias_case(name):
    g = load(name)
    lg = np.array(g["logits"], dtype=np.float32)
    wc = np.array(g["w_conf"], dtype=np.float32)
    return g, lg, wc


def test_reuse_bias_fig5_counts():
    g, lg, wc = _bias_case("reuse_bias_fig5.json")
    k, E = g["k"], g["E"]
    ex = g["expected"]
    ids0, _ = ml.route(lg, k)
    assert ids0.tolist() == ex["ids_before"]
    assert ml.union_permute(ids0, E)["n_unique"] == ex["union_before"] == 6
    lb = ml.reuse_bias(lg, wc, k, g["cap"], g["alpha"])
    biased_cols = sorted(set(np.nonzero((lb != lg).any(axis=0))[0].tolist()))
    assert biased_cols == ex["preferred_set"]
    ids1, _ = ml.route(lb, k)
    assert ids1.tolist() == ex["ids_after"]
    assert ml.union_permute(ids1, E)["n_unique"] == ex["union_after"] == 4
    assert lb[3].tolist() == ex["t4_biased_logits"]
    # high-confidence T1, T2 keep their experts (the page's Fig. 5 reading)
    assert ids1[0].tolist() == ids0[0].tolist() and ids1[1].tolist() == ids0[1].tolist()


def test_reuse_bias_weighting_and_lambda():
    g, lg, wc = _bias_case("reuse_bias_weighting.json")
    ex = g["expected"]
    lb = ml.reuse_bias(lg, wc, g["k"], g["cap"], g["alpha"])
    diff = lb.astype(np.float64) - lg.astype(np.float64)
    cols = sorted(set(np.nonzero((diff != 0).any(axis=0))[0].tolist()))
    assert cols == ex["preferred_set"]
    for b, lam in enumerate(ex["lambda"]):
        for e in cols:
            assert diff[b, e] == lam


def test_reuse_bias_invariants_random():
    rng = np.random.default_rng(3)
    for it in range(60):
        E = int(rng.integers(6, 64))
        k = int(rng.integers(1, min(8, E - 1) + 1))
        T = int(rng.integers(1, 9))
        cap = int(rng.integers(k, 3 * k + 1))
        lg = (rng.standard_normal((T, E)) - 0.05 * np.arange(E)).astype(np.float32)
        wc = rng.uniform(0, 1, T).astype(np.float32)
        wc[0] = 1.0
        ids0, _ = ml.route(lg, k)
        # alpha = 0 is the identity
        assert np.array_equal(ml.reuse_bias(lg, wc, k, cap, 0.0), lg)
        alpha = float(rng.choice([0.1, 0.25, 0.5, 1.0, 4.0]))
        lb = ml.reuse_bias(lg, wc, k, cap, alpha)
        ids1, _ = ml.route(lb, k)
        U0 = set(ids0.ravel().tolist())
        U1 = set(ids1.ravel().tolist())
        # S2-MoE: the bias only re-selects onto experts other tokens already chose
        assert U1 <= U0
        estar = set(np.nonzero((lb != lg).any(axis=0))[0].tolist())
        assert len(estar) <= cap and estar <= U0
        for t in range(T):
            # a token whose whole top-k lies in E* keeps its choice
            if set(ids0[t].tolist()) <= estar:
                assert ids1[t].tolist() == ids0[t].tolist()


# ------------------------------------------------------------------ FFN
def test_ffn_hand_value():
    g = load("ffn_hand.json")
    Wgu = np.array(g["W_gate"] + g["W_up"], dtype=np.float64)
    Wd = np.array(g["W_down"], dtype=np.float64)
    o = ml.ffn_token_slot(np.array(g["x"], dtype=np.float64), Wgu, Wd)
    np.testing.assert_allclose(o, g["o"], rtol=1e-15)


def test_silu_closed_forms():
    a = np.array([0.0, 1.0, -1.0, 40.0, -40.0, 3.5])
    s = ml.silu(a)
    assert s[0] == 0.0
    assert abs(s[1] - 1 / (1 + math.exp(-1))) < 1e-16
    assert abs(s[3] - 40.0) < 1e-12 and abs(s[4]) < 1e-15
    # silu(-a) = silu(a) - a
    np.testing.assert_allclose(ml.silu(-a), s - a, atol=1e-13)


def test_moe_layer_equals_dense_masked_evaluation():
    """Per-token MoE output equals dense evaluation of that token's own top-k experts:
    evaluate every expert on every token at once (einsum over all E) and mask the
    gate to the token's top-k weights."""
    rng = np.random.default_rng(4)
    E, H, I, T, k = 6, 8, 5, 4, 3
    Wgu = rng.standard_normal((E, 2 * I, H))
    Wd = rng.standard_normal((E, H, I))
    x = rng.standard_normal((T, H))
    lg = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = ml.route(lg, k)
    y = ml.moe_layer(x, ids, w, lambda e: (Wgu[e], Wd[e]))
    a = np.einsum("eih,th->tei", Wgu[:, :I], x)
    b = np.einsum("eih,th->tei", Wgu[:, I:], x)
    h = a / (1 + np.exp(-a)) * b
    o = np.einsum("ehi,tei->teh", Wd, h)
    gate = np.zeros((T, E))
    for t in range(T):
        gate[t, ids[t]] = w[t]
    ref = np.einsum("te,teh->th", gate, o)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_single_token_k1_is_plain_swiglu_mlp():
    rng = np.random.default_rng(5)
    H, I = 7, 4
    Wg, Wu, Wd = rng.standard_normal((I, H)), rng.standard_normal((I, H)), rng.standard_normal((H, I))
    x = rng.standard_normal((1, H))
    lg = np.array([[0.3, 2.0, -1.0]], dtype=np.float32)
    ids, w = ml.route(lg, 1)
    assert ids.tolist() == [[1]] and w.tolist() == [[1.0]]
    y = ml.moe_layer(x, ids, w, lambda e: (np.vstack([Wg, Wu]), Wd))
    g = Wg @ x[0]
    np.testing.assert_allclose(y[0], Wd @ (g * scipy.special.expit(g) * (Wu @ x[0])), rtol=1e-13)


# ------------------------------------------------------------------ bytes
def test_expert_bytes_page_arithmetic():
    # EcoSpec section 1: a DeepSeek FP8 expert is 44 MB of HBM traffic ...
    b = vs.expert_bytes(7168, 2048, "e4m3")
    assert 44.0e6 <= b <= 44.1e6
    # ... and 0.2 extra experts per layer over 61 MoE layers cost about 0.5 GB.
    extra = 0.2 * b * 61
    assert 0.5e9 <= extra <= 0.55e9
    # Table 2 DeepSeek-V3.1: 97.3 -> 96.8 GB is 0.5 GB for 31.4 -> 31.2 experts/layer.
    assert abs(0.2 * 61 * b / 1e9 - (97.3 - 96.8)) < 0.05
    assert vs.expert_bytes(4096, 1536, "bf16") == 37748736

"""Input-generator checks (host side)."""
import numpy as np
import torch

from workload import CONFIGS, make_workload, small_case
from workload import counter_hash as ch
from workload import gen


def test_splitmix64_published_vector():
    # Reference SplitMix64 outputs for seed 1234567 (Steele, Lea, Flood 2014;
    # the vector accompanying the public-domain reference implementation).
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    got = [ch.mix64_int(1234567 + (i + 1) * ch.GOLDEN) for i in range(5)]
    assert got == want
    arr = ch.hash_at(1234567, np.arange(5, dtype=np.uint64))
    assert [int(v) for v in arr] == want


def test_value_maps_exact():
    h = ch.hash_at(ch.stream_key(7, 3), np.arange(4096, dtype=np.uint64))
    v = ch.grid8_values(h)
    bits = ch.grid8_bf16_bits(h)
    assert np.array_equal(gen.bf16_bits_to_f32(bits), v)  # exact in bf16
    assert np.all(np.abs(v) <= 255 * 2.0 ** -13)
    c = ch.e4m3_codes(h)
    assert not np.any((c & 0x7F) == 0x7F)
    s = ch.scale_values(h)
    assert np.all((s >= 2.0 ** -13) & (s < 2.0 ** -12))


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.array([1.00390625, 1.01171875, -1.00390625, 0.0, -0.0], np.float32)])
    ours = gen.bf16_bits_rne(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_tree_and_footprints():
    for name in ("toy", "batched_qwen_like"):
        cfg = CONFIGS[name]
        if name != "toy":
            cfg = cfg.replace(L=2)
        wl = make_workload(cfg)
        par = wl.parent
        assert len(par) == 14 and all(par[t] < t for t in range(14))
        for s in range(cfg.nseq):
            for t in range(14):
                if par[t] >= 0:
                    assert wl.P[s, t] <= wl.P[s, par[t]]
                # k experts per layer in each own footprint
                bits = np.unpackbits(wl.own_fp[s, t].view(np.uint8), bitorder="little")
                per_layer = bits[: cfg.L * cfg.E].reshape(cfg.L, cfg.E).sum(axis=1)
                assert np.all(per_layer == cfg.k)
        assert wl.T == int(np.sum(wl.gamma + 1))
        if cfg.ragged:
            assert np.all((wl.gamma >= 0) & (wl.gamma <= cfg.gamma_max))


def test_expert_slice_regeneration():
    cfg = small_case()
    w3 = gen.expert_weights_host(cfg, 1, 3)
    keys = gen.weight_stream_keys(cfg, 1)
    full = ch.fill_host(gen.weight_kind(cfg), keys["gate_up"], 0, cfg.E * 2 * cfg.I * cfg.H)
    full = full.reshape(cfg.E, 2 * cfg.I, cfg.H)
    assert np.array_equal(full[3], w3["gate_up"])


def test_perturbed_footprints_accuracy_and_shape():
    import numpy as np
    from workload import gen
    cfg = gen.small_case("perturb", L=3, E=32, k=4, seed=4)
    wl = gen.make_workload(cfg)
    assert np.array_equal(gen.perturbed_footprints(wl, 1.0), wl.own_fp)
    for acc in (0.93, 0.82, 0.5, 0.0):
        fp = gen.perturbed_footprints(wl, acc, seed=1)
        kept = tot = 0
        for s in range(wl.P.shape[0]):
            for t in range(wl.P.shape[1]):
                for l in range(cfg.L):
                    lo, hi = l * cfg.E, (l + 1) * cfg.E
                    pred = {b - lo for b in range(lo, hi) if (fp[s, t, b // 32] >> (b % 32)) & 1}
                    true = {b - lo for b in range(lo, hi) if (wl.own_fp[s, t, b // 32] >> (b % 32)) & 1}
                    assert len(pred) == cfg.k  # still k distinct experts per layer
                    kept += len(pred & true)
                    tot += cfg.k
        assert abs(kept / tot - acc) < 0.08

"""GPU parity of moe_router_logits against the fp64 router oracle.

The kernel accumulates in fp32 with at most n = 8*ceil(H/1024) + 8 roundings
on any path from a product to a logit (fixed order: per-thread FMAs over its
8-element groups, a 5-level warp butterfly, 3 adds over the warps), so every
logit must lie within gamma_n * sum_h |x_h w_eh| of the exact value
(gamma_n = n u / (1 - n u), u = 2^-24).  The bound is tight enough that one
dropped or doubled term of typical size fails it.
"""
import ctypes
import math

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


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def make_inputs(T, H, E, xdt, wdt, seed):
    from workload import gen
    rng = np.random.default_rng(seed)
    xs = rng.standard_normal((T, H)).astype(np.float32)
    x_store = gen.bf16_bits_rne(xs).view(np.int16) if xdt == "bf16" else xs
    cfg = gen.MoEConfig("router_case", L=1, H=H, E=E, k=1, I=64,
                        dtype="bf16" if wdt == "bf16" else "f32", seed=seed)
    w_store = gen.router_weights_host(cfg, 0)
    if wdt == "bf16":
        w_store = w_store.view(np.int16)
    return x_store, w_store


def oracle_with_bound(x_store, w_store, xdt, wdt):
    from oracle import router as orr
    x = orr.decode(x_store, xdt)
    w = orr.decode(w_store, wdt)
    ref = orr.router_logits(x, w)
    H = x.shape[1]
    n = 8 * math.ceil(H / 1024) + 8
    u = 2.0 ** -24
    gamma = n * u / (1 - n * u)
    absdot = np.abs(x) @ np.abs(w).T
    return ref, gamma * absdot + 1e-12 * absdot


# Qwen-, GPT-OSS- and DeepSeek-like gates at full size, the batched token
# count, the toy fp32 gate, mixed dtypes, ragged token passes (T % 8 != 0),
# rows shorter than one pass of the CTA (H < 1024), partial chunks and long rows.
CASES = [(5, 4096, 128, "bf16", "bf16"), (5, 2880, 128, "bf16", "bf16"), (5, 7168, 256, "bf16", "bf16"),
         (24, 4096, 128, "bf16", "bf16"), (28, 4096, 128, "bf16", "bf16"), (5, 256, 16, "f32", "f32"),
         (37, 584, 3, "bf16", "f32"), (9, 2056, 7, "f32", "bf16"), (1, 8, 1, "bf16", "bf16"),
         (300, 1024, 64, "bf16", "bf16"), (3, 16384, 32, "f32", "f32"), (8, 4104, 1024, "bf16", "bf16")]


@pytest.mark.parametrize("T,H,E,xdt,wdt", CASES)
def test_router_logits_match_oracle(mv, T, H, E, xdt, wdt):
    xs, ws = make_inputs(T, H, E, xdt, wdt, seed=T * 7 + H + E)
    got = mv.router_logits(cuda(xs), cuda(ws))
    torch.cuda.synchronize()
    g = got.cpu().numpy().astype(np.float64)
    ref, bound = oracle_with_bound(xs, ws, xdt, wdt)
    err = np.abs(g - ref)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound)}"
    # the bound is not vacuous: it is well below a typical single term |x_h w_eh|
    from oracle import router as orr
    typical = np.mean(np.abs(orr.decode(xs, xdt))) * np.mean(np.abs(orr.decode(ws, wdt)))
    assert np.max(bound) < 0.25 * typical


def test_router_logits_deterministic(mv):
    xs, ws = make_inputs(24, 4096, 128, "bf16", "bf16", seed=3)
    x, w = cuda(xs), cuda(ws)
    a = mv.router_logits(x, w)
    b = mv.router_logits(x, w)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_router_then_route_ids(mv):
    """Ids chosen from the kernel's logits equal the oracle's wherever the
    oracle's ordering of the top k+1 logits is decided by more than the
    accumulation error (near-ties may legitimately resolve either way)."""
    from oracle import moe_layer as ml
    T, H, E, k = 28, 4096, 128, 8
    xs, ws = make_inputs(T, H, E, "bf16", "bf16", seed=11)
    logits = mv.router_logits(cuda(xs), cuda(ws))
    ids, _ = mv.route(logits, k)
    torch.cuda.synchronize()
    ref, bound = oracle_with_bound(xs, ws, "bf16", "bf16")
    rid, _ = ml.route(ref.astype(np.float32), k)
    gid = ids.cpu().numpy()
    decided = 0
    for t in range(T):
        top = np.sort(ref[t])[::-1][: k + 1]
        if np.min(top[:-1] - top[1:]) > 2 * np.max(bound[t]):
            decided += 1
            assert gid[t].tolist() == rid[t].tolist()
        else:
            assert len(set(gid[t].tolist())) == k
    assert decided >= T - 2


def test_router_empty_and_errors(mv):
    w = torch.zeros((16, 256), dtype=torch.int16, device="cuda")
    out = mv.router_logits(torch.zeros((0, 256), dtype=torch.int16, device="cuda"), w)
    assert out.shape == (0, 16)
    with pytest.raises(mv.MoEError):
        mv.router_logits(torch.zeros((2, 12), dtype=torch.int16, device="cuda"),
                         torch.zeros((4, 12), dtype=torch.int16, device="cuda"))
    with pytest.raises(mv.MoEError):
        mv.router_logits(torch.zeros((2, 64), dtype=torch.float32, device="cuda"),
                         torch.zeros((1025, 64), dtype=torch.float32, device="cuda"))
    # a misaligned activation pointer is refused on the host, before any launch
    from serving_router_softmax_gb300 import _lib as L
    lib = L.load()
    buf = torch.zeros((4, 72), dtype=torch.int16, device="cuda")
    lg = torch.empty((2, 16), dtype=torch.float32, device="cuda")
    cfg = L.RouterCfg(2, 64, 16, L.DTYPE_BF16, L.DTYPE_BF16)
    st = lib.moe_router_logits(buf.data_ptr() + 2, w.data_ptr(), ctypes.byref(cfg), lg.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == L.MOE_ERR_ARG


def test_router_nan_propagates_to_route_flag(mv):
    xs, ws = make_inputs(3, 256, 16, "f32", "f32", seed=5)
    xs = xs.copy()
    xs[1, 7] = np.nan
    logits = mv.router_logits(cuda(xs), cuda(ws))
    dev_err = mv.new_dev_err()
    ids, _ = mv.route(logits, 2, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() & 0x01
    assert ids[1].tolist() == [-1, -1]
    assert ids[0].min().item() >= 0 and ids[2].min().item() >= 0

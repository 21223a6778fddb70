"""moe_hot_list against the oracle's hot-list rule (S2-MoE write-up, system
implementation: hot experts from profiled activation frequencies): counts,
the hot list and the home-slot table must be bit-exact."""
import numpy as np
import pytest

from oracle import residency as R

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import serving_router_softmax_gb300 as m
    return m


CASES = [  # (E, n_ids, n_hot, first_slot, value range scale)
    (8, 40, 3, 0, 1), (16, 0, 4, 0, 1), (128, 5 * 8 * 16, 64, 0, 1), (128, 640, 0, 0, 1),
    (128, 640, 128, 0, 1), (256, 20000, 200, 37, 1), (1000, 4000, 333, 5, 1), (4096, 100000, 1024, 0, 1),
    (4096, 3000, 4095, 9, 1), (33, 999, 17, 0, 1), (64, 64 * 3, 20, 0, 0)]


@pytest.mark.parametrize("E,n,n_hot,first,skew", CASES)
def test_hot_list_matches_oracle(mv, E, n, n_hot, first, skew):
    rng = np.random.default_rng(E * 7 + n + n_hot)
    if skew:
        # skewed popularity with many equal counts (ties to the lower id)
        p = np.exp(-0.05 * rng.permutation(E))
        ids = rng.choice(E, size=n, p=p / p.sum()).astype(np.int32)
    else:
        ids = np.repeat(np.arange(E, dtype=np.int32), 3)[:n]  # every count equal
    if n:
        ids[rng.random(n) < 0.1] = -1  # ignored entries
    dev_err = mv.new_dev_err()
    hot, counts, home = mv.hot_list(torch.from_numpy(ids).cuda(), E, n_hot, first_slot=first, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    want_counts = R.activation_counts(ids, E)
    want_hot = R.hot_experts(want_counts, n_hot)
    assert counts.cpu().tolist() == want_counts.tolist()
    assert hot.cpu().tolist() == want_hot
    assert home.cpu().tolist() == R.home_slots(want_hot, E, first).tolist()


def test_hot_list_flags_bad_ids_and_skips_them(mv):
    ids = torch.tensor([0, 1, 1, 7, -3, 2, 2, 2], dtype=torch.int32, device="cuda")
    dev_err = mv.new_dev_err()
    hot, counts, home = mv.hot_list(ids, 4, 2, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() & mv._lib.DEV_BAD_ID
    assert counts.cpu().tolist() == [1, 2, 3, 0]
    assert hot.cpu().tolist() == [1, 2]


def test_hot_list_host_validation(mv):
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(mv.MoEError):
        mv.hot_list(ids, 4097, 1)
    with pytest.raises(mv.MoEError):
        mv.hot_list(ids, 8, 9)

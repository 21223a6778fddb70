"""Pins of the expert-residency oracle (hot list, staging plan) against hand-worked cases and invariants."""
import numpy as np
import pytest

from oracle import residency as R


def test_hot_list_by_count_ties_to_lower_id():
    counts = [5, 9, 9, 0, 3]
    assert R.hot_experts(counts, 0) == []
    assert R.hot_experts(counts, 1) == [1]          # 9 vs 9: the lower id
    assert R.hot_experts(counts, 2) == [1, 2]
    assert R.hot_experts(counts, 3) == [0, 1, 2]
    assert R.hot_experts(counts, 5) == [0, 1, 2, 3, 4]
    assert R.hot_experts([1, 1, 1, 1], 2) == [0, 1]
    assert R.hot_experts([0, 2, 7, 2], 2) == [1, 2]  # 2 vs 2 for the second place: id 1 before id 3
    with pytest.raises(ValueError):
        R.hot_experts(counts, 6)


def test_activation_counts_hand():
    ids = np.array([[0, 3], [3, 1], [-1, 3]])
    assert R.activation_counts(ids, 5).tolist() == [1, 1, 0, 3, 0]


def test_home_slots():
    home = R.home_slots([1, 4], 6, first_slot=10)
    assert home.tolist() == [-1, 10, -1, -1, 11, -1]


def test_stage_plan_hand():
    # E = 8; experts 1 and 4 resident in slots 0 and 1; slots 2..4 stage.
    home = R.home_slots([1, 4], 8)
    slot_of, staged, errors = R.stage_plan([0, 1, 3, 4, 6], home, n_slots=5, stage_first=2, n_stage=3)
    assert slot_of == {0: 2, 1: 0, 3: 3, 4: 1, 6: 4}
    assert staged == [0, 3, 6]
    assert errors == []
    assert R.staged_bytes([0, 1, 3, 4, 6], home, 100) == 300


def test_stage_plan_staging_range_may_sit_first():
    # Shared staging first, this layer's resident experts after it.
    home = R.home_slots([2], 4, first_slot=2)
    slot_of, staged, errors = R.stage_plan([0, 2, 3], home, n_slots=3, stage_first=0, n_stage=2)
    assert slot_of == {0: 0, 2: 2, 3: 1}
    assert staged == [0, 3] and errors == []


def test_stage_plan_capacity():
    home = R.home_slots([1, 4], 8)
    slot_of, staged, errors = R.stage_plan([0, 1, 3, 4, 6], home, n_slots=4, stage_first=2, n_stage=2)
    assert slot_of == {0: 2, 1: 0, 3: 3, 4: 1, 6: -1}
    assert staged == [0, 3]
    assert errors == ["capacity"]


def test_stage_plan_bad_home_and_id():
    home = R.home_slots([1, 4], 8)
    home[3] = 2  # inside the staging range
    home[5] = 9  # outside the pool
    slot_of, staged, errors = R.stage_plan([1, 3, 5, 6, 8], home, n_slots=5, stage_first=2, n_stage=3)
    assert slot_of == {1: 0, 3: -1, 5: -1, 6: 2}
    assert staged == [6]
    assert errors == ["bad_id"]


def test_stage_plan_invariants_random():
    rng = np.random.default_rng(5)
    for _ in range(200):
        E = int(rng.integers(1, 40))
        n_hot = int(rng.integers(0, E + 1))
        hot = sorted(rng.choice(E, size=n_hot, replace=False).tolist())
        n_stage = int(rng.integers(0, E + 1))
        home = R.home_slots(hot, E)
        n_slots = n_hot + n_stage
        U = int(rng.integers(0, E + 1))
        unique = sorted(rng.choice(E, size=U, replace=False).tolist())
        slot_of, staged, errors = R.stage_plan(unique, home, n_slots, n_hot, n_stage)
        cold = [e for e in unique if e not in hot]
        assert set(slot_of) == set(unique)
        if len(cold) <= n_stage:
            assert errors == []
            assert staged == cold
            slots = [slot_of[e] for e in unique]
            assert len(set(slots)) == len(slots)
            assert all(0 <= s < n_slots for s in slots)
            for e in unique:
                assert slot_of[e] == (hot.index(e) if e in hot else n_hot + cold.index(e))
        else:
            assert errors == ["capacity"]
            assert staged == cold[:n_stage]
            assert [slot_of[e] for e in cold[n_stage:]] == [-1] * (len(cold) - n_stage)

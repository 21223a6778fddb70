"""CPU oracle: expert-level residency (hot list and on-demand staging).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

Source: S2-MoE write-up, "system implementation: expert-level offloading in
llama.cpp".  The non-expert parameters and the frequently activated experts
stay in device memory; every other expert is fetched on demand when a token
needs it; with spare device memory, a hot-expert list found by offline
profiling of activation frequencies decides which experts stay resident.
Residency does not change what the layer computes: the FFN of a layer with a
pool equals the FFN of the fully resident layer (``oracle.moe_layer``).

Readings where the page is silent (the CUDA path applies the same ones):
* The hot list is the n_hot experts with the highest activation counts over
  the profiled routing decisions; equal counts go to the lower expert id.
* The fetch unit is one expert of one layer, and the layer's union (the
  experts its verify tokens route to) is what must be present before the
  FFN.  Cold experts of the union are staged in union order (ascending expert
  id, the order the union is written in): the c-th cold expert takes staging
  slot stage_first + c.  More cold experts than staging slots is an error;
  the excess get no slot.
* A resident expert keeps its home slot; a home slot inside the staging range
  or outside the pool is an error (that expert gets no slot).

Parity: pinned (tests/test_oracle_residency.py: hand-worked hot lists with
tied counts, activation counts and home slots, hand-worked staging plans
including a staging range placed first, the capacity limit and bad homes or
ids, and random plans against the invariants every plan must satisfy).
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np


def hot_experts(counts: Sequence[int], n_hot: int) -> List[int]:
    """The n_hot most frequently activated experts, by count, ties to the lower id; ascending id order."""
    counts = [int(c) for c in counts]
    if n_hot < 0 or n_hot > len(counts):
        raise ValueError("n_hot outside [0, E]")
    order = sorted(range(len(counts)), key=lambda e: (-counts[e], e))
    return sorted(order[:n_hot])


def activation_counts(ids: np.ndarray, E: int) -> np.ndarray:
    """Per-expert activation counts of a set of routing decisions (ids: any shape, -1 ignored)."""
    counts = np.zeros(E, dtype=np.int64)
    for e in np.asarray(ids).reshape(-1):
        if e >= 0:
            counts[int(e)] += 1
    return counts


def home_slots(hot: Sequence[int], E: int, first_slot: int = 0) -> np.ndarray:
    """Home-slot table: hot expert hot[j] lives in slot first_slot + j, every other expert is cold (-1)."""
    home = np.full(E, -1, dtype=np.int64)
    for j, e in enumerate(hot):
        home[int(e)] = first_slot + j
    return home


def stage_plan(unique: Sequence[int], home_slot: Sequence[int], n_slots: int, stage_first: int,
               n_stage: int) -> Tuple[Dict[int, int], List[int], List[str]]:
    """Slot of every union expert, the cold experts staged (in staging-slot order) and the errors seen.

    unique: the layer's union in the order it is written (ascending ids).
    Returns (slot_of, staged, errors): slot_of[e] is the slot the FFN reads
    expert e from (-1 for none); staged[c] is the expert copied into slot
    stage_first + c; errors holds "capacity" and/or "bad_id".
    """
    E = len(home_slot)
    slot_of: Dict[int, int] = {}
    staged: List[int] = []
    errors: List[str] = []
    n_cold = 0
    for e in unique:
        e = int(e)
        if e < 0 or e >= E:
            errors.append("bad_id")
            continue
        h = int(home_slot[e])
        if h == -1:
            if n_cold < n_stage:
                slot_of[e] = stage_first + n_cold
                staged.append(e)
            else:
                slot_of[e] = -1
                errors.append("capacity")
            n_cold += 1
        elif 0 <= h < n_slots and not (stage_first <= h < stage_first + n_stage):
            slot_of[e] = h
        else:
            slot_of[e] = -1
            errors.append("bad_id")
    return slot_of, staged, sorted(set(errors))


def staged_bytes(unique: Sequence[int], home_slot: Sequence[int], bytes_per_expert: int) -> int:
    """Bytes one layer moves from host memory: its union's cold experts times the bytes of one expert."""
    return sum(bytes_per_expert for e in unique if int(home_slot[int(e)]) == -1)

"""CPU oracle: EcoSpec cost-aware draft selection.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

Source: EcoSpec write-up ("Less Experts, Faster Decoding: Cost-Aware
Speculative Decoding for MoE"), section 3.2 (the expert buffer B, rebuilt from
the empty set every speculative step) and section 3.3 (the score
S(t) = P(t) / (|E_traj(t) \\ B| + eps), the greedy loop that picks the argmax,
adds it to S and merges its footprint into B until gamma nodes are chosen, and
the prefix-consistency argument).  Section 4.3 defines the static ablation:
the score's denominator is the size of the node's whole path footprint, not
updated by B.

Readings where the page is silent:
* E_traj(t) is the union of the own footprints of the draft nodes on the path
  from the root's child down to t (the root token's own footprint is not
  pre-seeded into B, since B starts empty).
* argmax ties go to the lower breadth-first node index (the page's loop takes
  the first maximum; we iterate in node order).
* gamma larger than the number of nodes selects every node.
* Scores are compared exactly: P is an fp32 number and eps a power of two, so
  every score is a rational number; we compare them with Python Fractions.

* Batch (``select_batch_global``; the page's batch ablation in section 4.3
  gives no algorithm): one buffer B shared by all sequences of the batch, and
  one greedy over the forest of their draft trees with the budget
  sum(gamma_i) and at most ``cap`` nodes per sequence.  Each sequence's depth
  is an outcome of the greedy (confident sequences whose experts overlap get
  more nodes), in the spirit of the width-vs-depth note's confidence gating.
  Ties go to the lower (sequence, node) index.

Parity: pinned (tests/test_oracle_eco.py: hand-worked trees, static mode equal
to a sort by static score, prefix closure, union bookkeeping, aggregate
marginal-vs-static comparison over seeded trees; batch mode: one sequence
equals the per-sequence greedy, a hand-worked batch, budget and cap
bookkeeping).
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Sequence, Set, Tuple

import numpy as np


def footprint_set(bits: np.ndarray, E: int) -> Set[Tuple[int, int]]:
    """(layer, expert) pairs of a uint32 bitset; bit l*E+e marks (l, e)."""
    out = set()
    for w, word in enumerate(np.asarray(bits, dtype=np.uint32).tolist()):
        b = 0
        while word:
            if word & 1:
                idx = 32 * w + b
                out.add((idx // E, idx % E))
            word >>= 1
            b += 1
    return out


def trajectory_footprints(parent: Sequence[int], own: List[Set]) -> List[Set]:
    """E_traj(t): union of own footprints along the path to t (section 3.3)."""
    traj: List[Set] = []
    for t, p in enumerate(parent):
        path_set = set(own[t])
        q = p
        while q >= 0:
            path_set |= own[q]
            q = parent[q]
        traj.append(path_set)
    return traj


def ecospec_select(P: Sequence[float], traj: List[Set], gamma: int, eps: float,
                   mode: int = 0) -> Tuple[List[int], Set]:
    """The literal greedy of section 3.3.

    mode 0: marginal cost |E_traj(t) \\ B|.  mode 1: static cost |E_traj(t)|.
    Returns (selected nodes in selection order, final buffer B).
    """
    n = len(P)
    S: List[int] = []
    chosen = set()
    B: Set = set()
    eps_q = Fraction(eps)
    Pq = [Fraction(float(np.float32(p))) for p in P]
    while len(S) < min(gamma, n):
        best = None
        best_score = None
        for t in range(n):
            if t in chosen:
                continue
            cost = len(traj[t] - B) if mode == 0 else len(traj[t])
            score = Pq[t] / (cost + eps_q)
            if best is None or score > best_score:
                best, best_score = t, score
        S.append(best)
        chosen.add(best)
        B |= traj[best]
    return S, B


def select_batch(P: np.ndarray, parent: np.ndarray, own_fp: np.ndarray, E: int,
                 gamma: Sequence[int], eps: float, mode: int = 0):
    """Independent selection per sequence (each with its own B and gamma_i).

    Returns (list of selected lists, list of union sizes |B|).
    """
    sels, sizes = [], []
    for s in range(P.shape[0]):
        own = [footprint_set(own_fp[s, t], E) for t in range(P.shape[1])]
        traj = trajectory_footprints([int(p) for p in parent], own)
        sel, B = ecospec_select(P[s].tolist(), traj, int(gamma[s]), eps, mode)
        sels.append(sel)
        sizes.append(len(B))
    return sels, sizes


def select_batch_global(P: np.ndarray, parent: np.ndarray, own_fp: np.ndarray, E: int,
                        gamma: Sequence[int], eps: float, cap: int):
    """Batch-global marginal selection (see the module notes).

    Returns (per-sequence selected lists in selection order, per-sequence
    union sizes of their own selected trajectories, batch union size |B|).
    """
    nseq, n = P.shape
    par = [int(p) for p in parent]
    trajs = []
    for s in range(nseq):
        own = [footprint_set(own_fp[s, t], E) for t in range(n)]
        trajs.append(trajectory_footprints(par, own))
    eps_q = Fraction(eps)
    Pq = [[Fraction(float(np.float32(p))) for p in P[s]] for s in range(nseq)]
    cap = min(cap, n)
    budget = sum(min(max(int(g), 0), n) for g in gamma)
    sels: List[List[int]] = [[] for _ in range(nseq)]
    chosen = set()
    B: Set = set()
    for _ in range(budget):
        best, best_score = None, None
        for s in range(nseq):
            if len(sels[s]) >= cap:
                continue
            for t in range(n):
                if (s, t) in chosen:
                    continue
                score = Pq[s][t] / (len(trajs[s][t] - B) + eps_q)
                if best is None or score > best_score:
                    best, best_score = (s, t), score
        if best is None:
            break
        s, t = best
        sels[s].append(t)
        chosen.add(best)
        B |= trajs[s][t]
    sizes = []
    for s in range(nseq):
        U: Set = set()
        for t in sels[s]:
            U |= trajs[s][t]
        sizes.append(len(U))
    return sels, sizes, len(B)

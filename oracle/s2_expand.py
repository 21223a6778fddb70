"""CPU oracle: S2-MoE routing-aware adaptive speculative expansion.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

Source: S2-MoE write-up, component 1 (routing-aware adaptive speculative
expansion).  Adding draft token i to the selected set S costs the target model
|E_i minus the union of E_j over j in S| new experts, each priced at T_exp, plus
the draft-side cost C_draft of extending it; its utility is the expected gain
p_i * T_AR over that cost; candidates are examined in draft-generation order
and every one whose utility is at least 1 is taken, until no candidate
qualifies.

Readings where the page is silent (the CUDA path applies the same ones):
* The page drafts a chain; on a draft tree a node is a candidate once its
  parent is selected (children of the root always are), which keeps the
  selection prefix-closed as verification needs.
* "Until no candidate qualifies": passes over the nodes in breadth-first
  (draft) order repeat until a pass takes nothing.  Taking a node only shrinks
  the other nodes' costs and only makes more nodes candidates, so the selected
  set is the least fixed point of a monotone rule and does not depend on the
  order in which candidates are examined; it is returned in node order.
* E_i is node i's own predicted footprint over all layers (bit l*E + e), p_i
  its path probability P, and C_draft one constant per token.
* U_i >= 1 is evaluated as p_i * T_AR >= n_new * T_exp + C_draft in fp64, in
  this operation order (the product p_i * T_AR and n_new * T_exp are exact, the
  addition rounds once).  The cross-multiplied form also covers a zero cost
  (utility +inf: the node is taken).
* A NaN or negative P, or a parent outside [-1, t), is an error: nothing is
  selected.
* Expert residency (the write-up's system implementation offloads experts
  and calibrates the expert cost from the expert's bytes and the bandwidth
  it is moved at): with a set of non-resident (cold) experts, every new
  expert that is also cold adds T_cold, the time to bring it over the host
  link: cost = (n_new * T_exp + n_new_cold * T_cold) + C_draft, in fp64 in
  that order.  No cold set, or T_cold = 0, gives the plain rule.

Parity: pinned (tests/test_oracle_s2.py: a hand-worked tree, the T_exp = 0
closed form (a plain confidence threshold), order independence against a
simultaneous-update iteration, prefix closure and the union bookkeeping).
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Set, Tuple

import numpy as np

from .eco_select import footprint_set


class S2Error(ValueError):
    pass


def s2_expand(P: Sequence[float], parent: Sequence[int], own_fp: np.ndarray, E: int, T_AR: float,
              T_exp: float, C_draft: float, T_cold: float = 0.0,
              cold: Optional[Set[Tuple[int, int]]] = None) -> Tuple[List[int], int]:
    """Selected nodes (ascending) and the size of the union of their footprints.

    cold: the (layer, expert) pairs that are not resident (None: all resident)."""
    N = len(parent)
    for t in range(N):
        if not (-1 <= parent[t] < t):
            raise S2Error("parent outside [-1, t)")
        if not (np.float32(P[t]) >= 0):
            raise S2Error("P is NaN or negative")
    own = [footprint_set(own_fp[t], E) for t in range(N)]
    t_ar = np.float64(np.float32(T_AR))
    t_exp = np.float64(np.float32(T_exp))
    c_draft = np.float64(np.float32(C_draft))
    t_cold = np.float64(np.float32(T_cold))
    cold = set() if cold is None else set(cold)
    gain = [np.float64(np.float32(P[t])) * t_ar for t in range(N)]
    chosen = [False] * N
    B = set()
    changed = True
    while changed:
        changed = False
        for i in range(N):  # draft order
            if chosen[i]:
                continue
            if parent[i] >= 0 and not chosen[parent[i]]:
                continue
            new = own[i] - B
            n_new = len(new)
            n_cold = len(new & cold)
            cost = (np.float64(n_new) * t_exp + np.float64(n_cold) * t_cold) + c_draft
            if gain[i] >= cost:
                chosen[i] = True
                B |= own[i]
                changed = True
    return [t for t in range(N) if chosen[t]], len(B)


def s2_expand_batch(P: np.ndarray, parent: Sequence[int], own_fp: np.ndarray, E: int, T_AR: float,
                    T_exp: float, C_draft: float, T_cold: float = 0.0,
                    cold: Optional[Set[Tuple[int, int]]] = None):
    """Independent expansion per sequence: P [nseq, N], own_fp [nseq, N, W]."""
    sels, sizes = [], []
    for s in range(P.shape[0]):
        sel, size = s2_expand(P[s], parent, own_fp[s], E, T_AR, T_exp, C_draft, T_cold, cold)
        sels.append(sel)
        sizes.append(size)
    return sels, sizes

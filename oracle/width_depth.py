"""CPU oracle: width versus depth, and the confidence-gated depth vector.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

Source: the width-vs-depth note ("AI模型宽深之辩：边际权衡探析").

* Section 1 (depth can be cheaper than width): verifying d consecutive
  positions of one sequence touches fewer distinct experts than verifying d
  tokens of d random sequences, because consecutive tokens co-activate
  experts.  ``layer_unions`` gives the per-layer union size of a set of
  verify tokens from their router logits (the union of their top-k sets, as
  in the EcoSpec write-up, section 2).

* Section 2 (where to spend depth): each step, choose a depth vector d (one
  speculation depth per live sequence) that maximises the expected batch
  throughput; in practice first pick one batch-common depth from the live
  sequences' confidences, then greedily truncate sequences whenever that
  raises the expected throughput.  The draft's confidence at each depth is
  the cumulative product of its per-token confidences, and the note finds it
  calibrated against the committed length.

Readings where the note is silent (the CUDA path applies the same ones):
* Expected committed tokens of sequence i verified to depth d_i:
  A_i(d_i) = 1 + c_i1 + ... + c_id_i, with c_ij the cumulative confidence at
  depth j (the probability that the first j drafts are all accepted, under
  calibration) and 1 for the token the verify step always yields.
* Expected step cost: the verify-cost model this library calibrates (the
  S2-MoE write-up, component 1: cost grows by T_exp per unique expert),
  cost(d) = C0 + T_exp * U(d), U(d) = number of distinct (layer, expert)
  pairs in the union of the predicted footprints of every verified position
  (each root token, position 0, always; positions 1..d_i of sequence i).
* Throughput(d) = sum_i A_i(d_i) / cost(d).
* Batch-common depth: d_i = min(D', max_i) for D' = 0..D; the largest
  throughput wins, equal throughputs go to the smaller D'.
* Greedy truncation: repeatedly take the single decrement d_i -> d_i - 1
  (d_i > 0) with the largest throughput, if it is strictly larger than the
  current one (equal candidates go to the lower i); stop when none is.
* Arithmetic: fp64, in this order: A_i(j) = A_i(j-1) + c_ij from A_i(0) = 1;
  num = sum over i ascending of A_i(d_i) starting from 0; den =
  C0 + (T_exp * U); throughput = num / den (IEEE operations, each rounded
  once, no fused multiply-add).  Confidences and the cost parameters are fp32
  values, converted exactly.

Parity: pinned (tests/test_oracle_width_depth.py: the expected committed
length against brute-force enumeration of acceptance outcomes; a hand-worked
two-sequence batch; one sequence against exhaustive search; T_exp = 0 and
zero-confidence closed forms; local optimality and no loss against the
common depth; union sizes against hand-counted top-k sets).
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Set

import numpy as np

from .moe_layer import topk_order


def layer_unions(logits: np.ndarray, k: int) -> List[int]:
    """Union size per layer of the tokens' top-k sets; logits [L, T, E]."""
    out = []
    for l in range(logits.shape[0]):
        u: Set[int] = set()
        for t in range(logits.shape[1]):
            u |= set(topk_order(logits[l, t], k))
        out.append(len(u))
    return out


def _bits(words: Sequence[int]) -> Set[int]:
    s = set()
    for w, word in enumerate(int(x) for x in words):
        b = 0
        while word:
            if word & 1:
                s.add(32 * w + b)
            word >>= 1
            b += 1
    return s


def expected_accepted(conf_row: Sequence[float], d: int) -> float:
    """A_i(d) = 1 + c_1 + ... + c_d in fp64, summed in depth order."""
    a = 1.0
    for j in range(d):
        a = a + float(np.float32(conf_row[j]))
    return a


class DepthModel:
    """Expected throughput of a depth vector (readings in the module notes)."""

    def __init__(self, conf: np.ndarray, fp: np.ndarray, C0: float, T_exp: float):
        self.conf = np.asarray(conf, dtype=np.float32)
        nseq, D = self.conf.shape
        self.nseq, self.D = nseq, D
        # prefix unions: pre[i][j] = footprints of positions 0..j of sequence i
        self.pre: List[List[Set[int]]] = []
        for i in range(nseq):
            acc: Set[int] = set()
            row = []
            for j in range(D + 1):
                acc = acc | _bits(fp[i, j])
                row.append(acc)
            self.pre.append(row)
        self.A = [[expected_accepted(self.conf[i], j) for j in range(D + 1)] for i in range(nseq)]
        self.C0 = float(np.float32(C0))
        self.T_exp = float(np.float32(T_exp))

    def union(self, d: Sequence[int]) -> int:
        u: Set[int] = set()
        for i, di in enumerate(d):
            u |= self.pre[i][di]
        return len(u)

    def throughput(self, d: Sequence[int]) -> float:
        num = 0.0
        for i, di in enumerate(d):
            num = num + self.A[i][di]
        den = self.C0 + (self.T_exp * float(self.union(d)))
        return num / den


def depth_policy(conf: np.ndarray, fp: np.ndarray, C0: float, T_exp: float,
                 max_depth: Optional[Sequence[int]] = None) -> Dict:
    """Confidence-gated depth vector (width-vs-depth note, section 2).

    conf [nseq, D] cumulative confidences (fp32, in [0, 1]); fp [nseq, D+1, W]
    uint32 predicted footprints (position 0 = the root token); C0, T_exp the
    cost model (fp32, finite, C0 > 0, T_exp >= 0);
    max_depth [nseq] per-sequence limits in [0, D] (default D).
    Returns {"depth": d, "common": D*, "thr_common", "thr"}.
    """
    c = np.asarray(conf, dtype=np.float32)
    if not np.all((c >= 0) & (c <= 1)):
        raise ValueError("confidences must lie in [0, 1]")
    if not (np.isfinite(np.float32(C0)) and np.float32(C0) > 0 and np.isfinite(np.float32(T_exp))
            and np.float32(T_exp) >= 0):
        raise ValueError("need C0 > 0 and T_exp >= 0, finite")
    m = DepthModel(conf, fp, C0, T_exp)
    nseq, D = m.nseq, m.D
    lim = [D] * nseq if max_depth is None else [min(max(int(v), 0), D) for v in max_depth]
    best_D, best_t = 0, None
    for Dc in range(D + 1):
        t = m.throughput([min(Dc, lim[i]) for i in range(nseq)])
        if best_t is None or t > best_t:
            best_D, best_t = Dc, t
    d = [min(best_D, lim[i]) for i in range(nseq)]
    thr_common = best_t
    cur = best_t
    while True:
        pick, pick_t = -1, cur
        for i in range(nseq):
            if d[i] == 0:
                continue
            cand = list(d)
            cand[i] -= 1
            t = m.throughput(cand)
            if t > pick_t:
                pick, pick_t = i, t
        if pick < 0:
            break
        d[pick] -= 1
        cur = pick_t
    return {"depth": d, "common": best_D, "thr_common": thr_common, "thr": cur}

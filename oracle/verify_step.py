"""CPU oracle: the whole speculative verify step and its byte accounting.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

Step (EcoSpec write-up section 2, the three steps of a round, and section 3):
1. per sequence, select gamma_i draft nodes with the cost-aware greedy;
2. the verify tokens of sequence i are its root token followed by its selected
   nodes in selection order; sequences are concatenated;
3. every MoE layer routes the verify tokens (optionally with the S2-MoE reuse
   bias, confidence weight w_b = the token's path probability, 1 for the root),
   forms the expert union and runs the SwiGLU experts and the weighted combine.

Byte accounting: an expert of hidden size H and intermediate size I stores
3*H*I weights (gate, up, down); FP8 experts add one fp32 scale per 128x128
block.  The EcoSpec write-up's figures pin this: a DeepSeek FP8 expert is
44 MB (section 1), and 0.2 extra experts per layer over 61 MoE layers cost
about 0.5 GB per round (section 1).

Parity: pinned (tests/test_oracle_step.py: hand-worked two-sequence forest for
the per-sequence, static and batch-global selections; verify rows root first
then the selected nodes in selection order; bias confidences 1 for a root and
the path probability for a node, checked through a hand-derived preferred set
that other weightings would change; the token-subset switch touching only the
FFN rows; tests/test_oracle_moe.py: the page's byte arithmetic).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

from . import eco_select as eco
from . import moe_layer as ml


def expert_bytes(H: int, I: int, dtype: str) -> int:
    """Weight bytes of one SwiGLU expert (gate + up + down), plus FP8 block scales."""
    elem = {"f32": 4, "bf16": 2, "e4m3": 1}[dtype]
    b = 3 * H * I * elem
    if dtype == "e4m3":
        b += 4 * (math.ceil(2 * I / 128) * math.ceil(H / 128) + math.ceil(H / 128) * math.ceil(I / 128))
    return b


def verify_rows(parent_len: int, sels: List[List[int]]) -> List[int]:
    """Row of each verify token in the [nseq, N+1] node table (row 0 = root)."""
    rows = []
    for s, sel in enumerate(sels):
        base = s * (parent_len + 1)
        rows.append(base)
        rows.extend(base + 1 + t for t in sel)
    return rows


def token_conf(P: np.ndarray, sels: List[List[int]]) -> np.ndarray:
    """Confidence weight of each verify token: its path probability, 1 for a root."""
    out = []
    for s, sel in enumerate(sels):
        out.append(np.float32(1.0))
        out.extend(np.float32(P[s, t]) for t in sel)
    return np.array(out, dtype=np.float32)


def run_selection(wl, mode: Optional[int] = None, cap: Optional[int] = None):
    """Per-sequence selection (modes 0, 1) or batch-global (mode 2, with at
    most ``cap`` nodes per sequence; default the largest gamma_i)."""
    cfg = wl.cfg
    mode = cfg.mode if mode is None else mode
    if mode == 2:
        cap = int(np.max(wl.gamma)) if cap is None else cap
        sels, sizes, _ = eco.select_batch_global(wl.P, wl.parent, wl.own_fp, cfg.E, wl.gamma, cfg.eps, cap)
        return sels, sizes
    return eco.select_batch(wl.P, wl.parent, wl.own_fp, cfg.E, wl.gamma, cfg.eps, mode)


def run_step(wl, experts_for_layer, layers: Optional[Sequence[int]] = None,
             tokens: Optional[Sequence[int]] = None, x_decode=None) -> Dict:
    """Oracle verify step.

    ``experts_for_layer(l)`` returns a callable e -> (W_gate_up, W_down) in fp64.
    ``x_decode`` maps stored hidden states to fp64.  ``tokens`` restricts the
    FFN (not the routing) to a sample of verify tokens.
    """
    cfg = wl.cfg
    sels, sizes = run_selection(wl)
    rows = verify_rows(wl.parent.shape[0], sels)
    conf = token_conf(wl.P, sels)
    L = cfg.L
    layers = list(range(L)) if layers is None else list(layers)
    per_layer = {}
    for l in layers:
        lg = wl.logits[l].reshape(-1, cfg.E)[rows]
        xs = wl.x[l].reshape(-1, cfg.H)[rows]
        x64 = x_decode(xs)
        per_layer[l] = ml.layer_forward(lg, x64, cfg.k, cfg.E, experts_for_layer(l),
                                        w_conf=conf if cfg.use_bias else None,
                                        cap=cfg.cap, alpha=cfg.alpha, tokens=tokens)
    return {"selected": sels, "union_size": sizes, "rows": rows, "conf": conf,
            "layers": per_layer}

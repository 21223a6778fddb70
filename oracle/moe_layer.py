"""CPU oracle: one MoE layer of the speculative verify step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

What it computes, with the passages it follows:

* ``route``: per token, softmax over the E gate logits, keep the top-k experts
  and their weights (EcoSpec write-up section 3.1, the predictor's
  "softmax, then top-K per layer" routing form; section 2, S_l(x_t) is the
  set a token routes to; S2-MoE write-up, background: each token passes only
  the router's top-k experts).  Weights are the softmax over the k selected
  logits, in fp64 (equal to renormalising the full softmax over the selected
  experts).
* ``reuse_bias``: S2-MoE write-up, component 2 (reuse-aware expert gating),
  steps 1-3 and the Fig. 5 walk-through.  The formulas were lost from the page;
  the reading used (also applied by the CUDA path) is, in fp32 with this op
  order:
    g_e   = sum over b ascending of w_b * [e in TopK(l_b)]   (plain adds)
    E*    = the `cap` experts with the largest g_e among g_e > 0
    lam_b = alpha * (l_b,(1) - l_b,(k+1))
    l'_b,e = l_b,e + lam_b  for e in E*, else l_b,e
  and the biased logits go through the unchanged router.
* ``union_permute``: the verify expert set is the union of the tokens' top-k
  sets (EcoSpec write-up section 2, the union formula); per-expert token groups
  in expert-ascending, token-ascending order; reuse ratio
  |union| / (s * k) with s the number of tokens (S2-MoE write-up, challenge 2).
* ``ffn_token_slot``: the expert FFN on one token, SwiGLU
  o = W_d (silu(W_g x) * (W_u x)), silu(a) = a / (1 + e^-a), in fp64 on the
  exactly decoded stored weights.
* ``moe_layer``: y_t = sum over slots j = 0..k-1 (in that order) of
  w_tj * FFN_{e(t,j)}(x_t).

Readings where the pages are silent: ties in top-k go to the lower expert id;
-0.0 equals +0.0; a NaN logit is an error; slot order is descending logit.

Parity: pinned (tests/test_oracle_moe.py: hand-derived routing and FFN
values, closed forms, union bounds and special cases, bias invariants and the
Fig. 5 counts, FP8/bf16 decoding against the format definitions).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np


class OracleError(ValueError):
    pass


# ----------------------------------------------------------------- decoding
def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp64 (bf16 is the top half of an IEEE fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _e4m3_value(c: int) -> float:
    """OCP FP8 E4M3 code -> value: sign, 4 exponent bits (bias 7), 3 mantissa
    bits, subnormals at exponent 0, S.1111.111 is NaN, no infinities."""
    sign = -1.0 if c & 0x80 else 1.0
    ex = (c >> 3) & 0xF
    man = c & 0x7
    if ex == 0xF and man == 0x7:
        return float("nan")
    if ex == 0:
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (ex - 7)


_E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """FP8 E4M3 codes -> fp64, through the 256-entry table of ``_e4m3_value``."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def expert_matrices(w: Dict[str, np.ndarray], dtype: str) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 (W_gate_up [2I, H], W_down [H, I]) from one expert's stored weights.

    FP8: every 128x128 block (output rows x reduction columns) is multiplied by
    its fp32 scale, in fp64.
    """
    gu, dn = w["gate_up"], w["down"]
    if dtype == "bf16":
        return decode_bf16(gu), decode_bf16(dn)
    if dtype == "f32":
        return np.asarray(gu, np.float32).astype(np.float64), np.asarray(dn, np.float32).astype(np.float64)
    if dtype == "e4m3":
        out = []
        for m, s in ((gu, w["scale_gate_up"]), (dn, w["scale_down"])):
            v = decode_e4m3(m)
            R, K = v.shape
            sc = np.asarray(s, np.float32).astype(np.float64)
            if R % 128 or K % 128:
                raise OracleError("FP8 blocks need both dimensions to be multiples of 128")
            # block (r // 128, c // 128) of the matrix times its scale
            v = (v.reshape(R // 128, 128, K // 128, 128) * sc[:, None, :, None]).reshape(R, K)
            out.append(v)
        return out[0], out[1]
    raise OracleError(f"dtype {dtype}")


# ----------------------------------------------------------------- routing
def topk_order(row: Sequence[float], k: int) -> List[int]:
    """Expert ids of the k largest logits, largest first; equal logits -> lower id."""
    vals = [float(v) for v in row]
    if any(math.isnan(v) for v in vals):
        raise OracleError("NaN logit")
    order = sorted(range(len(vals)), key=lambda e: (-vals[e], e))
    return order[:k]


def route(logits: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-k ids [T, k] (int32) and fp64 softmax weights over the selected logits."""
    T, E = logits.shape
    if not (1 <= k <= E):
        raise OracleError("k out of range")
    ids = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        sel = topk_order(logits[t], k)
        ids[t] = sel
        vals = [float(logits[t, e]) for e in sel]
        m = vals[0]
        ex = [math.exp(v - m) for v in vals]
        s = math.fsum(ex)
        w[t] = [v / s for v in ex]
    return ids, w


def reuse_bias(logits: np.ndarray, w_conf: np.ndarray, k: int, cap: int,
               alpha: float) -> np.ndarray:
    """Biased fp32 logits l' of S2-MoE component 2 (reading in the module docstring)."""
    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    if E < k + 1:
        raise OracleError("reuse bias needs E >= k+1")
    wc = np.asarray(w_conf, dtype=np.float32)
    if np.any(wc < 0) or np.any(np.isnan(wc)):
        raise OracleError("confidence weights must be >= 0")
    top = [topk_order(lg[b], k + 1) for b in range(T)]
    # Step 1: confidence-weighted importance, fp32, b ascending.
    g = [np.float32(0.0)] * E
    for b in range(T):
        for e in top[b][:k]:
            g[e] = np.float32(g[e] + wc[b])
    # Step 2: the preferred set E*.
    cand = [e for e in range(E) if g[e] > 0]
    cand.sort(key=lambda e: (-float(g[e]), e))
    estar = set(cand[:cap])
    # Step 3: additive bias with a per-token margin.
    out = lg.copy()
    a32 = np.float32(alpha)
    for b in range(T):
        v1 = lg[b, top[b][0]]
        vk1 = lg[b, top[b][k]]
        lam = np.float32(a32 * np.float32(v1 - vk1))
        for e in estar:
            out[b, e] = np.float32(lg[b, e] + lam)
    return out


def union_permute(ids: np.ndarray, E: int) -> Dict[str, np.ndarray]:
    """Unique experts, per-expert token groups (CSR) and the reuse ratio."""
    T, k = ids.shape
    pairs = []
    for t in range(T):
        if len(set(ids[t].tolist())) != k:
            raise OracleError("duplicate expert in a token's top-k")
        for j in range(k):
            e = int(ids[t, j])
            if not (0 <= e < E):
                raise OracleError("expert id out of range")
            pairs.append((e, t, j))
    uniq = sorted({e for e, _, _ in pairs})
    pairs.sort()
    offsets = [0]
    for e in uniq:
        offsets.append(offsets[-1] + sum(1 for p in pairs if p[0] == e))
    perm_token = np.array([t for _, t, _ in pairs], dtype=np.int32)
    perm_slot = np.array([j for _, _, j in pairs], dtype=np.int32)
    inv = np.zeros(T * k, dtype=np.int32)
    for pos, (_, t, j) in enumerate(pairs):
        inv[t * k + j] = pos
    # Reading: an empty verify set (T = 0) has reuse ratio 0 (the page defines
    # the ratio only for s >= 1 tokens).
    ratio = np.float32(np.float32(len(uniq)) / np.float32(T * k)) if T * k > 0 else np.float32(0.0)
    return {"n_unique": len(uniq), "unique": np.array(uniq, dtype=np.int32),
            "offsets": np.array(offsets, dtype=np.int32), "perm_token": perm_token,
            "perm_slot": perm_slot, "inv": inv, "reuse_ratio": ratio}


# ----------------------------------------------------------------- FFN
def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def ffn_token_slot(x: np.ndarray, Wgu: np.ndarray, Wd: np.ndarray) -> np.ndarray:
    """SwiGLU expert FFN of one token in fp64: W_d (silu(W_g x) * (W_u x))."""
    I = Wd.shape[1]
    a = Wgu[:I] @ x
    b = Wgu[I:] @ x
    return Wd @ (silu(a) * b)


def moe_layer(x: np.ndarray, ids: np.ndarray, w: np.ndarray, experts) -> np.ndarray:
    """y_t = sum_j w_tj * FFN_{ids[t,j]}(x_t), slots in order; x fp64 [T, H].

    ``experts(e)`` returns (W_gate_up fp64 [2I, H], W_down fp64 [H, I]).
    """
    T, k = ids.shape
    y = np.zeros((T, x.shape[1]), dtype=np.float64)
    cache = {}
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = experts(e)
            Wgu, Wd = cache[e]
            y[t] += w[t, j] * ffn_token_slot(x[t], Wgu, Wd)
    return y


def layer_forward(logits: np.ndarray, x: np.ndarray, k: int, E: int, experts,
                  w_conf: Optional[np.ndarray] = None, cap: int = 0, alpha: float = 0.0,
                  tokens: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Route (optionally biased), union/permute and the FFN for a subset of tokens."""
    lg = logits
    if w_conf is not None:
        lg = reuse_bias(logits, w_conf, k, cap, alpha)
    ids, w = route(lg, k)
    up = union_permute(ids, E)
    sel = list(range(ids.shape[0])) if tokens is None else list(tokens)
    y = moe_layer(x[sel], ids[sel], w[sel], experts)
    out = dict(up)
    out.update({"ids": ids, "w": w, "y": y, "tokens": np.array(sel, dtype=np.int32),
                "logits_used": lg})
    return out

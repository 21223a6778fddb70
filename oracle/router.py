"""CPU oracle: the router (gate) logits of the verify tokens.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

What it computes, with the passages it follows:

* ``router_logits``: the gate of an MoE layer scores every expert for every
  token as a linear map of the token's hidden state, logits[t, e] =
  sum_h x[t, h] * W_r[e, h] (S2-MoE write-up, background: each layer holds E
  expert FFNs and a router/gate picks each token's top-k of them; EcoSpec
  write-up section 2: S_l(x_t), the experts token t routes to at layer l, is a
  function of its hidden state x_t).  The pages print no formula for the
  gate; the plainest reading, a bias-free linear layer whose scores then go
  through the top-k/softmax of ``moe_layer.route``, is used.  Computed in fp64
  on the exactly decoded stored values.

Parity: pinned (tests/test_oracle_router.py: a hand-derived example, exact
brute force in rationals on small inputs, basis rows that select single
hidden components, linearity).
"""
from __future__ import annotations

import numpy as np

from .moe_layer import decode_bf16


def decode(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values as fp64: bf16 bit patterns or fp32 values."""
    if dtype == "bf16":
        return decode_bf16(np.asarray(a).view(np.uint16))
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype}")


def router_logits(x: np.ndarray, w_r: np.ndarray) -> np.ndarray:
    """logits [T, E] = x [T, H] . W_r [E, H]^T in fp64 (inputs already decoded)."""
    x = np.asarray(x, dtype=np.float64)
    w_r = np.asarray(w_r, dtype=np.float64)
    if x.ndim != 2 or w_r.ndim != 2 or x.shape[1] != w_r.shape[1]:
        raise ValueError("x must be [T, H] and W_r [E, H]")
    return x @ w_r.T

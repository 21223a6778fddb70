"""Seeded synthetic workloads for the MoE verify step.

This module only produces inputs: draft trees, router logits, hidden states,
the predicted (layer, expert) footprints that stand in for EcoSpec's expert
predictor, and the counter-hash keys of the expert weights.  It contains none
of the verify step's arithmetic (no routing weights, no unions, no selection,
no FFN); both the CUDA path and the CPU oracle consume what it returns.

Workload recipe (the pages' workloads, synthetic):

* Draft tree: EAGLE-3 shape, 3 forward steps keeping the top 2 children per
  node, so 2 + 4 + 8 = 14 draft nodes below the root (EcoSpec write-up, section
  2, the list of the three steps of a speculative round).  Nodes are numbered
  breadth-first, so a parent always has a smaller index than its children.
  Each internal node's two child probabilities are one Dirichlet(a, a) draw,
  sorted in decreasing order; the path probability is
  P(child) = fl32(P(parent) * fl32(q)), with P(root) = 1 (section 3.3, the
  definition of P(t_i) as the product along the path).
* Router logits per layer: ``-c * rank(e) + z``; ``rank`` is a seeded
  permutation of the experts per layer (expert popularity decaying roughly
  exponentially by rank, width-vs-depth note section 1) and ``z`` is an AR(1)
  process along tree edges, ``z_child = rho * z_parent + sqrt(1 - rho^2) * eps``
  with unit-normal ``eps`` (consecutive tokens co-activate experts, same
  section).  Rounded once to fp32.
* Predicted footprints: the predictor stand-in is an oracle predictor (the
  EcoSpec ablation with oracle expert sets, section 4.3): each node's own
  footprint in layer l is the k experts with the largest of its own layer-l
  logits.  Bit ``l * E + e`` of a node's bitset marks (layer l, expert e).
* Hidden states: unit normal per element, rounded to the storage type (bf16
  round-to-nearest-even, or fp32).
* Expert weights: counter-hash ``grid8`` values (bf16 / fp32) or ``e4m3``
  codes with fp32 per-128x128-block scales, see ``counter_hash``.
* Ragged depth (batched stress workload): sequence i gets
  gamma_i = min(6, #draft nodes with P >= tau), a confidence-gated budget in
  the spirit of the width-vs-depth note, section 2.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np

from . import counter_hash as ch

# Tree shape: 3 steps x top-2 (EAGLE-3).
TREE_DEPTH = 3
TREE_BRANCH = 2
EPS_DEFAULT = 2.0 ** -10


@dataclass(frozen=True)
class MoEConfig:
    name: str
    L: int
    H: int
    E: int
    k: int
    I: int
    dtype: str            # "f32" | "bf16" | "e4m3"
    nseq: int = 1
    gamma: int = 4
    ragged: bool = False
    gamma_max: int = 6
    tau: float = 0.1
    rho: float = 0.6
    c: float = 0.02
    dirichlet: float = 0.5
    use_bias: bool = False
    cap: int = 0
    alpha: float = 0.25
    mode: int = 0         # 0 marginal, 1 static
    eps: float = EPS_DEFAULT
    seed: int = 0
    tree_depth: int = TREE_DEPTH
    tree_branch: int = TREE_BRANCH
    chain_beta: float = 0.0   # > 0: per-sequence acceptance rate a ~ Beta(b, b), every child q = a

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)

    @property
    def W(self) -> int:
        """uint32 words per (layer, expert) footprint bitset."""
        return (self.L * self.E + 31) // 32

    @property
    def n_nodes(self) -> int:
        return sum(self.tree_branch ** d for d in range(1, self.tree_depth + 1))


# The five workloads.  The bias slope ``c`` of the Qwen-like shapes is set so
# that the mean union per layer under marginal-cost selection is near the
# 23.7 experts per layer the EcoSpec write-up quotes for Qwen3-235B (section 1,
# table of section 4.1); the GPT-OSS-like slope puts 60% of the mean router
# mass on the top 10% of experts; the DeepSeek-like slope is 0.05 per rank.
CONFIGS = {
    "toy": MoEConfig("toy", L=1, H=256, E=16, k=2, I=512, dtype="f32",
                     rho=0.7, c=0.3, dirichlet=1.0, seed=0),
    "qwen3_235b_like": MoEConfig("qwen3_235b_like", L=16, H=4096, E=128, k=8, I=1536,
                                 dtype="bf16", rho=0.6, c=0.02, dirichlet=0.5, seed=1),
    "gpt_oss_120b_like": MoEConfig("gpt_oss_120b_like", L=24, H=2880, E=128, k=4, I=2880,
                                   dtype="bf16", rho=0.7, c=0.0705, dirichlet=0.5,
                                   use_bias=True, cap=8, alpha=0.25, seed=2),
    "deepseek_v3_like": MoEConfig("deepseek_v3_like", L=8, H=7168, E=256, k=8, I=2048,
                                  dtype="e4m3", rho=0.5, c=0.05, dirichlet=0.5, seed=3),
    "batched_qwen_like": MoEConfig("batched_qwen_like", L=16, H=4096, E=128, k=8, I=1536,
                                   dtype="bf16", nseq=4, ragged=True, rho=0.6, c=0.02,
                                   dirichlet=0.5, tau=0.1, seed=4),
}

# Bytes per weight element by storage type.
ELEM_BYTES = {"f32": 4, "bf16": 2, "e4m3": 1}


def tree_parents(depth: int = TREE_DEPTH, branch: int = TREE_BRANCH) -> np.ndarray:
    """Parent index of every draft node, breadth-first; -1 means the root."""
    parents = []
    level_prev = [-1]
    nxt = 0
    for _ in range(depth):
        level = []
        for p in level_prev:
            for _ in range(branch):
                parents.append(p)
                level.append(nxt)
                nxt += 1
        level_prev = level
    return np.asarray(parents, dtype=np.int32)


def bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    r = ((u + rounding) >> np.uint64(16)).astype(np.uint16)
    return r


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    """One verify step's inputs (host arrays) plus the weight keys."""
    cfg: MoEConfig
    parent: np.ndarray          # [N] int32, -1 = root
    P: np.ndarray               # [nseq, N] float32 path probabilities
    own_fp: np.ndarray          # [nseq, N, W] uint32 own-footprint bitsets
    gamma: np.ndarray           # [nseq] int32
    logits: np.ndarray          # [L, nseq, N+1, E] float32; row 0 is the root
    x: np.ndarray               # [L, nseq, N+1, H] uint16 bf16 bits or float32
    weight_seed: int
    root_fp: np.ndarray = None  # [nseq, W] uint32 footprint of each root token (its own top-k per layer)
    T: int = field(init=False)

    def __post_init__(self):
        self.T = int(np.sum(self.gamma + 1))


def weight_stream_keys(cfg: MoEConfig, layer: int) -> dict:
    """Counter-hash keys of one layer's weight tensors."""
    seed = ch.mix64_int(0x5EED0000 + cfg.seed)
    base = layer * 16
    return {
        "gate_up": ch.stream_key(seed, base + 0),
        "down": ch.stream_key(seed, base + 1),
        "scale_gate_up": ch.stream_key(seed, base + 2),
        "scale_down": ch.stream_key(seed, base + 3),
    }


def router_stream_key(cfg: MoEConfig, layer: int) -> int:
    """Counter-hash key of one layer's router matrix W_r [E, H]."""
    return ch.stream_key(ch.mix64_int(0x5EED0000 + cfg.seed), layer * 16 + 4)


def router_dtype(cfg: MoEConfig) -> str:
    """Storage type of the router matrix: fp32 for fp32 models, else bf16
    (FP8 models keep their router in bf16)."""
    return "f32" if cfg.dtype == "f32" else "bf16"


def router_weights_host(cfg: MoEConfig, layer: int) -> np.ndarray:
    """Host copy of W_r [E, H] (storage bits for bf16, values for fp32); the
    same grid values as the expert weights, odd multiples of 2^-13."""
    kind = ch.KIND_GRID8_F32 if router_dtype(cfg) == "f32" else ch.KIND_GRID8_BF16
    n = cfg.E * cfg.H
    return ch.fill_host(kind, router_stream_key(cfg, layer), 0, n).reshape(cfg.E, cfg.H)


def weight_shapes(cfg: MoEConfig) -> dict:
    """Per-layer tensor shapes (expert-major, each expert contiguous).

    ``gate_up`` is [E, 2I, H]: rows 0..I-1 hold W_gate, rows I..2I-1 W_up.
    ``down`` is [E, H, I].  FP8 scales are per 128x128 block (output row block
    x reduction block) of each expert matrix.
    """
    s = {"gate_up": (cfg.E, 2 * cfg.I, cfg.H), "down": (cfg.E, cfg.H, cfg.I)}
    if cfg.dtype == "e4m3":
        s["scale_gate_up"] = (cfg.E, -(-2 * cfg.I // 128), -(-cfg.H // 128))
        s["scale_down"] = (cfg.E, -(-cfg.H // 128), -(-cfg.I // 128))
    return s


def weight_kind(cfg: MoEConfig) -> int:
    return {"bf16": ch.KIND_GRID8_BF16, "f32": ch.KIND_GRID8_F32, "e4m3": ch.KIND_E4M3}[cfg.dtype]


def expert_weights_host(cfg: MoEConfig, layer: int, expert: int) -> dict:
    """Host copy of one expert's weights (storage bits), regenerated from the keys."""
    keys = weight_stream_keys(cfg, layer)
    shp = weight_shapes(cfg)
    out = {}
    kind = weight_kind(cfg)
    for name in ("gate_up", "down"):
        _, r, c = shp[name]
        n = r * c
        out[name] = ch.fill_host(kind, keys[name], expert * n, n).reshape(r, c)
    if cfg.dtype == "e4m3":
        for name in ("scale_gate_up", "scale_down"):
            _, r, c = shp[name]
            n = r * c
            out[name] = ch.fill_host(ch.KIND_SCALE_F32, keys[name], expert * n, n).reshape(r, c)
    return out


def make_workload(cfg: MoEConfig) -> Workload:
    rng = np.random.default_rng([cfg.seed, 0xC0FFEE])
    parent = tree_parents(cfg.tree_depth, cfg.tree_branch)
    N = parent.shape[0]
    L, E, H, k = cfg.L, cfg.E, cfg.H, cfg.k

    # Path probabilities.
    P = np.zeros((cfg.nseq, N), dtype=np.float32)
    for s in range(cfg.nseq):
        child_q = {}
        if cfg.chain_beta > 0:
            # Acceptance is bimodal across sequences (width-vs-depth note,
            # section 2: drafts of a sequence tend to be all right or all
            # wrong): one rate a_s ~ Beta(b, b) per sequence, q = a_s at
            # every draft position, so P along a chain is a_s ** depth.
            a_s = np.float32(rng.beta(cfg.chain_beta, cfg.chain_beta))
            for t in range(N):
                child_q[t] = a_s
        for p in ([] if cfg.chain_beta > 0 else [-1] + list(range(N))):
            kids = [t for t in range(N) if parent[t] == p]
            if not kids:
                continue
            q = np.sort(rng.dirichlet([cfg.dirichlet] * len(kids)))[::-1].astype(np.float32)
            for t, qq in zip(kids, q):
                child_q[t] = qq
        for t in range(N):
            pp = np.float32(1.0) if parent[t] < 0 else P[s, parent[t]]
            P[s, t] = np.float32(pp * child_q[t])

    # Verify budgets.
    if cfg.ragged:
        gamma = np.array([min(cfg.gamma_max, int(np.sum(P[s] >= np.float32(cfg.tau))))
                          for s in range(cfg.nseq)], dtype=np.int32)
    else:
        gamma = np.full(cfg.nseq, min(cfg.gamma, N), dtype=np.int32)

    # Router logits: -c*rank + AR(1) along tree edges; row 0 = root.
    logits = np.zeros((L, cfg.nseq, N + 1, E), dtype=np.float32)
    a = math.sqrt(1.0 - cfg.rho ** 2)
    for l in range(L):
        rank = rng.permutation(E).astype(np.float64)
        bias = -cfg.c * rank
        for s in range(cfg.nseq):
            z = np.zeros((N + 1, E))
            z[0] = rng.standard_normal(E)
            for t in range(N):
                zp = z[0] if parent[t] < 0 else z[parent[t] + 1]
                z[t + 1] = cfg.rho * zp + a * rng.standard_normal(E)
            logits[l, s] = (bias[None, :] + z).astype(np.float32)

    # Own footprints from the node's own logits (oracle predictor stand-in).
    W = cfg.W
    own_fp = np.zeros((cfg.nseq, N, W), dtype=np.uint32)
    for s in range(cfg.nseq):
        for t in range(N):
            for l in range(L):
                top = np.argsort(-logits[l, s, t + 1], kind="stable")[:k]
                for e in top:
                    bit = l * E + int(e)
                    own_fp[s, t, bit // 32] |= np.uint32(1 << (bit % 32))

    # The root tokens' own footprints (their top-k per layer), same rule.
    root_fp = np.zeros((cfg.nseq, W), dtype=np.uint32)
    for s in range(cfg.nseq):
        for l in range(L):
            for e in np.argsort(-logits[l, s, 0], kind="stable")[:k]:
                bit = l * E + int(e)
                root_fp[s, bit // 32] |= np.uint32(1 << (bit % 32))

    # Hidden states.
    xs = rng.standard_normal((L, cfg.nseq, N + 1, H)).astype(np.float32)
    x = xs if cfg.dtype == "f32" else bf16_bits_rne(xs)

    return Workload(cfg=cfg, parent=parent, P=P, own_fp=own_fp, gamma=gamma,
                    logits=logits, x=x, weight_seed=cfg.seed, root_fp=root_fp)


def chain_config(base: MoEConfig, nseq: int, depth: int = 6, beta: float = 0.5, seed: int = 100,
                 gamma: int = 0) -> MoEConfig:
    """A batch of draft chains (one speculated token per position, the
    depth strategy of the width-vs-depth note, section 1) on the layer shapes
    of ``base``: ``depth`` draft positions per sequence, consecutive positions
    correlated through the AR(1) logits (rho of ``base``), acceptance rate
    a_s ~ Beta(beta, beta) per sequence (bimodal for beta < 1)."""
    return base.replace(name=f"{base.name}_chains", nseq=nseq, tree_depth=depth, tree_branch=1,
                        chain_beta=beta, gamma=gamma, ragged=False, mode=0, seed=seed)


def perturbed_footprints(wl: Workload, accuracy: float, seed: int = 0) -> np.ndarray:
    """Predicted footprints of an imperfect expert predictor: each of a node's
    k predicted experts per layer is kept with probability ``accuracy``, else
    replaced by a uniformly drawn expert outside the node's true top-k (so the
    top-K accuracy, the share of predicted experts that are real, is
    ``accuracy`` in expectation).  Input construction for the mismatch study;
    the true routing (the logits) is unchanged."""
    cfg = wl.cfg
    L, E, k = cfg.L, cfg.E, cfg.k
    nseq, N = wl.P.shape
    rng = np.random.default_rng([cfg.seed, 0xF00D, seed, int(round(accuracy * 1e6))])
    out = np.zeros_like(wl.own_fp)
    for s in range(nseq):
        for t in range(N):
            for l in range(L):
                top = np.argsort(-wl.logits[l, s, t + 1], kind="stable")[:k]
                others = np.setdiff1d(np.arange(E), top)
                keep = rng.random(k) < accuracy
                repl = rng.choice(others, size=int((~keep).sum()), replace=False)
                pred = np.concatenate([top[keep], repl])
                for e in pred:
                    bit = l * E + int(e)
                    out[s, t, bit // 32] |= np.uint32(1 << (bit % 32))
    return out


def small_case(name: str = "small_bf16", **kw) -> MoEConfig:
    """Shapes the oracle finishes in seconds that still span several 128-row
    tiles and a ragged tail; used by the parity tests."""
    base = dict(L=2, H=576, E=16, k=4, I=320, dtype="bf16", rho=0.6, c=0.05,
                dirichlet=0.5, seed=11)
    base.update(kw)
    return MoEConfig(name, **base)

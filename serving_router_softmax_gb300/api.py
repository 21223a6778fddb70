"""Thin PyTorch binding of libmoeverify: argument checks and pointer marshalling.

Every computation happens in the library's CUDA kernels; torch only provides
device memory and the current stream.  Calls raise ``MoEError`` on a non-OK
host status.  Device-side error bits land in the ``dev_err`` tensor (int32,
one element), which callers may pass in and inspect after synchronising.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import torch

from . import _lib as L


class MoEError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != L.MOE_OK:
        msg = L.load().moe_status_str(status).decode()
        raise MoEError(f"{what}: {msg} (status {status})")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise MoEError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise MoEError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t: torch.Tensor, dtype: torch.dtype, shape: Sequence[int], name: str):
    if t.dtype != dtype:
        raise MoEError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise MoEError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def new_dev_err(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


DTYPES = {"f32": L.DTYPE_F32, "bf16": L.DTYPE_BF16, "e4m3": L.DTYPE_E4M3_B128}


LAYOUTS = {"rowmajor": L.LAYOUT_ROWMAJOR, "tiled": L.LAYOUT_TILED}


@dataclass
class ExpertLayer:
    """One layer's expert weights on the device.

    Row-major layout: gate_up [E, 2I, H] (rows 0..I-1 gate, I..2I-1 up) and
    down [E, H, I]; storage float32, bf16 bits (int16/uint16/bfloat16) or
    uint8 FP8 codes, with FP8 scales [E, 2I/128, H/128] / [E, H/128, I/128].
    Tiled layout (bf16, from ``pack_tiled``): flat buffers; ``dims`` gives
    (H, I, E).
    """
    gate_up: torch.Tensor
    down: torch.Tensor
    dtype: str
    scales_gate_up: Optional[torch.Tensor] = None
    scales_down: Optional[torch.Tensor] = None
    layout: str = "rowmajor"
    dims: Optional[tuple] = None
    pool: Optional[L.ExpertPool] = None  # expert residency (see ExpertPool); None: all E experts resident

    @property
    def E(self):
        return self.dims[2] if self.dims else self.gate_up.shape[0]

    @property
    def I(self):
        return self.dims[1] if self.dims else self.gate_up.shape[1] // 2

    @property
    def H(self):
        return self.dims[0] if self.dims else self.gate_up.shape[2]

    def struct(self) -> L.LayerWeights:
        return L.LayerWeights(self.H, self.I, self.E, DTYPES[self.dtype], LAYOUTS[self.layout],
                              _ptr(self.gate_up), _ptr(self.down), _ptr(self.scales_gate_up),
                              _ptr(self.scales_down), C.pointer(self.pool) if self.pool is not None else None)


def expert_bytes(layer: ExpertLayer):
    """(gate/up, down) bytes of one expert of the layer in its layout (one pool slot)."""
    gu, dn = C.c_size_t(0), C.c_size_t(0)
    st = layer.struct()
    if L.load().moe_expert_bytes(C.byref(st), C.byref(gu), C.byref(dn)) == 0:
        raise MoEError("invalid layer")
    return gu.value, dn.value


def hot_list(ids: torch.Tensor, E: int, n_hot: int, first_slot: int = 0, dev_err=None, stream=None):
    """Hot-expert list from profiled routing decisions (moe_hot_list): returns device int32
    tensors (hot [n_hot] in ascending id order, counts [E], home_slot [E])."""
    if not 0 <= n_hot <= E:
        raise MoEError("n_hot outside [0, E]")
    ids = ids.contiguous()
    if ids.dtype != torch.int32:
        raise MoEError("ids must be int32")
    dev = ids.device
    hot = torch.empty(max(n_hot, 1), dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    home = torch.empty(E, dtype=torch.int32, device=dev)
    _check(L.load().moe_hot_list(_ptr(ids), ids.numel(), E, n_hot, first_slot, _ptr(counts), _ptr(hot),
                                 _ptr(home), _ptr(dev_err), _stream(stream)), "moe_hot_list")
    return hot[:n_hot], counts, home


def depth_policy(conf: torch.Tensor, fp: torch.Tensor, C0: float, T_exp: float,
                 max_depth: Optional[torch.Tensor] = None, dev_err=None, stream=None):
    """Confidence-gated depth vector (moe_depth_policy).  conf [nseq, D] fp32 cumulative
    confidences, fp [nseq, D+1, W] int32/uint32 footprints (row 0 = root).  Returns device
    tensors (depth [nseq] int32, common [1] int32, throughput [2] fp64: common, final)."""
    if conf.dim() != 2 or fp.dim() != 3:
        raise MoEError("conf [nseq, D] and fp [nseq, D+1, W] expected")
    nseq, D = conf.shape
    _need(conf, torch.float32, (nseq, D), "conf")
    if fp.shape[0] != nseq or fp.shape[1] != D + 1 or fp.dtype != torch.int32:
        raise MoEError("fp must be int32 [nseq, D+1, W]")
    if max_depth is not None:
        _need(max_depth, torch.int32, (nseq,), "max_depth")
    dev = conf.device
    depth = torch.empty(nseq, dtype=torch.int32, device=dev)
    common = torch.empty(1, dtype=torch.int32, device=dev)
    thr = torch.empty(2, dtype=torch.float64, device=dev)
    cfg = L.DepthCfg(nseq, D, fp.shape[2], C0, T_exp)
    _check(L.load().moe_depth_policy(_ptr(conf), _ptr(fp), _ptr(max_depth), C.byref(cfg), _ptr(depth),
                                     _ptr(common), _ptr(thr), _ptr(dev_err), _stream(stream)),
           "moe_depth_policy")
    return depth, common, thr


class HostExperts:
    """All E experts of every layer of a stack in page-locked host (Grace) memory, in the layers'
    layout (one row of ``gate_up[l]`` / ``down[l]`` per expert).  FP8 block scales stay on the
    device (they are indexed by expert id and always resident)."""

    def __init__(self, full_layers: List[ExpertLayer]):
        if not full_layers:
            raise MoEError("no layers")
        ref = full_layers[0]
        self.H, self.I, self.E, self.dtype, self.layout = ref.H, ref.I, ref.E, ref.dtype, ref.layout
        self.gate_up_bytes, self.down_bytes = expert_bytes(ref)
        self.scales = []
        self.gate_up, self.down = [], []
        for lay in full_layers:
            if (lay.H, lay.I, lay.E, lay.dtype, lay.layout) != (self.H, self.I, self.E, self.dtype, self.layout):
                raise MoEError("all layers share one shape")
            if lay.pool is not None:
                raise MoEError("expected fully resident layers")
            for src, dst, nb in ((lay.gate_up, self.gate_up, self.gate_up_bytes),
                                 (lay.down, self.down, self.down_bytes)):
                h = torch.empty((self.E, nb), dtype=torch.uint8, pin_memory=True)
                h.copy_(src.contiguous().view(torch.uint8).reshape(self.E, nb))
                dst.append(h)
            self.scales.append((lay.scales_gate_up, lay.scales_down))

    @property
    def L(self) -> int:
        return len(self.gate_up)


class ExpertPool:
    """Expert-level residency for a stack of layers on one Grace-Blackwell GPU.

    Every layer keeps all E experts in page-locked host (Grace) memory
    (``HostExperts``).  One pair of device buffers holds, for layer l, its
    hot experts in slots l * n_hot + j (hot[l][j], ascending ids), followed
    by n_stage staging slots that all layers share; a layer's cold experts of
    the union are copied there over NVLink-C2C by moe_stage_experts
    (moe_verify_step does it for every pooled layer).  ``layers`` gives the
    ExpertLayer views to pass to verify_ffn / VerifyStep.
    """

    def __init__(self, host, hot: Sequence[Sequence[int]], n_stage: int, device=None):
        if not isinstance(host, HostExperts):
            host = HostExperts(list(host))
        if len(hot) != host.L:
            raise MoEError("one hot list per layer required")
        n_hot = len(hot[0])
        if any(len(h) != n_hot for h in hot):
            raise MoEError("every layer needs the same number of hot experts")
        if n_stage < 0:
            raise MoEError("n_stage < 0")
        dev = torch.device(device) if device is not None else (
            host.scales[0][0].device if host.scales[0][0] is not None else torch.device("cuda"))
        self.host = host
        self.n_hot, self.n_stage, self.L = n_hot, n_stage, host.L
        self.n_slots = self.L * n_hot + n_stage
        self.stage_first = self.L * n_hot
        gu_b, dn_b = host.gate_up_bytes, host.down_bytes
        self.gate_up_bytes, self.down_bytes = gu_b, dn_b
        self.pool_gate_up = torch.empty((max(self.n_slots, 1), gu_b), dtype=torch.uint8, device=dev)
        self.pool_down = torch.empty((max(self.n_slots, 1), dn_b), dtype=torch.uint8, device=dev)
        self.host_gate_up, self.host_down = host.gate_up, host.down
        self.home_slot, self.slot_of = [], []
        self.layers: List[ExpertLayer] = []
        for l, hl in enumerate(hot):
            hl = sorted(int(e) for e in hl)
            if len(set(hl)) != len(hl) or any(e < 0 or e >= host.E for e in hl):
                raise MoEError("hot list: distinct ids in [0, E)")
            home = torch.full((host.E,), -1, dtype=torch.int32)
            for j, e in enumerate(hl):
                s_ = l * n_hot + j
                home[e] = s_
                self.pool_gate_up[s_].copy_(host.gate_up[l][e])
                self.pool_down[s_].copy_(host.down[l][e])
            home = home.to(dev)
            slot_of = torch.full((host.E,), -1, dtype=torch.int32, device=dev)
            st = L.ExpertPool(self.n_slots, self.stage_first, n_stage, home.data_ptr(),
                              host.gate_up[l].data_ptr(), host.down[l].data_ptr(), slot_of.data_ptr())
            self.home_slot.append(home)
            self.slot_of.append(slot_of)
            sgu, sdn = host.scales[l]
            self.layers.append(ExpertLayer(self.pool_gate_up, self.pool_down, host.dtype, sgu, sdn,
                                           layout=host.layout, dims=(host.H, host.I, host.E), pool=st))

    def resident_bytes(self) -> int:
        return self.n_slots * (self.gate_up_bytes + self.down_bytes)


def stage_experts(layer: ExpertLayer, union: Dict[str, torch.Tensor], n_staged: Optional[torch.Tensor] = None,
                  dev_err: Optional[torch.Tensor] = None, stream=None):
    """Copies the union's cold experts of a pooled layer into its staging slots (moe_stage_experts)."""
    if layer.pool is None:
        raise MoEError("layer has no expert pool")
    st = layer.struct()
    _check(L.load().moe_stage_experts(C.byref(st), _ptr(union["n_unique"]), _ptr(union["unique"]),
                                      _ptr(n_staged), _ptr(dev_err), _stream(stream)), "moe_stage_experts")


def pack_tiled(layer: ExpertLayer, stream=None) -> ExpertLayer:
    """Load-time repack of a row-major bf16 layer into the tiled layout."""
    lib = L.load()
    if layer.layout != "rowmajor" or layer.dtype not in ("bf16", "e4m3"):
        raise MoEError("pack_tiled needs a row-major bf16 or FP8 layer")
    st = layer.struct()
    gu_b, dn_b = C.c_size_t(0), C.c_size_t(0)
    if lib.moe_tiled_bytes(C.byref(st), C.byref(gu_b), C.byref(dn_b)) == 0:
        raise MoEError("layer shape cannot be tiled")
    dev = layer.gate_up.device
    if layer.dtype == "bf16":
        gu = torch.empty(gu_b.value // 2, dtype=torch.int16, device=dev)
        dn = torch.empty(dn_b.value // 2, dtype=torch.int16, device=dev)
    else:
        gu = torch.empty(gu_b.value, dtype=torch.uint8, device=dev)
        dn = torch.empty(dn_b.value, dtype=torch.uint8, device=dev)
    _check(lib.moe_pack_tiled(C.byref(st), _ptr(gu), _ptr(dn), _stream(stream)), "moe_pack_tiled")
    return ExpertLayer(gu, dn, layer.dtype, layer.scales_gate_up, layer.scales_down, layout="tiled",
                       dims=(layer.H, layer.I, layer.E))


# ------------------------------------------------------------------ calls
def _act_dtype(t: torch.Tensor, name: str) -> int:
    if t.dtype == torch.float32:
        return L.DTYPE_F32
    if t.dtype in (torch.int16, torch.bfloat16):
        return L.DTYPE_BF16
    raise MoEError(f"{name}: expected float32, bfloat16 or int16 (bf16 bits), got {t.dtype}")


def router_logits(x: torch.Tensor, w_router: torch.Tensor, out: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """Gate logits [T, E] fp32 = x [T, H] . w_router [E, H]^T (fp32 accumulation).

    ``x`` and ``w_router`` are float32, bfloat16 or int16 holding bf16 bits."""
    lib = L.load()
    T, H = x.shape
    E = w_router.shape[0]
    if w_router.shape != (E, H):
        raise MoEError(f"w_router: expected shape ({E}, {H}), got {tuple(w_router.shape)}")
    for t, n in ((x, "x"), (w_router, "w_router")):
        if not t.is_contiguous():
            raise MoEError(f"{n} must be contiguous")
    if out is None:
        out = torch.empty((T, E), dtype=torch.float32, device=x.device)
    _need(out, torch.float32, (T, E), "out")
    cfg = L.RouterCfg(T, H, E, _act_dtype(x, "x"), _act_dtype(w_router, "w_router"))
    _check(lib.moe_router_logits(_ptr(x), _ptr(w_router), C.byref(cfg), _ptr(out), _stream(stream)),
           "moe_router_logits")
    return out


def route(logits: torch.Tensor, k: int, w_conf: Optional[torch.Tensor] = None, cap: int = 0,
          alpha: float = 0.0, dev_err: Optional[torch.Tensor] = None, stream=None):
    """Top-k ids [T, k] int32 and weights [T, k] fp32 (optionally reuse-biased)."""
    lib = L.load()
    T, E = logits.shape
    _need(logits, torch.float32, (T, E), "logits")
    use_bias = w_conf is not None
    if use_bias:
        _need(w_conf, torch.float32, (T,), "w_conf")
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    cfg = L.RouteCfg(T, E, k, int(use_bias), cap, alpha)
    _check(lib.moe_route(_ptr(logits), _ptr(w_conf), C.byref(cfg), _ptr(ids), _ptr(w),
                         _ptr(dev_err), _stream(stream)), "moe_route")
    return ids, w


def union_permute(ids: torch.Tensor, E: int, dev_err: Optional[torch.Tensor] = None,
                  stream=None) -> Dict[str, torch.Tensor]:
    lib = L.load()
    T, k = ids.shape
    _need(ids, torch.int32, (T, k), "ids")
    dev = ids.device
    cap = min(E, T * k)
    out = {
        "n_unique": torch.empty(1, dtype=torch.int32, device=dev),
        "unique": torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
        "offsets": torch.empty(cap + 1, dtype=torch.int32, device=dev),
        "perm_token": torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
        "perm_slot": torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
        "inv": torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
        "reuse_ratio": torch.empty(1, dtype=torch.float32, device=dev),
    }
    _check(lib.moe_union_permute(_ptr(ids), T, k, E, _ptr(out["n_unique"]), _ptr(out["unique"]),
                                 _ptr(out["offsets"]), _ptr(out["perm_token"]),
                                 _ptr(out["perm_slot"]), _ptr(out["inv"]),
                                 _ptr(out["reuse_ratio"]), _ptr(dev_err), _stream(stream)),
           "moe_union_permute")
    return out


def ffn_workspace_bytes(layer: ExpertLayer, T: int, k: int) -> int:
    st = layer.struct()
    return int(L.load().moe_verify_ffn_workspace(C.byref(st), T, k))


def verify_ffn(x: torch.Tensor, k: int, layer: ExpertLayer, union: Dict[str, torch.Tensor],
               w: torch.Tensor, y: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """y [T, H] fp32 = sum_j w[t, j] * FFN_{ids[t, j]}(x[t])."""
    lib = L.load()
    T, H = x.shape
    if H != layer.H:
        raise MoEError("x hidden size does not match the layer")
    _need(w, torch.float32, (T, k), "w")
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _need(y, torch.float32, (T, H), "y")
    need = ffn_workspace_bytes(layer, T, k)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    st = layer.struct()
    _check(lib.moe_verify_ffn(_ptr(x), T, k, C.byref(st), _ptr(union["n_unique"]),
                              _ptr(union["unique"]), _ptr(union["offsets"]),
                              _ptr(union["perm_token"]), _ptr(union["inv"]), _ptr(w), _ptr(y),
                              _ptr(workspace), workspace.numel(), _ptr(dev_err), _stream(stream)),
           "moe_verify_ffn")
    return y


def eco_select(P: torch.Tensor, parent: torch.Tensor, own_fp: torch.Tensor, gamma_max: int,
               gamma_per_seq: Optional[torch.Tensor] = None, eps: float = 2.0 ** -10,
               mode: int = 0, dev_err: Optional[torch.Tensor] = None, stream=None):
    """Selected node ids [nseq, gamma_max] (selection order, -1 padded) and |B| [nseq]."""
    lib = L.load()
    nseq, N = P.shape
    W = own_fp.shape[-1]
    _need(P, torch.float32, (nseq, N), "P")
    _need(parent, torch.int32, (nseq, N), "parent")
    if own_fp.dtype not in (torch.int32, torch.uint32):
        raise MoEError("own_fp must be int32/uint32 words")
    if tuple(own_fp.shape) != (nseq, N, W):
        raise MoEError("own_fp shape")
    if gamma_per_seq is not None:
        _need(gamma_per_seq, torch.int32, (nseq,), "gamma_per_seq")
    sel = torch.empty((nseq, max(gamma_max, 1)), dtype=torch.int32, device=P.device)
    usz = torch.empty(nseq, dtype=torch.int32, device=P.device)
    cfg = L.EcoCfg(N, W, gamma_max, mode, eps)
    _check(lib.eco_select(_ptr(P), _ptr(parent), _ptr(own_fp), nseq, _ptr(gamma_per_seq),
                          C.byref(cfg), _ptr(sel), _ptr(usz), _ptr(dev_err), _stream(stream)),
           "eco_select")
    return sel[:, :gamma_max], usz


@dataclass
class StepSpec:
    L: int
    nseq: int
    N: int
    W: int
    E: int
    k: int
    H: int
    I: int
    dtype: str
    T: int
    gamma_max: int
    layout: str = "rowmajor"
    mode: int = 0
    eps: float = 2.0 ** -10
    use_bias: bool = False
    cap: int = 0
    alpha: float = 0.0

    def struct(self) -> L.StepCfg:
        return L.StepCfg(self.L, self.nseq, self.N, self.W, self.E, self.k, self.H, self.I,
                         DTYPES[self.dtype], LAYOUTS[self.layout], self.T, self.gamma_max, self.mode, self.eps,
                         int(self.use_bias), self.cap, self.alpha)


def step_workspace_bytes(spec: StepSpec) -> int:
    st = spec.struct()
    return int(L.load().moe_verify_step_workspace(C.byref(st)))


class VerifyStep:
    """Pre-bound whole verify step: owns the output tensors and the workspace,
    so each call enqueues the L-layer step with no allocation."""

    def __init__(self, spec: StepSpec, layers: List[ExpertLayer], device="cuda"):
        if len(layers) != spec.L:
            raise MoEError("one ExpertLayer per layer required")
        self.spec = spec
        self.layers = layers
        self.device = torch.device(device)
        self._cfg = spec.struct()
        arr = (L.LayerWeights * spec.L)()
        for i, ly in enumerate(layers):
            arr[i] = ly.struct()
        self._layers = arr
        nbytes = step_workspace_bytes(spec)
        if nbytes == 0:
            raise MoEError("unsupported step configuration")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.selected = torch.empty((spec.nseq, max(spec.gamma_max, 1)), dtype=torch.int32,
                                    device=self.device)
        self.union_size = torch.empty(spec.nseq, dtype=torch.int32, device=self.device)
        self.n_unique = torch.empty(spec.L, dtype=torch.int32, device=self.device)
        self.y = torch.empty((spec.L, spec.T, spec.H), dtype=torch.float32, device=self.device)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=self.device)

    def __call__(self, P, parent, own_fp, gamma_per_seq, node_logits, node_x, stream=None):
        lib = L.load()
        _check(lib.moe_verify_step(C.byref(self._cfg), _ptr(P), _ptr(parent), _ptr(own_fp),
                                   _ptr(gamma_per_seq), _ptr(node_logits), _ptr(node_x),
                                   self._layers, _ptr(self.selected), _ptr(self.union_size),
                                   _ptr(self.n_unique), _ptr(self.y), _ptr(self.workspace),
                                   self.workspace.numel(), _ptr(self.dev_err), _stream(stream)),
               "moe_verify_step")
        return self.y

    def capture(self, P, parent, own_fp, gamma_per_seq, node_logits, node_x, steps: int = 1):
        """Records `steps` verify steps on these input tensors into a CUDA graph and returns it;
        `graph.replay()` then runs them with no host launch work.  The inputs are read at replay
        time, so new values are copied into the same tensors between replays.  The step makes no
        allocation and no host synchronisation, which is what makes it capturable."""
        args = (P, parent, own_fp, gamma_per_seq, node_logits, node_x)
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self(*args)  # warm-up outside the capture (one-time attribute setup)
        torch.cuda.current_stream(self.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(steps):
                self(*args)
        return graph


class VerifyPlan:
    """The control path of a verify step (selection, then every layer's
    routing and expert union) with its output tensors bound once."""

    def __init__(self, spec: StepSpec, device="cuda"):
        self.spec = spec
        self.device = torch.device(device)
        self._cfg = spec.struct()
        d, i32, f32 = self.device, torch.int32, torch.float32
        T, k, Lc = spec.T, spec.k, spec.L
        cap = min(spec.E, T * k)
        self.selected = torch.empty((spec.nseq, max(spec.gamma_max, 1)), dtype=i32, device=d)
        self.union_size = torch.empty(spec.nseq, dtype=i32, device=d)
        self.verify_rows = torch.empty(T, dtype=i32, device=d)
        self.verify_conf = torch.empty(T, dtype=f32, device=d)
        self.ids = torch.empty((Lc, T, k), dtype=i32, device=d)
        self.w = torch.empty((Lc, T, k), dtype=f32, device=d)
        self.n_unique = torch.empty(Lc, dtype=i32, device=d)
        self.unique = torch.empty((Lc, cap), dtype=i32, device=d)
        self.offsets = torch.empty((Lc, cap + 1), dtype=i32, device=d)
        self.perm_token = torch.empty((Lc, T * k), dtype=i32, device=d)
        self.perm_slot = torch.empty((Lc, T * k), dtype=i32, device=d)
        self.inv = torch.empty((Lc, T * k), dtype=i32, device=d)
        self.reuse_ratio = torch.empty(Lc, dtype=f32, device=d)
        self.dev_err = torch.zeros(1, dtype=i32, device=d)

    def __call__(self, P, parent, own_fp, gamma_per_seq, node_logits, stream=None):
        lib = L.load()
        _check(lib.moe_verify_plan(C.byref(self._cfg), _ptr(P), _ptr(parent), _ptr(own_fp), _ptr(gamma_per_seq),
                                   _ptr(node_logits), _ptr(self.selected), _ptr(self.union_size),
                                   _ptr(self.verify_rows), _ptr(self.verify_conf), _ptr(self.ids), _ptr(self.w),
                                   _ptr(self.n_unique), _ptr(self.unique), _ptr(self.offsets),
                                   _ptr(self.perm_token), _ptr(self.perm_slot), _ptr(self.inv),
                                   _ptr(self.reuse_ratio), _ptr(self.dev_err), _stream(stream)),
               "moe_verify_plan")
        return self

    def capture(self, P, parent, own_fp, gamma_per_seq, node_logits, steps: int = 1):
        """Records `steps` control paths on these input tensors into a CUDA graph and returns it
        (as VerifyStep.capture: no host launch work at replay; inputs are read at replay time)."""
        args = (P, parent, own_fp, gamma_per_seq, node_logits)
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self(*args)  # warm-up outside the capture
        torch.cuda.current_stream(self.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(steps):
                self(*args)
        return graph


def s2_expand(P: torch.Tensor, parent: torch.Tensor, own_fp: torch.Tensor, T_AR: float, T_exp: float,
              C_draft: float = 0.0, dev_err: Optional[torch.Tensor] = None, stream=None,
              T_cold: float = 0.0, cold_fp: Optional[torch.Tensor] = None):
    """S2-MoE utility expansion per sequence: (selected [nseq, N] ascending
    then -1, n_selected [nseq], union_size [nseq]).  ``cold_fp`` [W] int32
    marks non-resident experts (bit l*E + e); each new cold expert costs
    T_cold on top of T_exp."""
    lib = L.load()
    nseq, N = P.shape
    W = own_fp.shape[-1]
    _need(P, torch.float32, (nseq, N), "P")
    _need(parent, torch.int32, (nseq, N), "parent")
    _need(own_fp, torch.int32, (nseq, N, W), "own_fp")
    dev = P.device
    selected = torch.empty((nseq, N), dtype=torch.int32, device=dev)
    n_sel = torch.empty(nseq, dtype=torch.int32, device=dev)
    usize = torch.empty(nseq, dtype=torch.int32, device=dev)
    if cold_fp is not None:
        _need(cold_fp, torch.int32, (W,), "cold_fp")
    cfg = L.S2Cfg(N, W, T_AR, T_exp, C_draft, T_cold, _ptr(cold_fp))
    _check(lib.s2_expand(_ptr(P), _ptr(parent), _ptr(own_fp), nseq, C.byref(cfg), _ptr(selected), _ptr(n_sel),
                         _ptr(usize), _ptr(dev_err), _stream(stream)), "s2_expand")
    return selected, n_sel, usize


def profile_begin(max_launches: int = 65536, classes: Optional[Sequence[str]] = None):
    """Start event timing of the library's launches (all classes by default)."""
    names = L.PROF_CLASSES if classes is None else classes
    mask = 0
    for n in names:
        mask |= 1 << L.PROF_CLASSES.index(n)
    _check(L.load().moe_profile_begin(max_launches, mask), "moe_profile_begin")


def profile_end() -> Dict[str, Dict[str, float]]:
    n = len(L.PROF_CLASSES)
    ms = (C.c_float * n)()
    cnt = (C.c_int32 * n)()
    _check(L.load().moe_profile_end(ms, cnt, n), "moe_profile_end")
    return {name: {"ms": float(ms[i]), "launches": int(cnt[i])} for i, name in enumerate(L.PROF_CLASSES)}


def launch_count() -> int:
    return int(L.load().moe_launch_count())


def set_nvtx(on: bool) -> None:
    """NVTX ranges around each step/plan enqueue, its selection and its layers (off by default)."""
    _check(L.load().moe_set_nvtx(1 if on else 0), "moe_set_nvtx")

"""Device-side materialisation of a workload: weights filled on the GPU with
the counter hash (workload/fill.cu, same definition as counter_hash.py) and
the host arrays copied over.  Input generation only."""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

from . import counter_hash as ch
from . import gen

_GEN_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoegen.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_GEN_LIB):
            raise ImportError(f"{_GEN_LIB} not built (run __graft_entry__.build())")
        _lib = C.CDLL(_GEN_LIB)
        _lib.gen_fill.argtypes = [C.c_void_p, C.c_int, C.c_uint64, C.c_uint64, C.c_uint64, C.c_void_p]
        _lib.gen_fill.restype = C.c_int
    return _lib


def fill(t: torch.Tensor, kind: int, key: int, idx0: int = 0):
    st = _load().gen_fill(t.data_ptr(), kind, t.numel(), key, idx0,
                          torch.cuda.current_stream().cuda_stream)
    if st != 0:
        raise RuntimeError(f"gen_fill failed ({st})")


def make_layer_tensors(cfg: gen.MoEConfig, layer: int, device="cuda"):
    """(gate_up, down, scales_gate_up, scales_down) device tensors of one layer,
    in the row-major layout."""
    shp = gen.weight_shapes(cfg)
    keys = gen.weight_stream_keys(cfg, layer)
    tdt = {"f32": torch.float32, "bf16": torch.int16, "e4m3": torch.uint8}[cfg.dtype]
    kind = gen.weight_kind(cfg)
    gu = torch.empty(shp["gate_up"], dtype=tdt, device=device)
    dn = torch.empty(shp["down"], dtype=tdt, device=device)
    fill(gu, kind, keys["gate_up"])
    fill(dn, kind, keys["down"])
    sgu = sdn = None
    if cfg.dtype == "e4m3":
        sgu = torch.empty(shp["scale_gate_up"], dtype=torch.float32, device=device)
        sdn = torch.empty(shp["scale_down"], dtype=torch.float32, device=device)
        fill(sgu, ch.KIND_SCALE_F32, keys["scale_gate_up"])
        fill(sdn, ch.KIND_SCALE_F32, keys["scale_down"])
    return gu, dn, sgu, sdn


def make_router_tensor(cfg: gen.MoEConfig, layer: int, device="cuda"):
    """W_r [E, H] of one layer on the device (int16 bf16 bits or float32)."""
    f32 = gen.router_dtype(cfg) == "f32"
    w = torch.empty((cfg.E, cfg.H), dtype=torch.float32 if f32 else torch.int16, device=device)
    fill(w, ch.KIND_GRID8_F32 if f32 else ch.KIND_GRID8_BF16, gen.router_stream_key(cfg, layer))
    return w


def workload_tensors(wl: gen.Workload, device="cuda"):
    """Host arrays of the workload as device tensors (int16 view for bf16 bits)."""
    cfg = wl.cfg
    nseq = cfg.nseq
    t = {
        "P": torch.from_numpy(wl.P.copy()).to(device),
        "parent": torch.from_numpy(np.tile(wl.parent, (nseq, 1)).astype(np.int32)).to(device),
        "own_fp": torch.from_numpy(wl.own_fp.view(np.int32).copy()).to(device),
        "gamma": torch.from_numpy(wl.gamma.copy()).to(device),
        "logits": torch.from_numpy(wl.logits.copy()).to(device),
    }
    if cfg.dtype == "f32":
        t["x"] = torch.from_numpy(wl.x.copy()).to(device)
    else:
        t["x"] = torch.from_numpy(wl.x.view(np.int16).copy()).to(device)
    return t

"""Benchmark of the MoE speculative verify step on GB300.

One step = EcoSpec selection over the draft tree(s) + every MoE layer's route
(optionally reuse-biased), expert union/permutation, grouped SwiGLU expert FFN
and combine, on the workload's synthetic inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Metric: HBM GB/s on the bytes of the unique experts the step must read
(sum over layers of |union| x expert bytes) divided by the device time of the
step.  Also reported: verify-step latency, tokens/s, the roofline of the
dominant kernel (FFN gate/up), clocks during the timed region, the end-to-end
number through the C ABI with host buffers, and the CPU oracle baseline.
Multi-GPU: independent replicas (the path has no exchange step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "qwen3_235b_like"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-residency", action="store_true", help="skip the expert-residency measurement")
    ap.add_argument("--residency", action="store_true",
                    help="run the expert-residency measurement even on a --layers/--experts profiling run")
    ap.add_argument("--residency-fracs", default="1,0.75,0.5,0.25,0",
                    help="hot fractions of the residency sweep (comma-separated)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: keep the first N layers of the workload (recorded in config)")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling only: use this many experts per layer (recorded in config)")
    ap.add_argument("--workloads", default="all", choices=["all", "none"],
                    help="all: after the headline workload, measure every other workload too")
    ap.add_argument("--quick", action="store_true",
                    help="skip the headline's sweeps (cost model, reuse bias, residency)")
    ap.add_argument("--cpu-layers", type=int, default=0,
                    help="layers in the CPU oracle sample (0: auto, about 10-30 s)")
    return ap.parse_args()


def dist_setup(n):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(v, ws, op_name):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    # NCCL reduces device tensors; gloo (the CPU tests of this path) host tensors.
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=getattr(dist.ReduceOp, op_name))
    return float(t.item())


def max_over_ranks(v, ws):
    return _reduce(v, ws, "MAX")


def sum_over_ranks(v, ws):
    return _reduce(v, ws, "SUM")


def job_throughput(bytes_local, ms_local, ws):
    """Whole-job GB/s of independent replicas: the bytes every rank moved over
    the slowest rank's time; returns (GB/s, that time in ms)."""
    ms_total = max_over_ranks(ms_local, ws)
    total = sum_over_ranks(bytes_local, ws)
    return total / (ms_total / 1e3) / 1e9, ms_total


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks/throttle sampling around and during the timed region.

    A reader thread collects one line every 50 ms with its host time.  Entering
    waits (at most 3 s) until the first line has arrived, so the sampler is
    live before the caller loads the GPU; the caller marks the timed region
    (`mark_start`, `mark_end`) and keeps the same load on the GPU for a few
    hundred ms on either side of it, so that a region of tens of ms still
    has samples under its own load around it."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []  # (host time, line)
        self.t_start = self.t_end = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        t0 = time.perf_counter()
        while not self.lines and time.perf_counter() - t0 < 3.0 and self.proc.poll() is None:
            time.sleep(0.01)
        self.lines.clear()  # the first line may precede the load
        return self

    def mark_start(self):
        self.t_start = time.perf_counter()

    def mark_end(self):
        self.t_end = time.perf_counter()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.reader.join(timeout=5)

    def summary(self):
        sm, smax, reasons, inside = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in list(self.lines):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
            if self.t_start is not None and self.t_end is not None and self.t_start <= t <= self.t_end:
                inside += 1
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        loaded = [v for v in sm if v > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_min_mhz": min(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm), "samples_in_timed_region": inside,
                "interval_ms": self.INTERVAL_MS,
                "window": "the timed region plus about 0.3 s of the same work before and after it"}


def kernel_source_hash():
    """Hash of the sources that define the bf16 FFN kernels (their translation
    unit, its PTX wrappers, the stream-K order and the next-layer L2
    prefetch); ties committed ncu traffic to the code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "serving_router_softmax_gb300", "csrc")
    for f in ("ffn_tc.cu", "ffn_internal.cuh", "tc_ptx.cuh", "stream_k.cuh", "l2_prefetch.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(config_name):
    """Per-launch DRAM bytes of the gate/up kernel from a committed ncu summary,
    only if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", f"ffn_gate_up_traffic_{config_name}.txt")
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if "=" in line and not line.startswith("#"):
            k, v = line.split("=", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_unit_expert"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------- our arm
def expert_bytes(cfg):
    elem = {"f32": 4, "bf16": 2, "e4m3": 1}[cfg.dtype]
    b = 3 * cfg.H * cfg.I * elem
    if cfg.dtype == "e4m3":
        b += 4 * ((2 * cfg.I // 128) * (cfg.H // 128) + (cfg.H // 128) * (cfg.I // 128))
    return b


def gate_up_bytes(cfg):
    elem = {"f32": 4, "bf16": 2, "e4m3": 1}[cfg.dtype]
    b = 2 * cfg.H * cfg.I * elem
    if cfg.dtype == "e4m3":
        b += 4 * (2 * cfg.I // 128) * (cfg.H // 128)
    return b


def cost_model_and_expansion(mv, cfg, layers, layout, dev, stream, steps=20):
    """The verify-cost model of the S2-MoE write-up (Fig. 6), checked on this
    GPU: the whole step at several draft budgets and both selection modes,
    step time fitted against the total expert union (T_exp = slope, R^2,
    MAPE); then s2_expand on the workload's trees with that T_exp, T_AR = the
    measured step with no draft token (one autoregressive token: the root
    alone) and C_draft = 0."""
    import torch
    from workload import gen
    from workload import device as wdev

    pts = []
    # 0 marginal, 1 static, 2 batch-global (batches only), 3 confidence only:
    # the marginal greedy with empty predicted footprints takes the top-gamma
    # nodes by path probability, the selection of a confidence-driven drafter.
    modes = (0, 1, 2, 3) if cfg.nseq > 1 else (0, 1, 3)
    for mode in modes:
        for g in (0, 1, 2, 3, 4, 5, 6, 8):
            c2 = cfg.replace(gamma=g, mode=0 if mode == 3 else mode, ragged=False)
            wl2 = gen.make_workload(c2)
            t2 = wdev.workload_tensors(wl2, dev)
            if mode == 3:
                t2["own_fp"].zero_()
            spec = mv.StepSpec(L=c2.L, nseq=c2.nseq, N=wl2.parent.shape[0], W=c2.W, E=c2.E, k=c2.k, H=c2.H,
                               I=c2.I, dtype=c2.dtype, T=wl2.T, gamma_max=int(wl2.gamma.max()), mode=c2.mode,
                               eps=c2.eps, use_bias=c2.use_bias, cap=c2.cap, alpha=c2.alpha, layout=layout)
            step = mv.VerifyStep(spec, layers, dev)

            def one():
                step(t2["P"], t2["parent"], t2["own_fp"], t2["gamma"], t2["logits"], t2["x"])

            for _ in range(3):
                one()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                one()
            e1.record(stream)
            torch.cuda.synchronize()
            pts.append({"gamma": g, "mode": ["marginal", "static", "batch_global", "confidence"][mode],
                        "tokens": int(wl2.T),
                        "union_experts": int(step.n_unique.sum().item()),
                        "ms": e0.elapsed_time(e1) / steps})
            del step
    # Predictor mismatch: marginal selection at gamma = 4 from footprints of
    # an imperfect predictor (top-K accuracy a), verified against the true
    # routing; the union is what the step actually loads.
    mism = []
    for acc in (1.0, 0.93, 0.82, 0.5):
        c2 = cfg.replace(gamma=4, mode=0, ragged=False)
        wl2 = gen.make_workload(c2)
        t2 = wdev.workload_tensors(wl2, dev)
        if acc < 1.0:
            t2["own_fp"] = torch.from_numpy(gen.perturbed_footprints(wl2, acc).view(np.int32).copy()).to(dev)
        spec = mv.StepSpec(L=c2.L, nseq=c2.nseq, N=wl2.parent.shape[0], W=c2.W, E=c2.E, k=c2.k, H=c2.H, I=c2.I,
                           dtype=c2.dtype, T=wl2.T, gamma_max=int(wl2.gamma.max()), mode=0, eps=c2.eps,
                           use_bias=c2.use_bias, cap=c2.cap, alpha=c2.alpha, layout=layout)
        step = mv.VerifyStep(spec, layers, dev)
        for _ in range(3):
            step(t2["P"], t2["parent"], t2["own_fp"], t2["gamma"], t2["logits"], t2["x"])
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step(t2["P"], t2["parent"], t2["own_fp"], t2["gamma"], t2["logits"], t2["x"])
        e1.record(stream)
        torch.cuda.synchronize()
        mism.append({"topk_accuracy": acc, "union_experts": int(step.n_unique.sum().item()),
                     "ms": e0.elapsed_time(e1) / steps})
        del step

    x = np.array([p["union_experts"] for p in pts], dtype=np.float64)
    y = np.array([p["ms"] for p in pts], dtype=np.float64) * 1e3  # us
    A = np.stack([np.ones_like(x), x], axis=1)
    (a, b), *_ = np.linalg.lstsq(A, y, rcond=None)
    pred = a + b * x
    r2 = 1.0 - float(np.sum((y - pred) ** 2) / np.sum((y - y.mean()) ** 2))
    mape = float(np.mean(np.abs(pred - y) / y))
    model = {"points": pts, "predictor_mismatch": mism, "T_exp_us": float(b), "intercept_us": float(a),
             "r2": r2, "mape": mape,
             "fit": "step_us = intercept + T_exp * (sum over layers of unique experts)"}

    # S2-MoE expansion on the workload's own trees with the calibrated cost.
    wl = gen.make_workload(cfg)
    t = wdev.workload_tensors(wl, dev)
    T_exp = max(float(b), 0.0)  # a least-squares slope; never negative as a cost
    T_AR = 1e3 * next(p["ms"] for p in pts if p["gamma"] == 0)
    sel, n_sel, usize = mv.s2_expand(t["P"], t["parent"], t["own_fp"], T_AR, T_exp, 0.0)
    for _ in range(3):
        mv.s2_expand(t["P"], t["parent"], t["own_fp"], T_AR, T_exp, 0.0)
    torch.cuda.synchronize()
    mv.profile_begin(max_launches=128, classes=["s2_expand"])
    for _ in range(100):
        mv.s2_expand(t["P"], t["parent"], t["own_fp"], T_AR, T_exp, 0.0)
    torch.cuda.synchronize()
    sp = mv.profile_end()["s2_expand"]
    expansion = {"T_AR_us": T_AR, "T_exp_us": T_exp, "C_draft_us": 0.0,
                 "selected_per_seq": n_sel.cpu().tolist(), "predicted_union_experts": usize.cpu().tolist(),
                 "draft_nodes": int(wl.parent.shape[0]),
                 "us_per_call": sp["ms"] * 1e3 / max(sp["launches"], 1)}
    return model, expansion


def reuse_bias_sweep(mv, cfg, layers, layout, dev, stream, steps=20):
    """S2-MoE reuse-aware gating on the bench's workload: the whole step with
    the bias off and at alpha in {0.1, 0.25, 0.5, 1} (cap = the workload's, or
    8), reporting the mean union per layer, the reuse ratio and the step time.
    The bias only re-ranks experts inside E* (a subset of the unbiased union),
    so the union can only shrink; what it costs in routing fidelity is the
    write-up's accuracy question, out of scope here."""
    import torch
    from workload import gen
    from workload import device as wdev
    cap = cfg.cap if cfg.use_bias else 8
    pts = []
    for alpha in (None, 0.1, 0.25, 0.5, 1.0):
        c2 = cfg.replace(use_bias=alpha is not None, cap=cap, alpha=alpha if alpha is not None else 0.25)
        wl2 = gen.make_workload(c2)
        t2 = wdev.workload_tensors(wl2, dev)
        spec = mv.StepSpec(L=c2.L, nseq=c2.nseq, N=wl2.parent.shape[0], W=c2.W, E=c2.E, k=c2.k, H=c2.H,
                           I=c2.I, dtype=c2.dtype, T=wl2.T, gamma_max=int(wl2.gamma.max()), mode=c2.mode,
                           eps=c2.eps, use_bias=c2.use_bias, cap=c2.cap, alpha=c2.alpha, layout=layout)
        step = mv.VerifyStep(spec, layers, dev)
        args = (t2["P"], t2["parent"], t2["own_fp"], t2["gamma"], t2["logits"], t2["x"])
        for _ in range(3):
            step(*args)
        torch.cuda.synchronize()
        if int(step.dev_err.item()) != 0:
            raise RuntimeError(f"device error bits {int(step.dev_err.item())}")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step(*args)
        e1.record(stream)
        torch.cuda.synchronize()
        nu = step.n_unique.cpu().tolist()
        plan = mv.VerifyPlan(spec, dev)
        plan(t2["P"], t2["parent"], t2["own_fp"], t2["gamma"], t2["logits"])
        torch.cuda.synchronize()
        pts.append({"alpha": alpha, "cap": cap if alpha is not None else None,
                    "union_per_layer": sum(nu) / len(nu),
                    "reuse_ratio": float(plan.reuse_ratio.mean().item()),
                    "ms_per_step": e0.elapsed_time(e1) / steps})
        del step, plan
    return {"points": pts, "tokens": int(gen.make_workload(cfg).T),
            "note": "alpha None = bias off; union and time at the workload's own draft tree"}


def host_mem_available():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def residency_expansion(mv, cfg, layout, dev, expansion, T_cold, hot_frac=0.5):
    """S2-MoE expansion priced for residency: every layer keeps its hot_frac
    most routed experts (from a calibration workload) resident, a new cold
    expert costs T_cold (measured) on top of T_exp.  Compared with the plain
    expansion on the same trees: nodes taken, predicted union and its cold
    part (host-side bookkeeping of the outputs)."""
    import torch
    from workload import gen
    from workload import device as wdev

    cal = cfg.replace(seed=cfg.seed + 1000)
    wl_cal = gen.make_workload(cal)
    t_cal = wdev.workload_tensors(wl_cal, dev)
    spec_cal = mv.StepSpec(L=cal.L, nseq=cal.nseq, N=wl_cal.parent.shape[0], W=cal.W, E=cal.E, k=cal.k,
                           H=cal.H, I=cal.I, dtype=cal.dtype, T=wl_cal.T, gamma_max=int(wl_cal.gamma.max()),
                           mode=cal.mode, eps=cal.eps, use_bias=cal.use_bias, cap=cal.cap, alpha=cal.alpha,
                           layout=layout)
    plan = mv.VerifyPlan(spec_cal, dev)
    plan(t_cal["P"], t_cal["parent"], t_cal["own_fp"], t_cal["gamma"], t_cal["logits"])
    torch.cuda.synchronize()
    n_hot = int(round(hot_frac * cfg.E))
    cold_bits = np.zeros(cfg.W, dtype=np.uint32)
    for l in range(cfg.L):
        hot = set(mv.hot_list(plan.ids[l].reshape(-1), cfg.E, n_hot)[0].cpu().tolist())
        for e in range(cfg.E):
            if e not in hot:
                b = l * cfg.E + e
                cold_bits[b // 32] |= np.uint32(1 << (b % 32))
    wl = gen.make_workload(cfg)
    t = wdev.workload_tensors(wl, dev)
    cold_t = torch.from_numpy(cold_bits.view(np.int32).copy()).to(dev)

    def is_cold(l, e):
        b = l * cfg.E + e
        return bool((int(cold_bits[b // 32]) >> (b % 32)) & 1)

    # T_AR under the same residency: the measured all-resident step with no
    # draft token plus T_cold for every cold expert the root tokens route to.
    c0 = cfg.replace(gamma=0, ragged=False)
    wl0 = gen.make_workload(c0)
    t0 = wdev.workload_tensors(wl0, dev)
    spec0 = mv.StepSpec(L=c0.L, nseq=c0.nseq, N=wl0.parent.shape[0], W=c0.W, E=c0.E, k=c0.k, H=c0.H, I=c0.I,
                        dtype=c0.dtype, T=wl0.T, gamma_max=0, mode=c0.mode, eps=c0.eps, use_bias=c0.use_bias,
                        cap=c0.cap, alpha=c0.alpha, layout=layout)
    plan0 = mv.VerifyPlan(spec0, dev)
    plan0(t0["P"], t0["parent"], t0["own_fp"], t0["gamma"], t0["logits"])
    torch.cuda.synchronize()
    nu0 = plan0.n_unique.cpu().tolist()
    root_cold = sum(is_cold(l, int(e)) for l in range(cfg.L) for e in plan0.unique[l][:nu0[l]].cpu().tolist())
    T_AR = expansion["T_AR_us"] + T_cold * root_cold
    out = {"hot_frac": hot_frac, "T_cold_us": T_cold, "T_exp_us": expansion["T_exp_us"],
           "T_AR_resident_us": expansion["T_AR_us"], "root_cold_experts": root_cold, "T_AR_us": T_AR,
           "T_AR": "all-resident step with no draft token + T_cold * cold experts of the root tokens"}
    for name, kw in (("plain", {}), ("residency_aware", {"T_cold": T_cold, "cold_fp": cold_t})):
        sel, n_sel, _ = mv.s2_expand(t["P"], t["parent"], t["own_fp"], T_AR, expansion["T_exp_us"], 0.0, **kw)
        sel, n_sel = sel.cpu().numpy(), n_sel.cpu().tolist()
        unions, colds = [], []
        for s_ in range(cfg.nseq):
            u = np.zeros(cfg.W, dtype=np.uint32)
            for node in sel[s_, :n_sel[s_]]:
                u |= wl.own_fp[s_][node]
            unions.append(int(sum(bin(int(w)).count("1") for w in u)))
            colds.append(int(sum(bin(int(w)).count("1") for w in (u & cold_bits))))
        gains = [float(sum(np.float64(wl.P[s_][node]) for node in sel[s_, :n_sel[s_]])) * T_AR
                 for s_ in range(cfg.nseq)]
        out[name] = {"selected_per_seq": n_sel, "predicted_union_experts": unions,
                     "predicted_cold_experts": colds,
                     "predicted_gain_us": gains,
                     "predicted_cost_us": [unions[i] * expansion["T_exp_us"] + colds[i] * T_cold
                                           for i in range(cfg.nseq)]}
    return out


def residency_measure(mv, cfg, layers, layout, dev, stream, expansion=None, n_layers=2, steps=10,
                      fracs=(1.0, 0.75, 0.5, 0.25, 0.0)):
    """Expert-level residency (S2-MoE write-up, system implementation): the
    first n_layers layers of the workload with every expert in page-locked
    Grace memory and a profiled hot list resident in HBM; each step stages
    its union's cold experts over NVLink-C2C (moe_stage_experts inside the
    step).  Hot lists come from the routing counts of a calibration workload
    (another seed), not the timed one.  Reported per hot fraction: step time,
    staging time and bytes, the staging kernel's link rate; plus the copy
    engine's host->device rate over the same link and the cold-expert cost
    fitted from the step times."""
    import torch
    from workload import gen
    from workload import device as wdev

    c2 = cfg.replace(L=min(n_layers, cfg.L))
    need = c2.L * c2.E * expert_bytes(c2)
    if host_mem_available() < 2 * need:
        return {"skipped": f"needs {2 * need / 2**30:.1f} GiB of free host memory"}
    host = mv.HostExperts(layers[:c2.L])
    ebytes = host.gate_up_bytes + host.down_bytes

    # Copy-engine reference over the same link: one 1 GiB pinned -> device copy.
    src = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    best = None
    for _ in range(5):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        dst.copy_(src, non_blocking=True)
        a1.record(stream)
        torch.cuda.synchronize()
        ms = a0.elapsed_time(a1)
        best = ms if best is None else min(best, ms)
    ce_gbs = (1 << 30) / (best / 1e3) / 1e9
    del src, dst

    # Offline profiling: routing counts of a calibration workload.
    cal = cfg.replace(L=c2.L, seed=cfg.seed + 1000)
    wl_cal = gen.make_workload(cal)
    t_cal = wdev.workload_tensors(wl_cal, dev)
    spec_cal = mv.StepSpec(L=cal.L, nseq=cal.nseq, N=wl_cal.parent.shape[0], W=cal.W, E=cal.E, k=cal.k,
                           H=cal.H, I=cal.I, dtype=cal.dtype, T=wl_cal.T, gamma_max=int(wl_cal.gamma.max()),
                           mode=cal.mode, eps=cal.eps, use_bias=cal.use_bias, cap=cal.cap, alpha=cal.alpha,
                           layout=layout)
    plan_cal = mv.VerifyPlan(spec_cal, dev)
    plan_cal(t_cal["P"], t_cal["parent"], t_cal["own_fp"], t_cal["gamma"], t_cal["logits"])
    torch.cuda.synchronize()
    prof_ids = [plan_cal.ids[l].reshape(-1).clone() for l in range(cal.L)]

    wl2 = gen.make_workload(c2)
    t2 = wdev.workload_tensors(wl2, dev)
    spec = mv.StepSpec(L=c2.L, nseq=c2.nseq, N=wl2.parent.shape[0], W=c2.W, E=c2.E, k=c2.k, H=c2.H, I=c2.I,
                       dtype=c2.dtype, T=wl2.T, gamma_max=int(wl2.gamma.max()), mode=c2.mode, eps=c2.eps,
                       use_bias=c2.use_bias, cap=c2.cap, alpha=c2.alpha, layout=layout)
    plan = mv.VerifyPlan(spec, dev)
    plan(t2["P"], t2["parent"], t2["own_fp"], t2["gamma"], t2["logits"])
    torch.cuda.synchronize()
    n_unique = plan.n_unique.cpu()
    unique = [plan.unique[l][:int(n_unique[l])].cpu() for l in range(c2.L)]
    args = (t2["P"], t2["parent"], t2["own_fp"], t2["gamma"], t2["logits"], t2["x"])

    def timed(step):
        for _ in range(3):
            step(*args)
        torch.cuda.synchronize()
        if int(step.dev_err.item()) != 0:
            raise RuntimeError(f"device error bits {int(step.dev_err.item())}")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step(*args)
        e1.record(stream)
        torch.cuda.synchronize()
        mv.profile_begin(max_launches=steps * c2.L + 16, classes=["stage_experts"])
        for _ in range(steps):
            step(*args)
        torch.cuda.synchronize()
        st = mv.profile_end()["stage_experts"]
        return e0.elapsed_time(e1) / steps, st["ms"] / steps

    base = mv.VerifyStep(spec, layers[:c2.L], dev)
    resident_ms, _ = timed(base)
    y_ref = base.y.clone()
    del base
    cap_union = min(c2.E, wl2.T * c2.k)
    pts = []
    for frac in fracs:
        n_hot = int(round(frac * c2.E))
        hot = [mv.hot_list(prof_ids[l], c2.E, n_hot)[0].cpu().tolist() for l in range(c2.L)]
        pool = mv.ExpertPool(host, hot, n_stage=min(c2.E - n_hot, cap_union), device=dev)
        step = mv.VerifyStep(spec, pool.layers, dev)
        ms, stage_ms = timed(step)
        same = bool(torch.equal(step.y, y_ref))
        cold = sum(int((pool.home_slot[l].cpu()[unique[l].long()] == -1).sum()) for l in range(c2.L))
        pts.append({"hot_frac": frac, "n_hot": n_hot, "n_stage": pool.n_stage,
                    "device_gb": pool.n_slots * ebytes / 1e9, "cold_experts_per_step": cold,
                    "staged_gb_per_step": cold * ebytes / 1e9, "ms_per_step": ms,
                    "stage_ms_per_step": stage_ms,
                    "stage_gbs": (cold * ebytes / 1e9) / (stage_ms / 1e3) if cold and stage_ms > 0 else None,
                    "output_equals_resident": same})
        del step, pool
        torch.cuda.empty_cache()
    x = np.array([0.0] + [p["cold_experts_per_step"] for p in pts], dtype=np.float64)
    y = np.array([resident_ms] + [p["ms_per_step"] for p in pts], dtype=np.float64) * 1e3
    A = np.stack([np.ones_like(x), x], axis=1)
    (a, b), *_ = np.linalg.lstsq(A, y, rcond=None)
    pred = a + b * x
    r2 = 1.0 - float(np.sum((y - pred) ** 2) / max(np.sum((y - y.mean()) ** 2), 1e-30))
    res = {"layers": c2.L, "expert_mb": ebytes / 1e6, "union_experts": [int(v) for v in n_unique],
           "resident_ms_per_step": resident_ms, "copy_engine_h2d_gbs": ce_gbs, "points": pts,
           "T_cold_us": float(b), "intercept_us": float(a), "r2": r2,
           "fit": "step_us = intercept + T_cold * (cold experts staged per step)",
           "T_cold_us_at_copy_engine_rate": ebytes / (ce_gbs * 1e9) * 1e6,
           "hot_list": "per layer, the most routed experts of a calibration workload (seed + 1000)"}
    if expansion is not None:
        res["s2_expand"] = residency_expansion(mv, cfg, layout, dev, expansion, max(float(b), 0.0))
    return res


def router_measure(mv, cfg, wl, dev, stream, iters=200):
    """Gate logits of the step's verify tokens (T x H activations against one
    layer's E x H gate), timed with CUDA events over back-to-back launches that
    cycle through enough distinct gate matrices to exceed L2."""
    import torch
    from workload import device as wdev

    T = wl.T
    rows = wl.x[0].reshape(-1, cfg.H)[:T]
    x = torch.from_numpy(rows.copy() if cfg.dtype == "f32" else rows.view(np.int16).copy()).to(dev)
    first = wdev.make_router_tensor(cfg, 0, dev)
    per = first.numel() * first.element_size()
    n_mats = max(2, -(-(256 << 20) // per))
    mats = [first] + [wdev.make_router_tensor(cfg, l, dev) for l in range(1, n_mats)]
    out = torch.empty((T, cfg.E), dtype=torch.float32, device=dev)
    for i in range(3):
        mv.router_logits(x, mats[i % n_mats], out=out)
    torch.cuda.synchronize()
    # events around each launch (the library's profiler), so host-side call
    # overhead between launches is not counted as kernel time
    mv.profile_begin(max_launches=iters + 8, classes=["router_logits"])
    for i in range(iters):
        mv.router_logits(x, mats[i % n_mats], out=out)
    torch.cuda.synchronize()
    rp = mv.profile_end()["router_logits"]
    us = rp["ms"] * 1e3 / max(rp["launches"], 1)
    nbytes = per + x.numel() * x.element_size() + out.numel() * 4
    peak, peak_kind = peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    del mats
    torch.cuda.empty_cache()
    return {"T": T, "H": cfg.H, "E": cfg.E, "w_dtype": "f32" if cfg.dtype == "f32" else "bf16",
            "us_per_launch": us, "algorithmic_bytes": nbytes, "achieved_gbs": gbs,
            "frac_of_peak": gbs / peak, "peak_kind": peak_kind, "bound": "latency",
            "timed": f"CUDA events around each of {iters} launches over {n_mats} distinct gate matrices "
                     f"({n_mats * per / 2**20:.0f} MiB > L2)"}


def build_layers(mv, cfg, dev):
    """Device weights of every layer: filled row-major, then (bf16, FP8) packed
    once into the tiled layout the tensor-core FFN streams; a load-time step
    outside every timed region."""
    import torch
    from workload import device as wdev
    layout = "tiled" if cfg.dtype in ("bf16", "e4m3") else "rowmajor"
    layers = []
    for l in range(cfg.L):
        gu, dn, sgu, sdn = wdev.make_layer_tensors(cfg, l, dev)
        layer = mv.ExpertLayer(gu, dn, cfg.dtype, sgu, sdn)
        if layout == "tiled":
            layer = mv.pack_tiled(layer)
            del gu, dn, sgu, sdn
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        layers.append(layer)
    return layers, layout


def step_spec(mv, cfg, wl, layout):
    return mv.StepSpec(L=cfg.L, nseq=cfg.nseq, N=wl.parent.shape[0], W=cfg.W, E=cfg.E, k=cfg.k,
                       H=cfg.H, I=cfg.I, dtype=cfg.dtype, T=wl.T, gamma_max=int(wl.gamma.max()), mode=cfg.mode,
                       eps=cfg.eps, use_bias=cfg.use_bias, cap=cfg.cap, alpha=cfg.alpha, layout=layout)


def e2e_measure(mv, spec, layers, t, dev, stream, steps, ws, total_bytes):
    """End to end through the public API with host buffers, as a serving loop
    runs it: every step's inputs go host -> device from pinned memory and its
    result comes back device -> host, all inside the timed region.  Two
    input/output buffer sets: while step s runs (a CUDA graph of the whole
    step), step s+1's inputs are copied in and step s-1's result is copied out
    on two copy streams."""
    import torch
    names = ("P", "parent", "own_fp", "gamma", "logits", "x")
    pinned = [{k: t[k].cpu().pin_memory() for k in names} for _ in range(2)]
    steps2 = [mv.VerifyStep(spec, layers, dev) for _ in range(2)]
    y_host = [torch.empty(steps2[0].y.shape, dtype=steps2[0].y.dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pinned[0].values())
    d2h = y_host[0].numel() * y_host[0].element_size()
    dev_in = [{k: torch.empty_like(t[k]) for k in names} for _ in range(2)]
    for b in range(2):
        for k in names:
            dev_in[b][k].copy_(t[k])
    graphs = [steps2[b].capture(*[dev_in[b][k] for k in names]) for b in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def loop(n, start_event=None):
        if start_event is not None:
            s_in.wait_event(start_event)
            s_out.wait_event(start_event)
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_run[b])  # step i-2 has read this input set
                for k in names:
                    dev_in[b][k].copy_(pinned[b][k], non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # step i-2's result has left this output buffer
            graphs[b].replay()
            ev_run[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[b])
                y_host[b].copy_(steps2[b].y, non_blocking=True)
                ev_out[b].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    loop(4)
    torch.cuda.synchronize()
    barrier(ws)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    loop(steps, a0)
    a1.record(stream)
    torch.cuda.synchronize()
    for b in range(2):
        if int(steps2[b].dev_err.item()) != 0:
            raise SystemExit(f"device error {int(steps2[b].dev_err.item())} in the e2e loop")
    e2e_ms = max_over_ranks(a0.elapsed_time(a1), ws)
    del graphs, steps2
    return {"value": total_bytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms / steps,
            "loop": "pinned host inputs in and result out every step, double-buffered: the next step's "
                    "inputs and the previous step's result cross on two copy streams while a step runs "
                    "(CUDA graph replay)",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def measure_step(mv, cfg, wl, layers, layout, args, dev, stream, ws, local, config_name):
    """The step's measurements on one workload: pass A (headline: CUDA graph
    replays, clocks sampled), the same steps eager, pass B (events around the
    FFN gate/up and down launches only: the roofline of each), pass C
    (events around every launch: the per-kernel breakdown), the control path
    alone, and the end-to-end loop with host buffers."""
    import torch
    from workload import device as wdev

    t = wdev.workload_tensors(wl, dev)
    spec = step_spec(mv, cfg, wl, layout)
    step = mv.VerifyStep(spec, layers, dev)

    def one():
        step(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    if int(step.dev_err.item()) != 0:
        raise RuntimeError(f"device error bits {int(step.dev_err.item())}")
    n_unique = step.n_unique.cpu().tolist()
    bytes_step = sum(n_unique) * expert_bytes(cfg)
    y_first = step.y[0].cpu()

    # ---- the step as a CUDA graph: the library's step makes no allocation and
    # no host synchronisation, so one captured step replays with no host
    # launch work; it is the headline pass below (eager stays as a second pass).
    l0 = mv.launch_count()
    one()
    launches_per_step = mv.launch_count() - l0
    graph = None
    graph_error = None
    try:
        graph = step.capture(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
        graph.replay()
        torch.cuda.synchronize()
    except RuntimeError as exc:  # capture unsupported: the eager pass is the headline
        graph, graph_error = None, f"unavailable: {exc}"

    def timed(fn):
        barrier(ws)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        return e0.elapsed_time(e1)

    # ---- pass A (headline): device-timed region, inputs resident in HBM,
    # unique-expert bytes per step >> L2; no per-kernel events.
    def keep_loaded(fn, seconds=0.3):
        # untimed repeats of the same step around the timed region, so that
        # the clock samples see this load (the region itself is tens of ms)
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            for _ in range(4):
                fn()
            torch.cuda.synchronize()

    step_fn = graph.replay if graph is not None else one
    with ClockSampler(local) as clk:
        keep_loaded(step_fn)
        clk.mark_start()
        ms_local = timed(step_fn)
        clk.mark_end()
        keep_loaded(step_fn)
    value, ms_total = job_throughput(bytes_step * args.steps, ms_local, ws)
    ms_step = ms_total / args.steps
    total_bytes = sum_over_ranks(bytes_step * args.steps, ws)
    tokens = sum_over_ranks(wl.T * args.steps, ws)
    # ---- the same K steps launched one by one from the host.
    eager_ms = max_over_ranks(timed(one), ws) / args.steps
    if graph is not None:
        del graph

    # ---- pass B: the same K steps with CUDA events around the FFN gate/up
    # and down launches only, on the stream they run on.
    mv.profile_begin(max_launches=2 * args.steps * cfg.L + 16, classes=["ffn_gate_up", "ffn_down"])
    torch.cuda.synchronize()
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(args.steps):
        one()
    b1.record(stream)
    torch.cuda.synchronize()
    pb = mv.profile_end()
    ms_pass_b = b0.elapsed_time(b1)

    # ---- pass C: per-kernel breakdown (events around every launch).
    n_c = min(args.steps, 50)
    mv.profile_begin(max_launches=n_c * (1 + 6 * cfg.L) + 16)
    for _ in range(n_c):
        one()
    torch.cuda.synchronize()
    prof = mv.profile_end()

    # ---- control path alone (selection + every layer's routing and union,
    # the same kernels and launch chain as in the step, without the FFN).
    plan = mv.VerifyPlan(spec, dev)

    def one_plan():
        plan(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"])

    for _ in range(3):
        one_plan()
    torch.cuda.synchronize()
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    n_plan = min(args.steps, 100)
    c0.record(stream)
    for _ in range(n_plan):
        one_plan()
    c1.record(stream)
    torch.cuda.synchronize()
    ctrl_eager_ms = c0.elapsed_time(c1) / n_plan
    # The headline step is timed as CUDA-graph replays, so its control path
    # is too (the same launches, without the host's per-launch work).
    g_plan = plan.capture(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"])
    for _ in range(3):
        g_plan.replay()
    torch.cuda.synchronize()
    c0.record(stream)
    for _ in range(n_plan):
        g_plan.replay()
    c1.record(stream)
    torch.cuda.synchronize()
    ctrl_ms = c0.elapsed_time(c1) / n_plan
    del g_plan, plan

    # ---- roofline of the FFN kernels, from pass B.
    peak, peak_kind = peaks()
    lines = {}
    for cls, per_unit in (("ffn_gate_up", gate_up_bytes(cfg)), ("ffn_down", expert_bytes(cfg) - gate_up_bytes(cfg))):
        k_ms = pb[cls]["ms"]
        nb = sum(n_unique) * per_unit * args.steps
        ach = nb / (k_ms / 1e3) / 1e9 if k_ms > 0 else None
        lines[cls] = {"bound": "hbm", "kernel": cls, "achieved": ach, "peak": peak, "peak_kind": peak_kind,
                      "unit": "GB/s", "frac": (ach / peak) if ach else None,
                      "algorithmic_bytes_per_launch": sum(n_unique) * per_unit / cfg.L,
                      "avg_launch_us": k_ms * 1e3 / max(pb[cls]["launches"], 1),
                      "launches": pb[cls]["launches"]}
    roofline = dict(lines["ffn_gate_up"])
    # Both FFN launches together: unaffected by the L2 prefetch that moves
    # part of the next layer's gate/up bytes into the down launch's time.
    pair_ms = pb["ffn_gate_up"]["ms"] + pb["ffn_down"]["ms"]
    pair_gbs = sum(n_unique) * expert_bytes(cfg) * args.steps / (pair_ms / 1e3) / 1e9 if pair_ms > 0 else None
    roofline["ffn_pair_frac"] = pair_gbs / peak if pair_gbs else None
    if cfg.dtype in ("bf16", "e4m3") and layout == "tiled" and cfg.L > 1:
        roofline["l2_prefetch"] = ("each down launch but the last asks L2 to fetch 30 MB of the next layer's "
                                   "predicted experts' gate/up weights (the selection's footprint union), which "
                                   "that gate/up launch then reads from L2: its fraction counts those bytes, the "
                                   "down fraction carries their time; ffn_pair_frac is unaffected")
    traffic_unit = committed_traffic(config_name)
    roofline["traffic"] = traffic_unit * sum(n_unique) / cfg.L if traffic_unit is not None else None
    roofline["timed_in"] = "pass B: the K timed steps repeated with events around the FFN launches only"
    roofline["pass_b_ms_per_step"] = ms_pass_b / args.steps
    roofline["ffn_down"] = lines["ffn_down"]

    e2e = e2e_measure(mv, spec, layers, t, dev, stream, args.steps, ws, total_bytes)
    core = {
        "value": value, "ms_per_step": ms_step, "latency_us": ms_step * 1e3,
        "tokens_per_s": tokens / (ms_total / 1e3),
        "unique_experts_per_layer": n_unique, "unique_expert_gb_per_step": bytes_step / 1e9,
        "frac_of_peak_step": value / peak / ws, "frac_of_8tbs_step": value / 8000.0 / ws,
        "roofline": roofline,
        "kernel_ms_per_step": {k: v["ms"] / n_c for k, v in prof.items()},
        "launch": "CUDA graph replay of the whole step" if graph_error is None else "eager (" + graph_error + ")",
        "eager_ms_per_step": eager_ms,
        "control_path_ms": ctrl_ms,
        "control_path_frac": ctrl_ms / max(ms_step, 1e-9),
        "control_path_eager_ms": ctrl_eager_ms,
        "control_path_eager_frac": ctrl_eager_ms / max(eager_ms, 1e-9),
        "control_path_frac_events": sum(prof[k]["ms"] for k in ("eco_select", "route", "union_permute"))
        / n_c / max(ms_step, 1e-9),
        "clocks": clk.summary(),
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "launches_per_step": launches_per_step,
    }
    del step
    return core, y_first


def gamma_sweep(mv, cfg, layers, layout, dev, stream, steps=20):
    """EcoSpec's draft-budget ablation (write-up section 4.3, gamma 3..6) on
    the workload, under marginal-cost and static-cost selection: the union per
    layer, the verify tokens and the step time (CUDA graph replays)."""
    import torch
    from workload import gen
    from workload import device as wdev
    pts = []
    for mode in (0, 1):
        for g in (3, 4, 5, 6):
            c2 = cfg.replace(gamma=g, mode=mode, ragged=False)
            wl2 = gen.make_workload(c2)
            t2 = wdev.workload_tensors(wl2, dev)
            step = mv.VerifyStep(step_spec(mv, c2, wl2, layout), layers, dev)
            args = (t2["P"], t2["parent"], t2["own_fp"], t2["gamma"], t2["logits"], t2["x"])
            for _ in range(3):
                step(*args)
            torch.cuda.synchronize()
            if int(step.dev_err.item()) != 0:
                raise RuntimeError(f"device error bits {int(step.dev_err.item())}")
            graph = step.capture(*args)
            graph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            nu = step.n_unique.cpu().tolist()
            ms = e0.elapsed_time(e1) / steps
            pts.append({"gamma": g, "selection": ["marginal", "static"][mode], "verify_tokens": int(wl2.T),
                        "union_per_layer": sum(nu) / len(nu), "ms_per_step": ms,
                        "gbs": sum(nu) * expert_bytes(c2) / (ms / 1e3) / 1e9})
            del graph, step
    return {"points": pts, "batch": cfg.nseq,
            "note": "every sequence verifies gamma draft nodes; EcoSpec write-up section 4.3 sweeps gamma 3..6"}


def _graph_ms(mv, spec, layers, t, dev, stream, steps):
    """Step time (CUDA graph replays) and per-layer unions of one workload."""
    import torch
    step = mv.VerifyStep(spec, layers, dev)
    args = (t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"], t["x"])
    for _ in range(3):
        step(*args)
    torch.cuda.synchronize()
    if int(step.dev_err.item()) != 0:
        raise RuntimeError(f"device error bits {int(step.dev_err.item())}")
    graph = step.capture(*args)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    nu = step.n_unique.cpu().tolist()
    del graph, step
    return e0.elapsed_time(e1) / steps, nu


def width_depth_measure(mv, cfg, layers, layout, dev, stream, steps=20):
    """The width-vs-depth note on this GPU, with the workload's layers.

    Section 1: verifying d consecutive positions of one sequence (the root and
    d - 1 chained drafts) against one token from each of d independent
    sequences: union per layer (mean over 8 seeds, from the plan) and the step
    time (first seed, CUDA graph replays).

    Section 2: batches of draft chains (6 positions, acceptance bimodal across
    sequences): every fixed depth 0..6 against the confidence-gated depth
    vector (moe_depth_policy, its cost model fitted to the fixed-depth step
    times).  Expected committed tokens per step = sum_i (1 + c_i1 + ... +
    c_id_i) under calibrated confidences; expected tokens/s = that / step."""
    import torch
    from workload import gen
    from workload import device as wdev

    def spec_of(c, wl):
        return step_spec(mv, c, wl, layout)

    sec1 = []
    for d in (2, 3, 4, 5, 6, 7):
        row = {"positions": d}
        for kind in ("depth", "width"):
            unions, ms = [], None
            for rep in range(8):
                if kind == "depth":
                    c = gen.chain_config(cfg, 1, depth=6, seed=2000 + 10 * d + rep, gamma=d - 1)
                else:
                    c = gen.chain_config(cfg, d, depth=6, seed=3000 + 10 * d + rep, gamma=0)
                wl = gen.make_workload(c)
                t = wdev.workload_tensors(wl, dev)
                spec = spec_of(c, wl)
                if rep == 0:
                    ms, nu = _graph_ms(mv, spec, layers, t, dev, stream, steps)
                else:
                    plan = mv.VerifyPlan(spec, dev)
                    plan(t["P"], t["parent"], t["own_fp"], t["gamma"], t["logits"])
                    torch.cuda.synchronize()
                    nu = plan.n_unique.cpu().tolist()
                    del plan
                unions.append(sum(nu) / len(nu))
            row[kind] = {"union_per_layer": sum(unions) / len(unions), "ms_per_step": ms}
        sec1.append(row)

    # Section 2.  Every fixed depth on several seeded batches per batch size;
    # one cost model fitted to all of them; then the gated depth vector.
    runs = []
    for nseq in (1, 2, 4, 8):
        for rep in range(4):
            c = gen.chain_config(cfg, nseq, depth=6, seed=4000 + 100 * nseq + rep)
            wl = gen.make_workload(c)
            conf = wl.P.astype(np.float32)
            A = 1.0 + np.concatenate([np.zeros((nseq, 1)), np.cumsum(conf.astype(np.float64), axis=1)], axis=1)
            fixed = []
            for Dc in range(7):
                c2 = c.replace(gamma=Dc)
                wl2 = gen.make_workload(c2)
                t2 = wdev.workload_tensors(wl2, dev)
                ms, nu = _graph_ms(mv, spec_of(c2, wl2), layers, t2, dev, stream, steps // 2)
                fixed.append({"union_experts": int(sum(nu)), "ms": ms, "exp_tokens": float(A[:, Dc].sum())})
            runs.append({"nseq": nseq, "c": c, "wl": wl, "conf": conf, "A": A, "fixed": fixed})
    x = np.array([f["union_experts"] for r in runs for f in r["fixed"]], np.float64)
    y = np.array([f["ms"] for r in runs for f in r["fixed"]], np.float64) * 1e3
    (C0, T_exp), *_ = np.linalg.lstsq(np.stack([np.ones_like(x), x], 1), y, rcond=None)
    pred = C0 + T_exp * x
    r2 = 1.0 - float(np.sum((y - pred) ** 2) / np.sum((y - y.mean()) ** 2))
    C0, T_exp = max(float(C0), 1.0), max(float(T_exp), 0.0)
    pol_us = []
    for r in runs:
        nseq, wl, conf = r["nseq"], r["wl"], r["conf"]
        fp = np.concatenate([wl.root_fp[:, None, :], wl.own_fp], axis=1)
        conf_d = torch.from_numpy(conf).to(dev)
        fp_d = torch.from_numpy(fp.view(np.int32)).to(dev)
        depth, common, thr = mv.depth_policy(conf_d, fp_d, C0, T_exp)
        torch.cuda.synchronize()
        mv.profile_begin(max_launches=64, classes=["depth_policy"])
        for _ in range(20):
            mv.depth_policy(conf_d, fp_d, C0, T_exp)
        torch.cuda.synchronize()
        pp = mv.profile_end()["depth_policy"]
        pol_us.append((nseq, pp["ms"] * 1e3 / max(pp["launches"], 1)))
        d = depth.cpu().numpy().astype(np.int32)
        # the step verifies each sequence's chain prefix of length d_i
        wl_g = gen.make_workload(r["c"].replace(gamma=int(d.max())))
        wl_g.gamma = d.copy()
        wl_g.T = int(np.sum(d + 1))
        t_g = wdev.workload_tensors(wl_g, dev)
        ms, nu = _graph_ms(mv, spec_of(r["c"], wl_g), layers, t_g, dev, stream, steps // 2)
        r["gated"] = {"depth": d.tolist(), "common": int(common.item()), "union_experts": int(sum(nu)), "ms": ms,
                      "exp_tokens": float(sum(r["A"][i, d[i]] for i in range(nseq)))}
    sec2 = []
    for nseq in (1, 2, 4, 8):
        rs = [r for r in runs if r["nseq"] == nseq]
        fixed_tps = [sum(r["fixed"][Dc]["exp_tokens"] for r in rs) / (sum(r["fixed"][Dc]["ms"] for r in rs) / 1e3)
                     for Dc in range(7)]
        gated_tps = sum(r["gated"]["exp_tokens"] for r in rs) / (sum(r["gated"]["ms"] for r in rs) / 1e3)
        best = int(np.argmax(fixed_tps))
        sec2.append({"batch": nseq, "batches": len(rs),
                     "fixed_expected_tokens_per_s": fixed_tps,
                     "gated_expected_tokens_per_s": gated_tps,
                     "best_fixed_depth": best,
                     "gated_over_best_fixed": gated_tps / fixed_tps[best],
                     "gated_depths": [r["gated"]["depth"] for r in rs],
                     "acceptance_rates": [[round(float(v), 4) for v in r["conf"][:, 0]] for r in rs],
                     "policy_us_per_call": float(np.mean([u for n, u in pol_us if n == nseq]))})
    sec2 = {"per_batch": sec2, "cost_model": {"C0_us": C0, "T_exp_us": T_exp, "r2": r2,
                                              "fit": "step_us = C0 + T_exp * union experts, all fixed-depth runs"}}
    return {"depth_vs_width": sec1, "confidence_gating": sec2,
            "workload": "draft chains of 6 positions on the workload's layer shapes, AR(1) logits along "
                        "each chain (consecutive positions co-activate), per-sequence acceptance "
                        "a ~ Beta(0.5, 0.5), confidence at depth j = a^j"}


def workload_entry(core, cfg, wl, extra=None):
    """The per-workload record of the bench line."""
    d = {"config": {"layers": cfg.L, "hidden": cfg.H, "experts": cfg.E, "top_k": cfg.k,
                    "intermediate": cfg.I, "weights": cfg.dtype, "batch": cfg.nseq, "verify_tokens": wl.T,
                    "gamma": wl.gamma.tolist(), "reuse_bias": cfg.use_bias,
                    "selection": "marginal" if cfg.mode == 0 else "static"}}
    for k in ("value", "ms_per_step", "latency_us", "tokens_per_s", "unique_expert_gb_per_step",
              "frac_of_peak_step", "frac_of_8tbs_step", "eager_ms_per_step", "control_path_ms",
              "control_path_frac", "control_path_eager_frac", "kernel_ms_per_step", "clocks", "e2e",
              "launches_per_step"):
        d[k] = core[k]
    d["unit"] = "GB/s"
    d["union_per_layer"] = sum(core["unique_experts_per_layer"]) / len(core["unique_experts_per_layer"])
    r = core["roofline"]
    d["roofline"] = {"gate_up_frac": r["frac"], "gate_up_gbs": r["achieved"],
                     "down_frac": r["ffn_down"]["frac"], "down_gbs": r["ffn_down"]["achieved"],
                     "ffn_pair_frac": r.get("ffn_pair_frac"),
                     "peak": r["peak"], "peak_kind": r["peak_kind"], "traffic": r["traffic"]}
    if extra:
        d.update(extra)
    return d


def other_workloads(mv, args, rank, ws, local, skip):
    """Every workload other than the headline one, each measured alone (its
    weights built, measured and freed before the next)."""
    import torch
    from workload import CONFIGS, gen
    out = {}
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    for name, cfg in CONFIGS.items():
        if name == skip:
            continue
        wl = gen.make_workload(cfg)
        layers, layout = build_layers(mv, cfg, dev)
        core, _ = measure_step(mv, cfg, wl, layers, layout, args, dev, stream, ws, local, name)
        extra = None
        if rank == 0 and cfg.nseq > 1:
            extra = {"gamma_sweep": gamma_sweep(mv, cfg, layers, layout, dev, stream),
                     "width_vs_depth": width_depth_measure(mv, cfg, layers, layout, dev, stream)}
        out[name] = workload_entry(core, cfg, wl, extra)
        del layers
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def ours(args, rank, ws, local):
    import torch

    import serving_router_softmax_gb300 as mv
    from workload import CONFIGS, gen

    cfg = CONFIGS[args.config]
    if args.layers:
        cfg = cfg.replace(L=min(args.layers, cfg.L))
    if args.experts:
        cfg = cfg.replace(E=args.experts, cap=min(cfg.cap, args.experts - cfg.k) if cfg.use_bias else cfg.cap)
    dev = torch.device("cuda", local)
    wl = gen.make_workload(cfg)
    layers, layout = build_layers(mv, cfg, dev)
    stream = torch.cuda.current_stream(dev)
    core, y_first = measure_step(mv, cfg, wl, layers, layout, args, dev, stream, ws, local, args.config)
    profiling = bool(args.layers or args.experts)

    # ---- verify-cost model check and S2-MoE expansion (rank 0 only).
    cost_model, expansion = (None, None)
    if rank == 0 and not profiling and not args.quick:
        cost_model, expansion = cost_model_and_expansion(mv, cfg, layers, layout, dev, stream)

    # ---- router logits, timed alone (the step routes the given node logits).
    router = router_measure(mv, cfg, wl, dev, stream)

    # ---- S2-MoE reuse-bias sweep (rank 0 only).
    bias_sweep = None
    if rank == 0 and not profiling and not args.quick:
        bias_sweep = reuse_bias_sweep(mv, cfg, layers, layout, dev, stream)

    # ---- draft-budget sweep on batched workloads (rank 0 only).
    gsweep = None
    if rank == 0 and cfg.nseq > 1 and not profiling:
        gsweep = gamma_sweep(mv, cfg, layers, layout, dev, stream)

    # ---- expert residency with on-demand staging from Grace memory (rank 0 only).
    residency = None
    if rank == 0 and not args.no_residency and (args.residency or (not profiling and not args.quick)):
        fracs = tuple(float(v) for v in args.residency_fracs.split(","))
        residency = residency_measure(mv, cfg, layers, layout, dev, stream, expansion, fracs=fracs)

    result = {
        "metric": "verify-step HBM GB/s on unique-expert bytes",
        "value": core["value"],
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": core["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded workload generator; counter-hash weights)",
        "config": {"workload": cfg.name + (f" (first {cfg.L} layers, profiling run)" if args.layers else "")
                   + (f" ({cfg.E} experts, profiling run)" if args.experts else ""),
                   "layers": cfg.L, "hidden": cfg.H, "experts": cfg.E,
                   "top_k": cfg.k, "intermediate": cfg.I, "weights": cfg.dtype,
                   "batch": cfg.nseq, "verify_tokens": wl.T, "gamma": wl.gamma.tolist(),
                   "reuse_bias": cfg.use_bias, "selection": "marginal" if cfg.mode == 0 else "static",
                   "weight_layout": layout,
                   "l2": "inputs larger than L2 (unique-expert bytes per step >> 129 MB)",
                   "parallelism": "replicas" if ws > 1 else "single-gpu"},
    }
    for k in ("latency_us", "tokens_per_s", "unique_experts_per_layer", "unique_expert_gb_per_step",
              "frac_of_peak_step", "frac_of_8tbs_step", "roofline", "kernel_ms_per_step", "launch",
              "eager_ms_per_step", "control_path_ms", "control_path_frac", "control_path_eager_ms",
              "control_path_eager_frac", "control_path_frac_events", "clocks", "e2e", "gpu_launches"):
        result[k] = core[k]
    result.update({"router_logits": router, "cost_model": cost_model, "s2_expand": expansion,
                   "residency": residency, "reuse_bias": bias_sweep, "gamma_sweep": gsweep})
    head_entry = workload_entry(core, cfg, wl, {"gamma_sweep": gsweep} if gsweep else None)
    del layers
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # ---- every other workload, measured the same way (the headline stays
    # the configuration named above).
    if args.workloads == "all" and not profiling:
        result["workloads"] = {cfg.name: head_entry}
        result["workloads"].update(other_workloads(mv, args, rank, ws, local, skip=cfg.name))
    return result, wl, cfg, y_first


# ---------------------------------------------------------------------- oracle
def oracle_prepare(cfg, wl, n_layers):
    """Routing of the sampled layers and host copies of their unique experts
    (input preparation, outside any timed region)."""
    from oracle import moe_layer as ml
    from oracle import verify_step as ovs
    from workload import gen

    sels, _ = ovs.run_selection(wl)
    rows = ovs.verify_rows(wl.parent.shape[0], sels)
    conf = ovs.token_conf(wl.P, sels)
    stored, unions = {}, []
    for l in range(n_layers):
        lg = wl.logits[l].reshape(-1, cfg.E)[rows]
        if cfg.use_bias:
            lg = ml.reuse_bias(lg, conf, cfg.k, cfg.cap, cfg.alpha)
        ids, _ = ml.route(lg, cfg.k)
        u = sorted(set(ids.ravel().tolist()))
        unions.append(len(u))
        for e in u:
            stored[(l, e)] = gen.expert_weights_host(cfg, l, e)
    return stored, sum(unions) * expert_bytes(cfg)


def oracle_run(cfg, wl, n_layers, stored):
    """One timed pass of the oracle verify step restricted to the sampled layers
    (selection, routing, union and FFN of every verify token; weight decoding
    included).  Returns seconds."""
    from oracle import moe_layer as ml
    from oracle import verify_step as ovs

    x_dec = (lambda a: np.asarray(a, np.float32).astype(np.float64)) if cfg.dtype == "f32" else ml.decode_bf16
    t0 = time.perf_counter()
    out = ovs.run_step(wl, lambda l: (lambda e: ml.expert_matrices(stored[(l, e)], cfg.dtype)),
                       layers=list(range(n_layers)), x_decode=x_dec)
    return time.perf_counter() - t0, out["layers"][0]["y"]


def oracle_baseline(cfg, wl, n_layers, target_s=12.0, max_reps=200):
    """Repeats the oracle sample for about target_s seconds; returns the time,
    the unique-expert bytes covered, the repetitions and the oracle's layer-0
    output of the last repetition."""
    stored, nbytes = oracle_prepare(cfg, wl, n_layers)
    times, y = [], None
    while sum(times) < target_s and len(times) < max_reps:
        dt, y = oracle_run(cfg, wl, n_layers, stored)
        times.append(dt)
    return sum(times), nbytes * len(times), len(times), y


def ffn_errors(y, ref, dtype):
    """FFN output error of the GPU step against the oracle on the same layer:
    row-wise normwise max_t |y_t - ref_t|_inf / |ref_t|_inf (the bound the
    parity tests hold), and element-wise max |y - ref| / max(|ref|, rms(ref))
    (each element's error relative to its own size, floored at the layer's
    rms so that near-zero outputs do not blow it up)."""
    den = np.max(np.abs(ref), axis=1)
    den = np.where(den == 0, 1.0, den)
    row = float(np.max(np.max(np.abs(y - ref), axis=1) / den))
    rms = float(np.sqrt(np.mean(ref * ref))) or 1.0
    elem = float(np.max(np.abs(y - ref) / np.maximum(np.abs(ref), rms)))
    return {"rowwise": row, "elementwise_rms_floor": elem, "bound": 1e-4 if dtype == "f32" else 2e-2}


def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max([i.get("num_threads", 1) for i in info] or [1])
    except Exception:
        return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def reference(args, rank, ws):
    """The reference arm: the CPU oracle as it stands, on the same workload."""
    from workload import CONFIGS, gen
    if rank != 0:
        return None
    cfg = CONFIGS[args.config]
    wl = gen.make_workload(cfg)
    n_layers = args.cpu_layers or 1
    stored, nbytes = oracle_prepare(cfg, wl, n_layers)
    times = []
    for i in range(args.warmup + args.steps):
        dt, _ = oracle_run(cfg, wl, n_layers, stored)
        if i >= args.warmup:
            times.append(dt)
    tot = sum(times)
    value = nbytes * len(times) / tot / 1e9
    cores = cpu_threads()
    sample = f"oracle verify step restricted to layer(s) 0..{n_layers - 1} of {cfg.L}, all {wl.T} verify tokens"
    return {
        "impl": "reference", "metric": "verify-step HBM GB/s on unique-expert bytes",
        "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot / len(times) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "layers_sampled": n_layers, "verify_tokens": wl.T},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        res = reference(args, rank, ws)
        if res is not None:
            print(json.dumps(res))
        return
    rank, ws, local = dist_setup(args.gpus)
    res, wl, cfg, y_first = ours(args, rank, ws, local)
    if rank == 0 and not args.no_cpu_baseline:
        n_layers = args.cpu_layers or 1
        dt, nbytes, reps, y_oracle = oracle_baseline(cfg, wl, n_layers)
        res["cpu_baseline"] = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cpu_threads(),
                               "kind": "oracle",
                               "sample": f"oracle verify step on layer(s) 0..{n_layers - 1} of {cfg.L}, all {wl.T} verify tokens, repeated {reps}x: {dt:.1f} s",
                               "parity_layer0": ffn_errors(y_first.numpy().astype(np.float64), y_oracle,
                                                           cfg.dtype)}
    if rank == 0:
        print(json.dumps(res))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

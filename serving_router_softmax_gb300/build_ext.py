"""Build the CUDA library in-tree with nvcc (sm_103a only).

``build()`` compiles every ``csrc/*.cu`` translation unit in parallel and
links ``libmoeverify.so`` next to this file; it also builds the input
generator's device fill (``workload/libmoegen.so``).  Objects go to
``_build/`` at the repository root.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoeverify.so")
GEN_SRC = os.path.join(ROOT, "workload", "fill.cu")
GEN_LIB = os.path.join(ROOT, "workload", "libmoegen.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; set NVCC or add CUDA to PATH")
    return cand


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def _newer(target, deps):
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    srcs = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs.append(os.path.join(ROOT, "include", "moe_verify.h"))
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    jobs = []
    for s, o in zip(srcs, objs):
        if force or not _newer(o, [s] + hdrs):
            jobs.append([nv, *ARCH, *FLAGS, "-I", os.path.join(ROOT, "include"), "-c", s, "-o", o])
    gen_job = None
    if force or not _newer(GEN_LIB, [GEN_SRC]):
        gen_job = [nv, *ARCH, *FLAGS, "-shared", GEN_SRC, "-o", GEN_LIB]
    all_jobs = jobs + ([gen_job] if gen_job else [])
    if all_jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(all_jobs), os.cpu_count() or 4)) as ex:
            outs = list(ex.map(_run, all_jobs))
        if verbose:
            for o in outs:
                if o.strip():
                    print(o)
    if force or jobs or not _newer(LIB, objs):
        _run([nv, *ARCH, "-shared", *objs, "-o", LIB, "-lcudart"])
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

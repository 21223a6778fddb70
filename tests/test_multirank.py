"""The multi-GPU path of bench.py on CPU: two gloo ranks run the same
aggregation code the NCCL ranks run (barrier, max time, summed bytes), and the
reference arm does its work on rank 0 only.  Replicas only: no data-path
collective exists to test."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        mx = bench.max_over_ranks(float(rank + 1), ws)
        sm = bench.sum_over_ranks(float(10 * (rank + 1)), ws)
        # rank r moved (r + 1) GB in (r + 1) * 100 ms: the job moved 3 GB in 200 ms
        gbs, ms = bench.job_throughput((rank + 1) * 1e9, (rank + 1) * 100.0, ws)
        out[rank] = (mx, sm, gbs, ms)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    for rank in (0, 1):
        mx, sm, gbs, ms = res[rank]
        assert mx == 2.0 and sm == 30.0
        assert ms == 200.0 and abs(gbs - 15.0) < 1e-12


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    gbs, ms = bench.job_throughput(2e9, 100.0, 1)
    assert ms == 100.0 and abs(gbs - 20.0) < 1e-12


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    a = argparse.Namespace(config="toy", steps=1, warmup=0, cpu_layers=1, gpus=2)
    assert bench.reference(a, 1, 2) is None  # a non-zero rank returns without work

"""bench.py's multi-rank path on CPU (gloo, world size 2): ranks are
independent replicas, the job's time is the slowest rank's and its
throughput counts every rank's work."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r reports (r + 1) * 10 ms: the job time is the slowest, 20 ms
    t = bench.max_over_ranks((rank + 1) * 10.0, world, "cpu")
    out[rank] = t
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_job_tflops_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_tflops(51.95e12, 1, 29.0)
    assert bench.job_tflops(51.95e12, 4, 29.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5

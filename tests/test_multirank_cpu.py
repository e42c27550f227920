"""The replica path of bench.py under torch.distributed, on CPU with gloo.

With N > 1 every rank runs its own replica of the layer; the job's time is
the slowest rank's and its throughput counts every rank's work.  Two gloo
ranks on 127.0.0.1 exercise the cross-rank reduction the bench uses.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports times (1 + r, 5 - r, 3): the job sees the maximum of each
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 3.0], dist, "cpu")
        dist.barrier()
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 5.0, 3.0]


def test_single_process_reduction_and_job_throughput():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1, 2.5]) == [1.0, 2.5]
    # 2 replicas of 1e12 FLOP in 1 ms: 2000 TFLOP/s for the job
    assert bench.job_tflops(2, 1e12, 1.0) == pytest.approx(2000.0)
    assert bench.job_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)

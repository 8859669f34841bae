"""The bench's N>1 path on CPU: two gloo ranks, replica timing reduced with
the max over ranks, whole-job value = ranks x per-rank work / slowest time."""

import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 100.0 + 10.0 * rank                 # rank 1 is the slow one
    got = bench.max_over_ranks(ms)
    val = bench.whole_job_tflops(1e12, world, got)
    q.put((rank, got, val))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, val in res:
        assert got == 110.0
        assert val == pytest.approx(2 * 1e12 / 0.110 / 1e12)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(2e12, 1, 1000.0) == pytest.approx(2.0)

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


def _split_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    hq0, hq1, hk0, hk1 = bench.head_partition(32, 8, world, rank)
    # every rank reports its ranges; per-rank work differs (per-head counts)
    ranges = [None] * world
    dist.all_gather_object(ranges, (hq0, hq1, hk0, hk1))
    flops = 1e12 * (1 + rank)                 # rank 1 carries twice the work
    job = bench.sum_over_ranks(flops)
    ms = bench.max_over_ranks(100.0 + 10.0 * rank)
    q.put((rank, ranges, job, ms))
    dist.destroy_process_group()


def test_kv_head_split_covers_every_head_once_and_sums_the_work():
    """--split kv-heads on two gloo ranks: the KV-head ranges tile [0, Hkv)
    and carry their query heads (h // G), and the whole-job value is the work
    of all ranks over the slowest rank's time."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 30500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_split_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ranges, job, ms in res:
        assert job == pytest.approx(3e12) and ms == 110.0
        kv = sorted(h for (_, _, a, b) in ranges for h in range(a, b))
        qh = sorted(h for (a, b, _, _) in ranges for h in range(a, b))
        assert kv == list(range(8)) and qh == list(range(32))
        for hq0, hq1, hk0, hk1 in ranges:
            assert all(hk0 <= h // 4 < hk1 for h in range(hq0, hq1))


def test_head_partition_rejects_uneven_splits():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.head_partition(24, 24, 8, 7) == (21, 24, 21, 24)
    with pytest.raises(ValueError):
        bench.head_partition(32, 8, 3, 0)

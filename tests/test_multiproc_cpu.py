"""bench.py's multi-rank path on the CPU: two gloo ranks.

On N GPUs the path runs N independent replicas, with no collective on the data path.  The
host side still has to take the max time over ranks and report whole-job
throughput.  These tests exercise that with world_size 2 over gloo.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.init_dist(world, "gloo")
    slowest = bench.max_over_ranks(dist, 1.5 + rank)     # rank 1 is the slowest
    bench.barrier(dist)
    job = bench.aggregate_throughput(100.0, world, slowest)
    q.put((rank, slowest, job))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[1] for g in got] == [2.5, 2.5]
    assert [g[2] for g in got] == [pytest.approx(80.0)] * 2   # 100 units x 2 ranks / 2.5 s


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.25) == 3.25
    assert bench.aggregate_throughput(10.0, 1, 2.0) == 5.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload = "tiny_w2"
        steps = 3
        warmup = 3
        gpus = 2
    assert bench.run_reference(Args()) == 0

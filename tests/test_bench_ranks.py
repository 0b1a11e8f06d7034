"""bench.py's multi-rank logic on CPU: two gloo ranks reduce their timings to
the slowest rank's, each rank runs its own replica seed, and the reported
rate counts every rank's work over that slowest time."""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, results):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r times [1 + r, 5 - r, 3] ms
        got = bench.max_over_ranks(dist, [1.0 + rank, 5.0 - rank, 3.0], "cpu")
        results[rank] = (got, bench.replica_seed(rank))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as manager:
        results = manager.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(results)
    assert res[0][0] == [2.0, 5.0, 3.0]
    assert res[1][0] == [2.0, 5.0, 3.0]
    assert res[0][1] == 2 and res[1][1] != res[0][1]


def test_single_process_is_the_identity():
    assert bench.max_over_ranks(None, [1.5, 2.5], "cpu") == [1.5, 2.5]


def test_whole_job_rate_counts_every_rank():
    # 100 units per rank, 2 ranks, slowest rank 10 ms -> 20,000 units/s
    assert bench.whole_job_rate(100.0, 2, 10.0) == pytest.approx(20000.0)
    assert bench.whole_job_rate(100.0, 1, 10.0) == pytest.approx(10000.0)

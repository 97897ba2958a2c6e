"""The N-rank bench path on CPU: world-size-2 gloo ranks on 127.0.0.1.

Requests are independent (results keyed by request id), so ranks shard the
batch with no data-path collective; only the step times meet, as a max over
ranks, and the job's throughput counts every rank's rows."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, times, q):
    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B = 5
        sh = bench.shard(rank, B, 1236)
        ids = list(range(sh["first_request"], sh["first_request"] + B))
        got = [None] * world
        dist.all_gather_object(got, {"ids": ids, "seed": sh["data_seed"]})
        mx = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        q.put((rank, got, mx, bench.job_value(B * 9, world, mx[0])))
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_requests_and_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [[1.5, 0.25], [2.0, 0.125]]  # per rank: step ms, kernel ms
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, mx, value in out:
        ids = [i for g in got for i in g["ids"]]
        assert sorted(ids) == list(range(10)) and len(set(ids)) == 10  # disjoint shards covering the job
        assert got[0]["seed"] != got[1]["seed"]  # each rank its own data
        assert mx == [2.0, 0.25]  # element-wise max over ranks
        assert value == pytest.approx(2 * 5 * 9 / 2.0e-3)  # every rank's rows over the slowest time


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3.0, 1.0], 1, torch.device("cpu")) == [3.0, 1.0]
    assert bench.job_value(90, 1, 1.0) == pytest.approx(90_000.0)
    assert bench.shard(0, 7, 10)["first_request"] == 0 and bench.shard(3, 7, 10)["first_request"] == 21

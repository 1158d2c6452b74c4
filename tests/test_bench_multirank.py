"""The benchmark's multi-rank aggregation (replicas only: no data exchange, the
job is as slow as its slowest rank) on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = [10.0 + 5.0 * rank, 20.0 - 3.0 * rank]       # rank 1 slower in the first
        got = bench.slowest_rank(times, world, torch.device("cpu"))
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    results = dict(q.get(timeout=10) for _ in range(world))
    assert results[0] == results[1] == [15.0, 20.0]


def test_single_rank_passthrough_and_job_throughput():
    assert bench.slowest_rank([1.5, 2.5], 1, None) == [1.5, 2.5]
    # 2 replicas, each 1 GB per 0.5 ms step -> 4000 GB/s for the job
    assert bench.whole_job_gbs(1e9, 2, 0.5) == pytest.approx(4000.0)

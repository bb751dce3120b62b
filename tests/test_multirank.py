"""Replicas-only multi-GPU logic of bench.py, exercised with two gloo ranks
on the CPU: the path shards by sequence with no data exchange, so the ranks
only agree on the slowest replica's time and rank 0 reports the job total."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [1.0 + rank, 5.0 - 2 * rank]          # rank 0: [1, 5], rank 1: [2, 3]
        got = bench.max_over_ranks(local, dist)
        q.put((rank, got, bench.job_throughput(world, 1_000_000_000, got[0])))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_reduction_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, gbs in res:
        assert got == [2.0, 5.0]
        # two replicas, 1 GB each, in the slowest replica's 2 ms: 1000 GB/s
        assert gbs == pytest.approx(1000.0)


def test_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 4.0], None) == [3.0, 4.0]
    assert bench.job_throughput(1, 2_000_000, 1.0) == pytest.approx(2.0)

"""The multi-GPU path of the benchmark is N independent replicas (decode
attention needs no exchange).  Its host logic -- barrier, slowest-rank time,
whole-job throughput, rank 0 alone reporting -- runs here on CPU with two gloo
ranks."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        my_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        mx = bench.max_over_ranks(my_ms, world)
        value = bench.job_throughput(1_000_000, 100, world, mx)
        dist.barrier()
        q.put((rank, mx, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, mx, value in got:
        assert mx == 15.0
        # 2 ranks x 100 steps x 1 MB over 15 ms
        assert value == pytest.approx(2 * 100 * 1e6 / 0.015 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(10**9, 10, 1, 1000.0) == pytest.approx(10.0)

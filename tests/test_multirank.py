"""The N > 1 bench path on CPU: two gloo ranks run the barrier and the
max-over-ranks timing reduction bench.py uses under torchrun (one independent
replica per GPU, no data-path collective)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms = 10.0 + 5.0 * rank           # rank 1 is the slower replica
        ms_max = bench.reduce_max(ms, world)
        value = bench.aggregate_gbs(1 << 30, 4, world, ms_max)
        q.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms_max, value in got:
        assert ms_max == 15.0
        # 2 replicas x 4 steps x 1 GiB in 15 ms
        assert abs(value - 2 * 4 * (1 << 30) / 0.015 / 1e9) < 1e-6


def test_single_rank_needs_no_process_group():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.aggregate_gbs(10**9, 2, 1, 1000.0) == 2.0

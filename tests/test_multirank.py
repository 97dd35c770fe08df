"""The N>1 path of bench.py on the CPU: two gloo ranks, each with its own batch
(weak scaling, no collective on the data path), combine their timings the way
the benchmark does: the slowest rank's time, and every rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, l = bench.dist_init()
    assert (w, r, l) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        total = bench.reduce_max(local_ms, dist, torch.device("cpu"))
        value = bench.weak_scaling_gbs(1e9, world, 4, total)
        dist.barrier()
        out.put((rank, total, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_rank_and_all_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r for r, _, _ in results] == [0, 1]
    for _, total, value in results:
        assert total == 15.0
        # 2 ranks x 4 steps x 1 GB in 15 ms
        assert value == pytest.approx(2 * 4 * 1e9 / 15e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.weak_scaling_gbs(2e9, 1, 10, 20.0) == pytest.approx(1000.0)

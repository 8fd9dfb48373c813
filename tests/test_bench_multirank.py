"""bench.py's multi-rank host path (replicas, weak scaling) on CPU: two
gloo ranks on 127.0.0.1 go through the same barrier, max-over-ranks and
aggregation helpers the GPU run uses under torchrun (no GPU, no data-path
collective)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        sec = bench.max_over_ranks(0.5 + rank, world)          # rank 1 is slower
        gbs = bench.aggregate_gbs(2e9, 10, world, sec)
        bench.barrier(world)
        q.put((rank, sec, gbs))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), q), nprocs=world, join=True,
                       start_method="spawn")
    got = sorted(q.get() for _ in range(world))
    # both ranks see rank 1's 1.5 s; the job streamed 2 ranks x 10 steps x 2 GB
    assert [g[1] for g in got] == [1.5, 1.5]
    assert got[0][2] == pytest.approx(2e9 * 10 * 2 / 1.5 / 1e9)
    assert got[0][2] == got[1][2]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.aggregate_gbs(1e9, 4, 1, 2.0) == pytest.approx(2.0)

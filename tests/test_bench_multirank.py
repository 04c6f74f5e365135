"""The benchmark's multi-rank host logic on CPU: two gloo ranks, barrier and
max-over-ranks time, rank-0-only output, as torchrun runs it across GPUs."""
from __future__ import annotations

import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, ws, lr = bench.dist_env()
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)
    got = bench.reduce_max(10.0 + 5.0 * rank, ws)
    # rank 1's node is short of host memory, rank 0's is not: both skip
    short = bench.host_memory_short(1 << 30, 2, ws, available=(1 << 40) if rank == 0 else (1 << 20))
    bench.barrier(ws)
    q.put((r, ws, lr, got, short))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=5) for _ in range(world))
    assert [r[0] for r in results] == [0, 1]
    assert all(r[1] == world and r[3] == 15.0 for r in results)
    assert all(r[4] for r in results)           # the host-memory check is collective


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert not bench.host_memory_short(1 << 30, 1, 1, available=1 << 40)
    assert bench.host_memory_short(1 << 30, 8, 1, available=8 << 30)

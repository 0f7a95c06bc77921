"""Multi-rank host logic of bench.py on CPU with two gloo ranks.

Each rank runs an independent replica (its own sequences, seeded by rank); the only
cross-rank operations are the barrier and the max / sum of timings and byte counts.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    ws, r = bench.init_dist("gloo")
    try:
        bench.barrier()
        mx = bench.reduce_over_ranks(10.0 + rank, "max")
        sm = bench.reduce_over_ranks(1.5 * (rank + 1), "sum")
        wl, _, _ = bench.build_workload("gpt", 3, 5, seed_offset=rank)
        q.put((rank, ws, r, mx, sm, wl.context_lens.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_shard():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, r, mx, sm, lens in res:
        assert ws == world and r == rank
        assert mx == 11.0 and sm == 4.5
    assert res[0][5] != res[1][5]          # each rank decodes its own sequences


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.5, "max") == 3.5
    assert bench.reduce_over_ranks(2.0, "sum") == 2.0

"""The N > 1 timing path of bench.py on CPU: two gloo ranks, the barrier and
the max-over-ranks reduction of the per-rank elapsed time (the bench reports
the slowest rank's time, replicas only)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (world, rank, rank)
        bench.barrier(world)
        per_rank = [3.5, 7.25][rank]
        out[rank] = bench.max_over_ranks(per_rank, world)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(out) == {0: 7.25, 1: 7.25}


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(1.5, 1) == 1.5


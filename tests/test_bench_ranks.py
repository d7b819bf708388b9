"""Host-side logic of the multi-rank bench: replicas only, no data-path
collective; the slowest rank's time and the sum of all ranks' work are what
the headline divides.  Run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        r, w, lr = bench.dist_env()
        t_max = bench.reduce_over_ranks(10.0 + rank, "max")      # per-rank time (ms)
        work = bench.reduce_over_ranks(1.5e12, "sum")             # per-rank FLOPs
        bench.barrier()
        q.put((rank, r, w, lr, t_max, work))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, r, w, lr, t_max, work in got:
        assert (r, w, lr) == (rank, world, rank)
        assert t_max == 11.0                     # the slowest rank
        assert work == 3.0e12                    # all ranks' work


def test_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_over_ranks(3.0, "max") == 3.0
    assert bench.reduce_over_ranks(3.0, "sum") == 3.0

"""The N>1 path of bench.py (independent replicas, no data-path collective) on CPU:
two gloo ranks, max-over-ranks timing and weak-scaling throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        mine = [10.0 + rank, 2.0 * (rank + 1), 7.0]
        got = bench.max_over_ranks(mine)
        thr = bench.replica_throughput(1, got[1] / 1e3 / 40, ws)
        q.put((rank, ws, r, local, got, thr))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, r, local, got, thr in out:
        assert ws == 2 and r == rank and local == rank
        assert got == [11.0, 4.0, 7.0]              # every rank sees the slowest rank's time
        assert thr == pytest.approx(2 * 40 / 4e-3)   # units of both ranks / slowest time


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.replica_throughput(4, 2.0, 1) == 2.0

"""Multi-rank host logic of the benchmark on CPU (gloo, world_size 2): every rank runs its own
replica, the slowest rank's time bounds the run, and throughput aggregates the units of all
ranks (weak scaling, no data-path collective)."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    seconds = 1.0 + rank                       # rank 1 is the slow one
    max_s = bench.reduce_max(seconds, w)
    value = bench.aggregate_throughput(100.0, w, max_s)
    dist.barrier()
    q.put((r, w, lr, max_s, value))
    dist.destroy_process_group()


def test_two_ranks_take_the_max_time_and_sum_units():
    pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r, w, lr, max_s, value) in enumerate(res):
        assert (r, w, lr) == (rank, 2, rank)
        assert max_s == 2.0                       # max over ranks
        assert value == pytest.approx(100.0 * 2 / 2.0)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.aggregate_throughput(257 * 10, 1, 2.0) == pytest.approx(1285.0)

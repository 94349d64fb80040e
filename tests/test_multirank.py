"""Host logic of the N>1 bench path on CPU with gloo, world size 2: the timed
region's max over ranks and the whole-job throughput."""
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
    r, w, l = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    t = bench.max_over_ranks(1.0 + rank, w)   # rank 1 is the slowest
    v = bench.aggregate(4096, 10, w, t)
    q.put((r, l, t, v))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, local, t, v in res:
        assert t == 2.0                       # max over ranks
        assert v == 4096 * 10 * 2 / 2.0       # all ranks' tokens / slowest time


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate(100, 4, 1, 2.0) == 200.0

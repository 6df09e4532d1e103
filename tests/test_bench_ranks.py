"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank gets its own
sampler seed and all ranks agree on the slowest rank's time. No GPU involved."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        slowest = bench.reduce_max(10.0 + 5.0 * rank, dist, "cpu")
        out[rank] = (slowest, bench.rank_seed(42, rank))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time_and_use_distinct_seeds():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] != res[1][1]


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5, None, "cpu") == 3.5

"""Host side of the vocabulary-shard step on CPU: the token ranges of the ranks, and the
exchange of shard records over torch.distributed (gloo, world size 2): every rank ends up with
all records stacked in rank (= token) order. No GPU involved: the records here are CPU
tensors with rank-specific contents."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from canvas_sampler_gb300.shards import gather_partials, shard_range
from canvas_sampler_gb300.sampler import ShardPartial


def test_shard_ranges_tile_the_vocabulary():
    for V, world in ((262144, 2), (262144, 8), (4096 * 3, 3), (2560, 4)):
        got = [shard_range(V, world, r) for r in range(world)]
        assert got[0][0] == 0 and got[-1][1] == V
        for (a0, b0), (a1, b1) in zip(got, got[1:]):
            assert b0 == a1 and a0 < b0
        assert all(a % 256 == 0 for a, _ in got)
    with pytest.raises(ValueError):
        shard_range(1000, 2, 0)
    with pytest.raises(ValueError):
        shard_range(512, 4, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, top_k, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        R, d = 6, 8
        p = ShardPartial.empty(1, 2, 3, d, top_k, device="cpu")
        p.rows.fill_(10.0 * rank)
        p.best.fill_(20.0 * rank + 1)
        p.O.copy_(torch.arange(R * d, dtype=torch.float32).view(1, R, d) + 1000.0 * rank)
        if top_k:
            p.cand.fill_(30.0 * rank + 2)
        g = gather_partials(p)
        res = {"rows": g.rows[:, 0, 0].tolist(), "best": g.best[:, 0, 0].tolist(),
               "O": g.O[:, 1, 2].tolist(), "shape": list(g.O.shape),
               "cand": None if g.cand is None else g.cand[:, 0, 0, 0].tolist()}
        out[rank] = res
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("top_k", [0, 4])
def test_two_ranks_gather_records_in_rank_order(top_k):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, top_k, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(2):
        assert res[r]["rows"] == [0.0, 10.0]
        assert res[r]["best"] == [1.0, 21.0]
        assert res[r]["O"] == [10.0, 1010.0]
        assert res[r]["shape"] == [2, 6, 8]
        assert res[r]["cand"] == (None if not top_k else [2.0, 32.0])

"""The step over a vocabulary split into shards (ds_sampler_step_shard on each token range,
ds_merge_shards over the gathered records) against the unsharded step and the oracle: s within
2e-5, the entropy within its tolerance, and sampled tokens, argmax and the state update
identical wherever the oracle's top-two perturbed logits are >= 1e-4 apart. Shards run one
after another in one process, or in two processes on the one GPU exchanging their records over
gloo (each process runs its own kernels; nothing on the GPU waits on the other process)."""
import os
import socket
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from canvas_sampler_gb300 import workloads as W
from canvas_sampler_gb300.sampler import CanvasState, Sampler, ShardPartial
from canvas_sampler_gb300.shards import gather_partials, shard_range

from _helpers import GpuCase, check_lock_update, compare_outputs, exact_f64, out_np, oracle_step, state_np

pytestmark = pytest.mark.gpu

REL_TOL = 2e-5


def _shard_step(case, state, n, seed=None):
    """Every shard's record in turn, then the merge with the first shard's sampler."""
    w = case.w
    seed = case.inp["seed"] if seed is None else seed
    samplers, parts = [], []
    for q in range(n):
        a, b = shard_range(w.V, n, q)
        sq = Sampler(b - a, w.d, canvas_len=w.L, max_batch=w.B, dtype=w.dtype, top_k=w.top_k,
                     max_steps=w.max_steps, impl="tensor")
        samplers.append(sq)
        parts.append(sq.step_shard(case.H, case.E[a:b], case.T, case.tau, state, seed, a, w.V))
    out = samplers[0].merge_shards(ShardPartial.stack(parts), case.T, case.tau, state, seed, w.V)
    torch.cuda.synchronize()
    for sq in samplers:
        assert sq.device_status() == 0
    return out


def _compare_with_full(g_sh, g_full, ref, rows):
    n_excl = 0
    for b, i in rows:
        err = np.linalg.norm(g_sh["s"][b, i] - g_full["s"][b, i]) / np.linalg.norm(g_full["s"][b, i])
        assert err <= REL_TOL, (b, i, err)
        if ref["gumbel_margin"][b, i] < 1e-4 or ref["topk_risk"][b, i]:
            n_excl += 1
            continue
        assert g_sh["sampled"][b, i] == g_full["sampled"][b, i], (b, i)
        assert abs(g_sh["conf"][b, i] - g_full["conf"][b, i]) <= REL_TOL * g_full["conf"][b, i]
    return n_excl


@pytest.mark.parametrize("top_k", [0, 8])
@pytest.mark.parametrize("n", [2, 4])
def test_shards_merge_to_the_full_step(n, top_k):
    w = replace(W.scaled(W.WORKLOADS["step_bf16_b8_v262144_d2816"], V=16384, d=256, B=2),
                top_k=top_k)
    case = GpuCase(w, impl="tensor")
    st_full, st_sh = case.state(), case.state()
    pre = state_np(st_full)
    g_full = out_np(case.run_step(st_full))
    g_sh = out_np(_shard_step(case, st_sh, n))
    ref = oracle_step(case, pre)
    rows = [(b, i) for b in range(w.B) for i in range(w.L)]
    rep = compare_outputs(g_sh, ref, rows, top_k=top_k)
    assert rep["excluded"] <= max(2, len(rows) // 50), rep
    check_lock_update(pre, g_sh, state_np(st_sh), ref, case.inp["tau"], case.inp["seed"], w.V,
                      w.max_steps)
    n_excl = _compare_with_full(g_sh, g_full, ref, rows)
    assert np.array_equal(g_sh["argmax"], g_full["argmax"])
    if n_excl == 0:
        for k, v in state_np(st_sh).items():
            assert np.array_equal(v, state_np(st_full)[k]), k


def test_shards_leave_finished_sequences_untouched():
    w = W.scaled(W.WORKLOADS["step_bf16_b8_v262144_d2816"], V=8192, d=256, B=2)
    inp = W.make_inputs(w)
    inp["done"][1] = 1
    case = GpuCase(w, inputs=inp, impl="tensor")
    st = case.state()
    pre = state_np(st)
    out = _shard_step(case, st, 2)
    post = state_np(st)
    for k in ("canvas", "lock", "step", "done"):
        assert np.array_equal(post[k][1], pre[k][1])
    assert torch.all(out.sampled[1] == 0) and torch.all(out.s[1] == 0)  # outputs untouched
    ref = oracle_step(case, pre)
    compare_outputs(out_np(out), ref, [(0, i) for i in range(w.L)])


def test_full_size_two_shards():
    w = W.WORKLOADS["step_bf16_b1_v262144_d2816"]
    case = GpuCase(w, impl="tensor")
    st_full, st_sh = case.state(), case.state()
    pre = state_np(st_full)
    g_full = out_np(case.run_step(st_full))
    g_sh = out_np(_shard_step(case, st_sh, 2))
    rows = [(0, i) for i in range(w.L)]
    for b, i in rows:
        err = np.linalg.norm(g_sh["s"][b, i] - g_full["s"][b, i]) / np.linalg.norm(g_full["s"][b, i])
        assert err <= REL_TOL, (i, err)
        assert abs(g_sh["entropy"][b, i] - g_full["entropy"][b, i]) <= REL_TOL * max(1.0, abs(g_full["entropy"][b, i]))
    assert np.array_equal(g_sh["argmax"], g_full["argmax"])
    differ = int(np.sum(g_sh["sampled"] != g_full["sampled"]))
    # the oracle at 16 positions, including any whose sample differs from the unsharded step's
    pos = sorted(set(np.linspace(0, w.L - 1, 16).astype(int).tolist()) |
                 set(np.nonzero(g_sh["sampled"][0] != g_full["sampled"][0])[0].tolist()))
    ref = oracle_step(case, pre, positions=np.array(pos))
    rep = compare_outputs(g_sh, ref, [(0, i) for i in pos])
    print(f"full-size two shards: {differ} samples differ from the unsharded step; oracle at "
          f"{rep['checked']} positions, {rep['excluded']} excluded")
    assert differ <= 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        w = W.WORKLOADS["loop8_bf16_b1_v32768_d1024"]
        case = GpuCase(w, impl="tensor")
        a, b = shard_range(w.V, world, rank)
        sq = Sampler(b - a, w.d, canvas_len=w.L, max_batch=w.B, dtype=w.dtype,
                     max_steps=w.max_steps, impl="tensor")
        st = case.state()
        part = sq.step_shard(case.H, case.E[a:b], case.T, case.tau, st, case.inp["seed"], a, w.V)
        torch.cuda.synchronize()
        # exchange over gloo through host memory, records in rank (= token) order
        host = ShardPartial(part.rows.cpu(), part.best.cpu(), part.O.cpu(), None)
        g = gather_partials(host)
        parts = ShardPartial(g.rows.cuda(), g.best.cuda(), g.O.cuda(), None)
        out = sq.merge_shards(parts, case.T, case.tau, st, case.inp["seed"], w.V)
        torch.cuda.synchronize()
        q.put((rank, out_np(out), state_np(st)))
    finally:
        dist.destroy_process_group()


def test_two_processes_exchange_records_over_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r, g, post = q.get(timeout=600)
        res[r] = (g, post)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # both ranks merged the same records into the same result
    for k in res[0][0]:
        assert np.array_equal(res[0][0][k], res[1][0][k]), k
    w = W.WORKLOADS["loop8_bf16_b1_v32768_d1024"]
    case = GpuCase(w, impl="tensor")
    pre = state_np(case.state())
    ref = oracle_step(case, pre)
    rows = [(0, i) for i in range(w.L)]
    rep = compare_outputs(res[0][0], ref, rows)
    assert rep["excluded"] <= 4
    check_lock_update(pre, res[0][0], res[0][1], ref, case.inp["tau"], case.inp["seed"], w.V,
                      w.max_steps)


def test_shards_with_the_entropy_budget_rule_and_schedule():
    # the pages' own sampler (entropy-budget acceptance, stop rule, temperature schedule) over
    # two shards: the same step as the unsharded sampler, state included, over three steps
    w = W.scaled(W.WORKLOADS["loop8_bf16_b1_v32768_d1024"], V=8192, d=256, B=2)
    inp = W.make_inputs(w)
    kw = dict(canvas_len=w.L, max_batch=w.B, dtype="bf16", max_steps=12, impl="tensor",
              lock_rule="entropy_budget", entropy_budget=0.1, stop_entropy=0.005,
              t_schedule=(0.8, 0.4))
    full = Sampler(w.V, w.d, **kw)
    shards = [Sampler(b - a, w.d, **kw) for a, b in (shard_range(w.V, 2, q) for q in range(2))]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    E, H = dev(inp["E"]), dev(inp["H"])
    T, tau = torch.from_numpy(inp["T"]).cuda(), torch.from_numpy(inp["tau"]).cuda()
    st_full = CanvasState.from_numpy(inp["canvas"], inp["lock"], inp["step"], inp["done"])
    st_sh = st_full.clone()
    for t in range(3):
        o_full = full.step(H, E, T, tau, st_full, inp["seed"])
        parts = []
        for q, sq in enumerate(shards):
            a, b = shard_range(w.V, 2, q)
            parts.append(sq.step_shard(H, E[a:b], T, tau, st_sh, inp["seed"], a, w.V))
        o_sh = shards[0].merge_shards(ShardPartial.stack(parts), T, tau, st_sh, inp["seed"], w.V)
        torch.cuda.synchronize()
        gf, gs = out_np(o_full), out_np(o_sh)
        rel = np.linalg.norm(gs["s"] - gf["s"], axis=-1) / np.linalg.norm(gf["s"], axis=-1)
        assert rel.max() <= REL_TOL
        assert np.all(np.abs(gs["entropy"] - gf["entropy"]) <= REL_TOL * np.maximum(1.0, gf["entropy"]))
        assert np.array_equal(gs["argmax"], gf["argmax"])
        same = (gs["sampled"] == gf["sampled"]).mean()
        assert same >= 0.99, same
        if np.array_equal(gs["sampled"], gf["sampled"]):
            for k in ("canvas", "lock", "step", "done", "prev_argmax"):
                assert torch.equal(getattr(st_sh, k), getattr(st_full, k)), (t, k)
        else:  # a near-tie sampled differently: continue both from the same state
            for k in ("canvas", "lock", "step", "done", "prev_argmax"):
                getattr(st_sh, k).copy_(getattr(st_full, k))

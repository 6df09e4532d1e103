"""GPU block-autoregressive driver (ds_block_loop): one graph runs every block's steps and
commits each finished canvas; against plain launches, against one-block runs, against the
oracle's draws for a block index, and the block index leaving no trace on later steps."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from canvas_sampler_gb300 import workloads as W
from canvas_sampler_gb300.sampler import StepOutputs

from _helpers import GpuCase, check_lock_update, compare_outputs, out_np, state_np

pytestmark = pytest.mark.gpu

FIXED = replace(W.scaled(W.WORKLOADS["loop8_bf16_b1_v32768_d1024"], V=8192, d=256, B=2),
                max_steps=8, tau=(0.9, 0.9))
STANDIN = replace(W.scaled(W.WORKLOADS["loop48_topk64_bf16_b4_v262144_d2816"], V=8192, d=256,
                           B=2), max_steps=10)


def _init(w, n_blocks, seed=3):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.integers(0, w.V, (n_blocks, w.B, w.L)).astype(np.int32)).cuda()


def _run(case, init, use_graph=True, first_block=0):
    w = case.w
    n = init.shape[0]
    state, out = case.state(), StepOutputs.empty(w.B, w.L, w.d)
    tokens = torch.full((n, w.B, w.L), -1, dtype=torch.int32, device="cuda")
    steps = torch.full((n, w.B), -1, dtype=torch.int32, device="cuda")
    kw = dict(first_block=first_block, use_graph=use_graph)
    if w.h_mode == "standin":
        Wt = torch.from_numpy(case.inp["W"].view(np.int16)).view(torch.bfloat16).cuda()
        Hb = torch.zeros(w.B, w.L, w.d, dtype=torch.bfloat16, device="cuda")
        case.sampler.block_loop(case.E, case.T, case.tau, state, case.inp["seed"], out, init,
                                tokens, steps, W=Wt, H_buf=Hb, **kw)
    else:
        case.sampler.block_loop(case.E, case.T, case.tau, state, case.inp["seed"], out, init,
                                tokens, steps, H=case.H, **kw)
    torch.cuda.synchronize()
    assert case.sampler.device_status() == 0
    return tokens, steps, state, out


@pytest.mark.parametrize("w", [FIXED, STANDIN], ids=["fixed_h", "standin_topk"])
def test_block_graph_equals_plain_launches(w):
    inp = W.make_inputs(w)
    init = _init(w, 3)
    a, b = GpuCase(w, inputs=inp), GpuCase(w, inputs=inp)
    ta, sa, _, oa = _run(a, init, use_graph=True)
    tb, sb, _, ob = _run(b, init, use_graph=False)
    assert torch.equal(ta, tb) and torch.equal(sa, sb)
    assert torch.equal(oa.s, ob.s) and torch.equal(oa.sampled, ob.sampled)
    assert int(sa.min()) >= 1 and int(sa.max()) <= w.max_steps
    assert int(ta.min()) >= 0 and int(ta.max()) < w.V


def test_blocks_equal_one_block_runs_and_differ_in_their_draws():
    w = FIXED
    inp = W.make_inputs(w)
    init = _init(w, 3)
    init[2] = init[1]  # the same noise in blocks 1 and 2: only the draws differ
    case = GpuCase(w, inputs=inp)
    tokens, steps, _, _ = _run(case, init)
    for k in range(3):
        tk, sk, _, _ = _run(case, init[k:k + 1].clone(), first_block=k)
        assert torch.equal(tk[0], tokens[k]) and torch.equal(sk[0], steps[k]), k
    assert not torch.equal(tokens[1], tokens[2])


def test_block_index_reaches_the_draws():
    # one step of block 5 from its initial canvas, against the oracle's step with block = 5
    w = replace(FIXED, max_steps=8)
    inp = W.make_inputs(w)
    case = GpuCase(w, inputs=inp)
    init = _init(w, 1, seed=9)
    state, out = case.state(), StepOutputs.empty(w.B, w.L, w.d)
    tokens = torch.zeros((1, w.B, w.L), dtype=torch.int32, device="cuda")
    steps = torch.zeros((1, w.B), dtype=torch.int32, device="cuda")
    case.sampler.block_loop(case.E, case.T, case.tau, state, inp["seed"], out, init, tokens,
                            steps, H=case.H, first_block=5, max_iters=1, use_graph=True)
    torch.cuda.synchronize()
    g, post = out_np(out), state_np(state)
    pre = {"canvas": init[0].cpu().numpy(), "lock": np.zeros((w.B, w.L), np.uint8),
           "step": np.zeros(w.B, np.int32), "done": np.zeros(w.B, np.uint8)}
    ref = oracle.sampler_step(oracle.bf16_bits_to_f64(inp["H"]), case.E64, inp["T"], inp["tau"],
                              pre["canvas"], pre["lock"], pre["step"], pre["done"], inp["seed"],
                              max_steps=w.max_steps, block=5)
    rep = compare_outputs(g, ref, [(b, i) for b in range(w.B) for i in range(w.L)])
    assert rep["checked"] > 0
    check_lock_update(pre, g, post, ref, inp["tau"], inp["seed"], w.V, w.max_steps, block=5)
    # and it is not block 0's draw
    ref0 = oracle.sampler_step(oracle.bf16_bits_to_f64(inp["H"]), case.E64, inp["T"], inp["tau"],
                               pre["canvas"], pre["lock"], pre["step"], pre["done"], inp["seed"],
                               max_steps=w.max_steps)
    assert not np.array_equal(ref0["sampled"], ref["sampled"])


def test_steps_after_a_block_run_draw_as_block_zero():
    w = FIXED
    inp = W.make_inputs(w)
    a, b = GpuCase(w, inputs=inp), GpuCase(w, inputs=inp)
    _run(a, _init(w, 2))
    ga = out_np(a.run_step(a.state()))
    gb = out_np(b.run_step(b.state()))
    for k in ("sampled", "conf", "s"):
        assert np.array_equal(ga[k], gb[k]), k

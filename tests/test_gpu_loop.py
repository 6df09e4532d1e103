"""GPU denoising loop: the CUDA-graph loop (device-side while condition) against plain
launches, resume, and teacher-forced parity of every step with the oracle."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from canvas_sampler_gb300 import workloads as W
from canvas_sampler_gb300.sampler import StepOutputs

from _helpers import GpuCase, check_lock_update, compare_outputs, out_np, oracle_step, standin_close, state_np

pytestmark = pytest.mark.gpu

FIXED = replace(W.scaled(W.WORKLOADS["loop8_bf16_b1_v32768_d1024"], V=8192, d=256, B=2),
                max_steps=8, tau=(0.9, 0.9))
STANDIN = replace(W.scaled(W.WORKLOADS["loop48_topk64_bf16_b4_v262144_d2816"], V=8192, d=256,
                           B=2), max_steps=12)


def _loop(case, use_graph, max_iters=None, state=None, out=None, H_buf=None):
    w = case.w
    state = case.state() if state is None else state
    out = StepOutputs.empty(w.B, w.L, w.d) if out is None else out
    if w.h_mode == "standin":
        Wt = torch.from_numpy(case.inp["W"].view(np.int16)).view(torch.bfloat16).cuda()
        H_buf = torch.zeros(w.B, w.L, w.d, dtype=torch.bfloat16, device="cuda") if H_buf is None else H_buf
        case.sampler.loop(case.E, case.T, case.tau, state, case.inp["seed"], out, W=Wt, H_buf=H_buf,
                          max_iters=max_iters, use_graph=use_graph)
    else:
        case.sampler.loop(case.E, case.T, case.tau, state, case.inp["seed"], out, H=case.H,
                          max_iters=max_iters, use_graph=use_graph)
    torch.cuda.synchronize()
    return state, out


@pytest.mark.parametrize("w", [FIXED, STANDIN], ids=["fixed_h", "standin_topk"])
def test_graph_loop_equals_plain_launches(w):
    inp = W.make_inputs(w)
    a, b = GpuCase(w, inputs=inp), GpuCase(w, inputs=inp)
    sa, oa = _loop(a, use_graph=True)
    sb, ob = _loop(b, use_graph=False)
    for k in ("canvas", "lock", "step", "done"):
        assert torch.equal(getattr(sa, k), getattr(sb, k)), k
    for k in ("s", "sampled", "conf"):
        assert torch.equal(getattr(oa, k), getattr(ob, k)), k
    assert sa.done.all() and int(sa.step.max()) <= w.max_steps
    # every sequence stops on its own: its step count is where it finished
    assert a.sampler.device_status() == 0


def test_graph_loop_resumes():
    inp = W.make_inputs(FIXED)
    a, b = GpuCase(FIXED, inputs=inp), GpuCase(FIXED, inputs=inp)
    sa, oa = _loop(a, use_graph=True)
    sb, ob = _loop(b, use_graph=True, max_iters=3)
    assert int(sb.step.max()) <= 3
    sb, ob = _loop(b, use_graph=True, state=sb, out=ob)
    for k in ("canvas", "lock", "step", "done"):
        assert torch.equal(getattr(sa, k), getattr(sb, k)), k


def test_graph_is_reused_and_relaunchable():
    inp = W.make_inputs(FIXED)
    a = GpuCase(FIXED, inputs=inp)
    s1, o1 = _loop(a, use_graph=True)
    ref = {k: getattr(s1, k).clone() for k in ("canvas", "lock", "step", "done")}
    # same buffers, state reset in place: the cached graph runs again and gives the same bits
    fresh = a.state()
    for k in ref:
        getattr(s1, k).copy_(getattr(fresh, k))
    o1.s.zero_()
    _loop(a, use_graph=True, state=s1, out=o1)
    assert len(a.sampler._keep) > 0
    for k in ref:
        assert torch.equal(getattr(s1, k), ref[k]), k


def test_fixed_h_loop_teacher_forced():
    case = GpuCase(FIXED)
    state = case.state()
    n_excl = 0
    for it in range(FIXED.max_steps):
        pre = state_np(state)
        if pre["done"].all():
            break
        out = case.run_step(state)
        g, post = out_np(out), state_np(state)
        ref = oracle_step(case, pre)
        rows = [(b, i) for b in range(FIXED.B) if not pre["done"][b] for i in range(FIXED.L)]
        n_excl += compare_outputs(g, ref, rows)["excluded"]
        check_lock_update(pre, g, post, ref, case.inp["tau"], case.inp["seed"], FIXED.V,
                          FIXED.max_steps)
    assert state.done.all().item()
    assert n_excl <= 8


def test_standin_loop_teacher_forced():
    w = STANDIN
    case = GpuCase(w)
    state = case.state()
    Wt = torch.from_numpy(case.inp["W"].view(np.int16)).view(torch.bfloat16).cuda()
    s_prev = torch.zeros(w.B, w.L, w.d, dtype=torch.float32, device="cuda")
    Hbuf = torch.zeros(w.B, w.L, w.d, dtype=torch.bfloat16, device="cuda")
    checked = excluded = 0
    for it in range(w.max_steps):
        pre = state_np(state)
        if pre["done"].all():
            break
        case.sampler.standin_hidden(Wt, s_prev, case.E, state.canvas, state.done, Hbuf)
        torch.cuda.synchronize()
        H_bits = Hbuf.view(torch.int16).cpu().numpy().view(np.uint16)
        active = pre["done"] == 0
        frac = standin_close(H_bits[active], case.inp["W"],
                             s_prev.cpu().numpy().astype(np.float64)[active], case.E64,
                             pre["canvas"][active])
        assert frac < 1e-2
        out = StepOutputs.empty(w.B, w.L, w.d)
        out.s.copy_(s_prev)
        case.sampler.step(Hbuf, case.E, case.T, case.tau, state, case.inp["seed"], out=out)
        torch.cuda.synchronize()
        g, post = out_np(out), state_np(state)
        ref = oracle_step(case, pre, H64=oracle.bf16_bits_to_f64(H_bits))
        rows = [(b, i) for b in range(w.B) if active[b] for i in range(w.L)]
        rep = compare_outputs(g, ref, rows, top_k=w.top_k)
        checked += rep["checked"]
        excluded += rep["excluded"]
        check_lock_update(pre, g, post, ref, case.inp["tau"], case.inp["seed"], w.V, w.max_steps)
        s_prev = out.s.clone()
    assert state.done.all().item()
    # near-uniform stand-in softmaxes put ~1.5% of positions at a top-64 boundary the oracle
    # calls ambiguous (a token within 1e-4 of the 64th logit could win); 3% bounds it
    print(f"standin loop: {checked} positions checked, {excluded} excluded")
    assert excluded <= max(2, int(0.03 * checked)), (excluded, checked)

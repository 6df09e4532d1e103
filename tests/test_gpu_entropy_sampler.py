"""GPU parity of the pages' default sampler (entropy-budget acceptance, stop on a confident and
stable canvas, linear temperature schedule 0.8 -> 0.4; sokufu.com "A diffusion language model
refines 256 tokens in 12 steps" and Table 2) against the fp64 oracle."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from canvas_sampler_gb300 import workloads as W
from canvas_sampler_gb300.sampler import CanvasState, Sampler, StepOutputs

from _helpers import compare_outputs, exact_f64, out_np, to_torch_input

pytestmark = pytest.mark.gpu

BUDGET, STOP, SCHED = 0.1, 0.005, (0.8, 0.4)


def _setup(B=2, V=8192, d=256, max_steps=12, impl="auto"):
    w = replace(W.scaled(W.WORKLOADS["loop8_bf16_b1_v32768_d1024"], V=V, d=d, B=B),
                max_steps=max_steps)
    inp = W.make_inputs(w)
    sampler = Sampler(w.V, w.d, canvas_len=w.L, max_batch=w.B, dtype="bf16",
                      max_steps=w.max_steps, impl=impl, lock_rule="entropy_budget",
                      entropy_budget=BUDGET, stop_entropy=STOP, t_schedule=SCHED)
    dev = dict(E=to_torch_input(inp["E"], "bf16"), H=to_torch_input(inp["H"], "bf16"),
               T=torch.from_numpy(inp["T"]).cuda(), tau=torch.from_numpy(inp["tau"]).cuda())
    return w, inp, sampler, dev


def _state_np(st):
    return {k: getattr(st, k).cpu().numpy() for k in ("canvas", "lock", "step", "done",
                                                      "prev_argmax")}


def _rule_on_gpu_outputs(w, inp, pre, g, post):
    """The rule applied to the GPU's own fp32 entropies / samples / argmax must reproduce the
    GPU's update; a difference is allowed only when fp32 and fp64 running sums (or the mean)
    can fall on different sides of the budget (or the stop threshold)."""
    n_amb = 0
    for b in range(w.B):
        if pre["done"][b]:
            for k in pre:
                assert np.array_equal(post[k][b], pre[k][b])
            continue
        cv, lk, st, dn, pa = oracle.entropy_budget_update(
            pre["canvas"][b], g["sampled"][b], g["entropy"][b].astype(np.float64),
            g["argmax"][b], pre["prev_argmax"][b], int(pre["step"][b]), inp["seed"], b, w.V,
            w.max_steps, BUDGET, STOP)
        same = (np.array_equal(cv, post["canvas"][b]) and np.array_equal(lk, post["lock"][b])
                and st == post["step"][b] and dn == post["done"][b])
        assert np.array_equal(pa, post["prev_argmax"][b])
        if not same:
            H = np.maximum(g["entropy"][b].astype(np.float64), 0)
            cum = np.cumsum(np.sort(H))
            assert (np.min(np.abs(cum - BUDGET)) < 1e-5 or abs(H.mean() - STOP) < 1e-6), b
            n_amb += 1
    return n_amb


def _decidable(ref, pre, b):
    """The oracle's lock decision for sequence b cannot flip under fp32 rounding of its inputs:
    no running sum near the budget at the acceptance boundary, no near-tie across that
    boundary, mean entropy not near the stop threshold, no near-tie in an accepted sample and
    no near-tie in any argmax (stability)."""
    H = np.maximum(ref["entropy"][b], 0)
    L = H.shape[0]
    order = np.lexsort((np.arange(L), H))
    cum = np.cumsum(H[order])
    n_acc = max(1, int(np.count_nonzero(cum <= BUDGET)))
    if abs(H.mean() - STOP) < 1e-5 or np.any(ref["argmax_gap"][b] < 1e-4):
        return False
    if abs(cum[n_acc - 1] - BUDGET) < 1e-4 or (n_acc < L and abs(cum[n_acc] - BUDGET) < 1e-4):
        return False
    if n_acc < L and H[order[n_acc]] - H[order[n_acc - 1]] < 1e-5:
        return False
    return not np.any(ref["gumbel_margin"][b][order[:n_acc]] < 1e-4)


def test_entropy_budget_loop_teacher_forced():
    w, inp, sampler, dev = _setup()
    state = CanvasState.from_numpy(inp["canvas"], inp["lock"], inp["step"], inp["done"])
    H64, E64 = exact_f64(inp["H"], "bf16"), exact_f64(inp["E"], "bf16")
    n_steps = n_checked = 0
    for _ in range(w.max_steps):
        pre = _state_np(state)
        if pre["done"].all():
            break
        out = sampler.step(dev["H"], dev["E"], dev["T"], dev["tau"], state, inp["seed"])
        torch.cuda.synchronize()
        g, post = out_np(out), _state_np(state)
        ref = oracle.sampler_step(H64, E64, inp["T"], inp["tau"], pre["canvas"], pre["lock"],
                                  pre["step"], pre["done"], inp["seed"], max_steps=w.max_steps,
                                  lock_rule=oracle.LOCK_ENTROPY_BUDGET, entropy_budget=BUDGET,
                                  stop_entropy=STOP, t_schedule=SCHED,
                                  prev_argmax=pre["prev_argmax"])
        rows = [(b, i) for b in range(w.B) if not pre["done"][b] for i in range(w.L)]
        compare_outputs(g, ref, rows)
        _rule_on_gpu_outputs(w, inp, pre, g, post)
        for b in range(w.B):
            if pre["done"][b] or not _decidable(ref, pre, b):
                continue
            n_checked += 1
            assert np.array_equal(post["lock"][b], ref["lock"][b]), b
            assert np.array_equal(post["canvas"][b], ref["canvas"][b]), b
            assert post["done"][b] == ref["done"][b]
        n_steps += 1
    assert n_steps >= 2 and n_checked >= 1
    assert state.done.all().item()


@pytest.mark.parametrize("impl", ["auto", "fused"])
def test_entropy_budget_graph_loop_equals_plain_launches(impl):
    # the fused pass is a cooperative launch: it must capture into the loop's graph too
    results = []
    for use_graph in (True, False):
        w, inp, sampler, dev = _setup(impl=impl)
        state = CanvasState.from_numpy(inp["canvas"], inp["lock"], inp["step"], inp["done"])
        out = StepOutputs.empty(w.B, w.L, w.d)
        sampler.loop(dev["E"], dev["T"], dev["tau"], state, inp["seed"], out, H=dev["H"],
                     use_graph=use_graph)
        torch.cuda.synchronize()
        results.append((_state_np(state), out_np(out)))
        assert sampler.device_status() == 0
    (sa, oa), (sb, ob) = results
    for k in sa:
        assert np.array_equal(sa[k], sb[k]), k
    assert np.array_equal(oa["sampled"], ob["sampled"])
    assert sa["done"].all()


def test_stop_takes_the_argmax_on_a_peaked_canvas():
    # very peaked logits: entropies ~0 and a stable argmax, so step 1 stops with the argmax
    w, inp, sampler, dev = _setup(B=1)
    H = inp["H"].copy()
    E32 = W.bf16_bits_to_f32(inp["E"])
    tgt = inp["targets"][0]
    H[0] = W.f32_to_bf16_bits(60.0 * E32[tgt] / np.linalg.norm(E32[tgt], axis=1, keepdims=True))
    Hd = to_torch_input(H, "bf16")
    state = CanvasState.from_numpy(inp["canvas"], inp["lock"], inp["step"], inp["done"])
    for k in range(2):
        out = sampler.step(Hd, dev["E"], dev["T"], dev["tau"], state, inp["seed"])
    torch.cuda.synchronize()
    g = out_np(out)
    assert state.done.item() == 1 and int(state.step.item()) == 2
    assert np.array_equal(state.canvas.cpu().numpy()[0], g["argmax"][0])
    assert np.array_equal(g["argmax"][0], tgt)

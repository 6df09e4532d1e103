"""The configured workloads at their full sizes, in the launch configuration the bench times.

The oracle recomputes sampled positions one by one (full vocabulary, fp64); the rest of each
step is checked through properties that hold at any size, and the lock / re-noise / stop
update is checked exactly against the rule applied to the GPU's own confidences.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from canvas_sampler_gb300 import workloads as W
from canvas_sampler_gb300.sampler import StepOutputs

from _helpers import GpuCase, check_lock_update, compare_outputs, exact_f64, out_np, oracle_step, standin_close, state_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _properties(g, w, active):
    for b in np.nonzero(active)[0]:
        assert np.all((g["sampled"][b] >= 0) & (g["sampled"][b] < w.V))
        assert np.all((g["argmax"][b] >= 0) & (g["argmax"][b] < w.V))
        assert np.all((g["conf"][b] > 0) & (g["conf"][b] <= 1.0 + 1e-6))
        assert np.all((g["entropy"][b] >= -1e-5) & (g["entropy"][b] <= math.log(w.V) + 1e-4))
        assert np.all(np.isfinite(g["s"][b]))


def _sample_positions(g, b, n):
    """Spread sample: both ends, lowest and highest confidence, and evenly spaced positions."""
    c = g["conf"][b]
    pos = {0, len(c) - 1, int(np.argmin(c)), int(np.argmax(c))}
    pos |= set(np.linspace(0, len(c) - 1, n).astype(int).tolist())
    return sorted(pos)


@pytest.mark.parametrize("impl", ["auto", "fused"])
@pytest.mark.parametrize("name,per_seq,B", [("step_bf16_b1_v262144_d2816", 12, 1),
                                            # two canvases: the race inside the paired
                                            # self-conditioning launch over two row pairs
                                            ("step_bf16_b8_v262144_d2816", 8, 2),
                                            ("step_bf16_b8_v262144_d2816", 3, 8)])
def test_full_size_step(name, per_seq, B, impl):
    w = W.WORKLOADS[name]
    if B != w.B:
        w = W.scaled(w, B=B)
    case = GpuCase(w, impl=impl)
    state = case.state()
    pre = state_np(state)
    out = case.run_step(state)
    g, post = out_np(out), state_np(state)
    active = pre["done"] == 0
    _properties(g, w, active)
    check_lock_update(pre, g, post, None, case.inp["tau"], case.inp["seed"], w.V, w.max_steps)
    rows = []
    for b in range(w.B):
        pos = _sample_positions(g, b, per_seq)
        rows += [(b, i) for i in pos]
    # oracle per sampled position, one sequence at a time (the others marked done)
    H64 = exact_f64(case.inp["H"], w.dtype)
    checked = 0
    s_elem = 0.0
    for b in range(w.B):
        pos = np.array([i for bb, i in rows if bb == b])
        only_b = np.ones(w.B, np.uint8)
        only_b[b] = 0
        ref = oracle.sampler_step(H64, case.E64, case.inp["T"].astype(np.float64),
                                  case.inp["tau"].astype(np.float64), pre["canvas"], pre["lock"],
                                  pre["step"], only_b, case.inp["seed"], top_k=w.top_k,
                                  max_steps=w.max_steps, positions=pos)
        rep = compare_outputs(g, ref, [(b, int(i)) for i in pos], top_k=w.top_k)
        checked += rep["checked"]
        s_elem = max(s_elem, rep["s_elem_max"])
    print(f"{name} ({impl}): {checked} positions against the oracle; largest elementwise "
          f"relative error of s on components >= 1% of the row's largest: {s_elem:.2e}")
    assert checked == len(rows)


def test_short_loop_full_size_teacher_forced():
    w = W.WORKLOADS["loop8_bf16_b1_v32768_d1024"]
    case = GpuCase(w)
    state = case.state()
    excl = 0
    for _ in range(w.steps):
        pre = state_np(state)
        if pre["done"].all():
            break
        out = case.run_step(state)
        g, post = out_np(out), state_np(state)
        ref = oracle_step(case, pre)
        excl += compare_outputs(g, ref, [(0, i) for i in range(w.L)])["excluded"]
        check_lock_update(pre, g, post, ref, case.inp["tau"], case.inp["seed"], w.V, w.max_steps)
    assert excl <= 8


def test_adaptive_topk_standin_loop_full_size():
    w = W.WORKLOADS["loop48_topk64_bf16_b4_v262144_d2816"]
    case = GpuCase(w)
    Wt = torch.from_numpy(case.inp["W"].view(np.int16)).view(torch.bfloat16).cuda()
    # graph loop and plain launches agree bit for bit
    results = []
    for use_graph in (True, False):
        state = case.state()
        out = StepOutputs.empty(w.B, w.L, w.d)
        Hbuf = torch.zeros(w.B, w.L, w.d, dtype=torch.bfloat16, device="cuda")
        case.sampler.loop(case.E, case.T, case.tau, state, case.inp["seed"], out, W=Wt, H_buf=Hbuf,
                          use_graph=use_graph)
        torch.cuda.synchronize()
        results.append((state_np(state), out_np(out)))
    (sa, oa), (sb, ob) = results
    for k in sa:
        assert np.array_equal(sa[k], sb[k]), k
    assert np.array_equal(oa["sampled"], ob["sampled"])
    assert sa["done"].all() and sa["step"].max() <= w.max_steps
    assert case.sampler.device_status() == 0
    # teacher-forced first step on sampled positions: stand-in H, then the step
    state = case.state()
    pre = state_np(state)
    s0 = torch.zeros(w.B, w.L, w.d, dtype=torch.float32, device="cuda")
    Hbuf = torch.zeros(w.B, w.L, w.d, dtype=torch.bfloat16, device="cuda")
    case.sampler.standin_hidden(Wt, s0, case.E, state.canvas, state.done, Hbuf)
    out = StepOutputs.empty(w.B, w.L, w.d)
    case.sampler.step(Hbuf, case.E, case.T, case.tau, state, case.inp["seed"], out=out)
    torch.cuda.synchronize()
    g, post = out_np(out), state_np(state)
    check_lock_update(pre, g, post, None, case.inp["tau"], case.inp["seed"], w.V, w.max_steps)
    H_bits = Hbuf.view(torch.int16).cpu().numpy().view(np.uint16)
    pos = np.array([0, 77, 255])
    E64 = case.E64
    for b in range(w.B):
        standin_close(H_bits[b, pos], case.inp["W"], np.zeros((len(pos), w.d)), E64,
                      pre["canvas"][b, pos])
    mask = np.ones(w.B, np.uint8)
    excluded = 0
    for b in range(w.B):
        m = mask.copy()
        m[b] = 0
        ref = oracle.sampler_step(oracle.bf16_bits_to_f64(H_bits), E64, case.inp["T"],
                                  case.inp["tau"], pre["canvas"], pre["lock"], pre["step"], m,
                                  case.inp["seed"], top_k=w.top_k, max_steps=w.max_steps,
                                  positions=pos)
        excluded += compare_outputs(g, ref, [(b, int(i)) for i in pos], top_k=w.top_k)["excluded"]
    assert excluded <= 2, excluded


def test_adaptive_topk_standin_loop_full_size_teacher_forced():
    """The full-size B = 4, top-64 stand-in loop run step by step (stand-in H from the previous
    step's s and the current canvas, then the step), teacher-forced against the oracle at the
    first, second, middle and last steps: the GPU's stand-in H against the oracle's, then the
    oracle's step on the GPU's H at >= 16 positions per sequence (both ends, the lowest and
    highest confidence, evenly spaced), and the lock update exactly against the rule applied
    to the GPU's own confidences. Near-uniform stand-in softmaxes put a few per cent of the
    positions at an ambiguous top-64 boundary; the exclusions are bounded and printed."""
    w = W.WORKLOADS["loop48_topk64_bf16_b4_v262144_d2816"]
    case = GpuCase(w)
    Wt = torch.from_numpy(case.inp["W"].view(np.int16)).view(torch.bfloat16).cuda()
    state = case.state()
    s_prev = torch.zeros(w.B, w.L, w.d, dtype=torch.float32, device="cuda")
    Hbuf = torch.zeros(w.B, w.L, w.d, dtype=torch.bfloat16, device="cuda")
    picked = {0, 1, w.max_steps // 2}
    records = {}
    last = None
    n_steps = 0
    for it in range(w.max_steps):
        pre = state_np(state)
        if pre["done"].all():
            break
        case.sampler.standin_hidden(Wt, s_prev, case.E, state.canvas, state.done, Hbuf)
        out = StepOutputs.empty(w.B, w.L, w.d)
        out.s.copy_(s_prev)
        case.sampler.step(Hbuf, case.E, case.T, case.tau, state, case.inp["seed"], out=out)
        torch.cuda.synchronize()
        rec = {"it": it, "pre": pre, "post": state_np(state), "g": out_np(out),
               "H_bits": Hbuf.view(torch.int16).cpu().numpy().view(np.uint16).copy(),
               "s_prev": s_prev.cpu().numpy().astype(np.float64)}
        if it in picked:
            records[it] = rec
        last = rec
        s_prev = out.s.clone()
        n_steps += 1
    assert state.done.all().item() and n_steps <= w.max_steps
    assert case.sampler.device_status() == 0
    records[last["it"]] = last
    E64 = case.E64
    checked = excluded = 0
    for it in sorted(records):
        r = records[it]
        pre, g, post = r["pre"], r["g"], r["post"]
        check_lock_update(pre, g, post, None, case.inp["tau"], case.inp["seed"], w.V, w.max_steps)
        active = pre["done"] == 0
        _properties(g, w, active)
        H64 = oracle.bf16_bits_to_f64(r["H_bits"])
        for b in np.nonzero(active)[0]:
            pos = np.array(_sample_positions(g, b, 16))
            standin_close(r["H_bits"][b, pos], case.inp["W"], r["s_prev"][b, pos], E64,
                          pre["canvas"][b, pos])
            only_b = np.ones(w.B, np.uint8)
            only_b[b] = 0
            ref = oracle.sampler_step(H64, E64, case.inp["T"], case.inp["tau"], pre["canvas"],
                                      pre["lock"], pre["step"], only_b, case.inp["seed"],
                                      top_k=w.top_k, max_steps=w.max_steps, positions=pos)
            rep = compare_outputs(g, ref, [(int(b), int(i)) for i in pos], top_k=w.top_k)
            checked += rep["checked"]
            excluded += rep["excluded"]
    print(f"full-size top-64 stand-in loop: {n_steps} steps; steps {sorted(records)} checked at "
          f"{checked} positions, {excluded} excluded")
    assert checked >= 16 * w.B * len(records) // 2
    assert excluded <= max(2, int(0.12 * checked)), (excluded, checked)


def test_largest_vocabulary_closed_form():
    """V = 2^24, the largest vocabulary the boundary accepts (d = 256, one canvas). E is zero
    except unit rows at K special tokens (first and last tokens, chunk and tile edges), and
    H_i = a_i e_k(i), so each position has exactly one hot token with logit a_i and 2^24 - 1
    tokens at 0: the softmax, entropy, argmax, confidences and s have closed forms for every
    position, and the oracle's Philox gives the exact Gumbel-max winner (no matmul) for a sample
    of positions. Logits above 19.6 put every other segment out of the race's reach; the others
    race all 2^24 tokens."""
    V, d, L, T = 1 << 24, 256, 256, 1.0
    special = np.array([0, 5, 8191, 8192, 262143, 1 << 23, 12345678, V - 256, V - 1], np.int64)
    K = len(special)
    a_vals = np.array([-5.0, 0.0, 3.0, 10.0, 17.0, 25.0, 40.0])
    k_of = np.arange(L) % K
    a = a_vals[np.arange(L) % len(a_vals)]
    E = torch.zeros(V, d, dtype=torch.bfloat16, device="cuda")
    E[torch.from_numpy(special).cuda(), torch.arange(K, device="cuda")] = 1.0
    Hn = np.zeros((1, L, d), np.float32)
    Hn[0, np.arange(L), k_of] = a
    H = torch.from_numpy(Hn).to(torch.bfloat16).cuda()
    seed = 20240601
    Tt = torch.full((1,), T, dtype=torch.float32, device="cuda")
    tau = torch.full((1,), 0.9, dtype=torch.float32, device="cuda")
    from canvas_sampler_gb300.sampler import CanvasState, Sampler
    sampler = Sampler(V, d, canvas_len=L, max_batch=1, dtype="bf16", max_steps=48)
    assert sampler.impl == "tensor"
    rng = np.random.default_rng(3)
    canvas = rng.integers(0, V, size=(1, L), dtype=np.int32)
    state = CanvasState.from_numpy(canvas, np.zeros((1, L), np.uint8), np.zeros(1, np.int32),
                                   np.zeros(1, np.uint8))
    out = sampler.step(H, E, Tt, tau, state, seed)
    torch.cuda.synchronize()
    g = out_np(out)
    del E
    # closed forms (fp64)
    hot = special[k_of]
    m = np.maximum(a, 0.0)
    l = np.exp(a - m) + (V - 1) * np.exp(-m)
    p_hot, p_oth = np.exp(a - m) / l, np.exp(-m) / l
    ent = -(p_hot * np.log(p_hot) + (V - 1) * p_oth * np.log(p_oth))
    s_ref = np.tile(p_oth[:, None], (1, d))
    s_ref[:, K:] = 0.0
    s_ref[np.arange(L), k_of] = p_hot
    # ties at 0 go to the lowest token: token 0 unless it is the hot token below 0
    arg_ref = np.where(a > 0, hot, np.where((a < 0) & (hot == 0), 1, 0))
    assert np.array_equal(g["argmax"][0], arg_ref)
    assert np.all(np.abs(g["entropy"][0] - ent) <= 2e-5 * np.maximum(1.0, ent))
    err = np.linalg.norm(g["s"][0] - s_ref, axis=1) / np.linalg.norm(s_ref, axis=1)
    assert err.max() <= 2e-5, err.max()
    # every sample is the hot token or a 0-logit token; its confidence is the matching p
    x = g["sampled"][0]
    c_ref = np.where(x == hot, p_hot, p_oth)
    assert np.all(np.abs(g["conf"][0] - c_ref) <= 2e-5 * c_ref)
    # exact winners for a sample of positions, one per logit value. With 2^24 draws of a 24-bit
    # uniform about two tokens share the largest draw, so exact ties of the top perturbed logits
    # are common here; they go to the lowest token on both sides and are checked too. Only
    # near-ties (a nonzero margin below 1e-4) are left out.
    checked = 0
    for i in range(len(a_vals)):
        u = oracle.gumbel_uniforms(seed, 0, [i], 0, V)[0]
        v = -np.log(-np.log(u))
        v[hot[i]] += a[i]
        top2 = np.partition(v, -2)[-2:]
        if 0.0 < top2[1] - top2[0] < 1e-4:
            continue
        assert x[i] == int(np.argmax(v)), (i, x[i], int(np.argmax(v)))
        checked += 1
    assert checked >= len(a_vals) - 1

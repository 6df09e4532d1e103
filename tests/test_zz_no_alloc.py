"""The no-allocation step entry point against the regular one.

ds_sampler_step_noalloc serves callers that cannot allocate device memory at step time (a
serving engine that has reserved nearly all HBM for its own pools, or a latency-critical path
that must not let cudaMalloc synchronise the device); it keeps its scratch in one fixed array
inside the library instead of a sampler's workspace. This file runs last so that a failure here
cannot hide failures elsewhere, and it passes both alone and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from canvas_sampler_gb300 import _lib as C
from canvas_sampler_gb300 import workloads as W
from canvas_sampler_gb300.sampler import CanvasState, Sampler, StepOutputs

from _helpers import GpuCase, compare_outputs, out_np, oracle_step, state_np

pytestmark = pytest.mark.gpu

REL_TOL = 2e-5


def _inputs(B=2, V=8192, d=256):
    w = W.scaled(W.WORKLOADS["step_bf16_b8_v262144_d2816"], V=V, d=d, B=B)
    inp = W.make_inputs(w)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return w, inp, dev(inp["E"]), dev(inp["H"]), torch.from_numpy(inp["T"]).cuda(), \
        torch.from_numpy(inp["tau"]).cuda()


def _args(sampler, H, E, T, tau, state, out, seed):
    return sampler._step_args(H, E, T, tau, state, out, seed)


def _close(a: StepOutputs, b: StepOutputs, ref: dict, rows):
    """a (no-allocation step) against b (the sampler's step) within the tests' tolerance, on the
    rows where the oracle's (ref) top-two perturbed logits are at least 1e-4 apart: elsewhere
    the two steps' different probability representations (row-relative there, tile-relative
    here) may pick either of two near-tied tokens. Returns the number of excluded rows."""
    ga, gb = out_np(a), out_np(b)
    excluded = 0
    for bb, i in rows:
        if ref["gumbel_margin"][bb, i] < 1e-4:
            excluded += 1
            continue
        assert ga["sampled"][bb, i] == gb["sampled"][bb, i], (bb, i)
        ca, cb = float(ga["conf"][bb, i]), float(gb["conf"][bb, i])
        assert abs(ca - cb) <= REL_TOL * max(abs(cb), 1e-30), (bb, i, ca, cb)
    for bb, i in rows:
        if ref["argmax_gap"][bb, i] >= 1e-4:
            assert ga["argmax"][bb, i] == gb["argmax"][bb, i], (bb, i)
    x, y = a.entropy.double(), b.entropy.double()
    assert torch.all((x - y).abs() <= REL_TOL * y.abs().clamp_min(1.0)), "entropy"
    rel = (a.s.double() - b.s.double()).norm(dim=-1) / b.s.double().norm(dim=-1)
    assert rel.max().item() <= REL_TOL
    return excluded


def test_no_alloc_step_matches_the_sampler_step_twice_in_a_row():
    lib = C.load_library()
    w, inp, E, H, T, tau = _inputs()
    case = GpuCase(w, inputs=inp)
    ref = case.sampler
    cfg = ref._cfg
    st_ref = CanvasState.from_numpy(inp["canvas"], inp["lock"], inp["step"], inp["done"])
    st_new = st_ref.clone()
    rows = [(b, i) for b in range(w.B) for i in range(w.L)]
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # the second call continues the canvas from the first call's state
        pre = state_np(st_new)
        oracle_ref = oracle_step(case, pre)
        out_ref = ref.step(H, E, T, tau, st_ref, inp["seed"])
        out_new = StepOutputs.empty(w.B, w.L, w.d)
        a = _args(ref, H, E, T, tau, st_new, out_new, inp["seed"])
        rc = lib.ds_sampler_step_noalloc(ctypes.byref(cfg), ctypes.byref(a), stream)
        assert rc == C.DS_OK, C.status_string(rc)
        status = ctypes.c_int32(-1)
        assert lib.ds_sampler_noalloc_status(stream, ctypes.byref(status)) == C.DS_OK
        assert status.value == C.DS_OK
        torch.cuda.synchronize()
        excluded = _close(out_new, out_ref, oracle_ref, rows)
        assert excluded <= max(2, len(rows) // 100), excluded
        # the no-allocation step against the oracle as well
        rep = compare_outputs(out_np(out_new), oracle_ref, rows)
        assert rep["excluded"] <= max(2, len(rows) // 100)
        if excluded == 0:
            for k in ("canvas", "lock", "step", "done"):
                assert torch.equal(getattr(st_new, k), getattr(st_ref, k)), (call, k)
        else:  # a near-tie may lock a different token: continue both from the same state
            for k in ("canvas", "lock", "step", "done"):
                getattr(st_ref, k).copy_(getattr(st_new, k))
    assert int(st_new.step[0]) == 2


def test_no_alloc_status_reads_and_clears():
    lib = C.load_library()
    status = ctypes.c_int32(-1)
    assert lib.ds_sampler_noalloc_status(None, ctypes.byref(status)) == C.DS_OK
    assert status.value == C.DS_OK
    assert lib.ds_sampler_noalloc_status(None, None) == C.DS_ERR_INVALID_ARG


def test_no_alloc_step_rejects_what_does_not_fit():
    lib = C.load_library()
    w, inp, E, H, T, tau = _inputs(B=1, V=32768, d=256)
    ref = Sampler(w.V, w.d, canvas_len=w.L, max_batch=1, dtype="bf16")
    st = CanvasState.from_numpy(inp["canvas"], inp["lock"], inp["step"], inp["done"])
    out = StepOutputs.empty(1, w.L, w.d)
    out.sampled.fill_(-3)
    cfg = C.ds_sampler_config(max_batch=1, canvas_len=w.L, d_model=w.d, dtype=0, vocab=w.V,
                              top_k=0, max_steps=48, impl=0)
    a = _args(ref, H, E, T, tau, st, out, 1)
    rc = lib.ds_sampler_step_noalloc(ctypes.byref(cfg), ctypes.byref(a), None)
    assert rc == C.DS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out.sampled == -3)  # nothing was enqueued


def test_no_alloc_topk_step_matches_oracle():
    # the no-allocation top-k path materialises y (the tensor-core logits in fp32), selects each
    # chunk's top k from it and splits exp(y - m) for the self-conditioning GEMM; the sampler's
    # own top-k path selects from the stored probabilities instead: both against the oracle
    from dataclasses import replace
    lib = C.load_library()
    w = replace(W.scaled(W.WORKLOADS["loop8_bf16_b1_v32768_d1024"], V=8192, d=512, B=2), top_k=8)
    case = GpuCase(w, impl="tensor")
    pre = state_np(case.state())
    cfg = case.sampler._cfg
    st = case.state()
    out = StepOutputs.empty(w.B, w.L, w.d)
    a = _args(case.sampler, case.H, case.E, case.T, case.tau, st, out, case.inp["seed"])
    rc = lib.ds_sampler_step_noalloc(ctypes.byref(cfg), ctypes.byref(a),
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == C.DS_OK, C.status_string(rc)
    torch.cuda.synchronize()
    ref = oracle_step(case, pre)
    rows = [(b, i) for b in range(w.B) for i in range(w.L)]
    rep = compare_outputs(out_np(out), ref, rows, top_k=w.top_k)
    assert rep["checked"] == len(rows)
    assert rep["excluded"] <= max(2, len(rows) // 100)
    # the sampler's step on the same inputs
    out2 = case.run_step(case.state())
    rep2 = compare_outputs(out_np(out2), ref, rows, top_k=w.top_k)
    assert rep2["excluded"] <= max(2, len(rows) // 100)

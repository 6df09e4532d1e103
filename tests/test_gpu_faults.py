"""The bounded-wait failure path on the GPU, without faulting or hanging it: a kernel waits on a
barrier that nothing completes, gives up after a short limit and reports a time-out through the
device error word; the context stays usable and the next step is unaffected."""
import numpy as np
import pytest
import torch

from canvas_sampler_gb300 import _lib as C
from canvas_sampler_gb300 import workloads as W

from _helpers import GpuCase, out_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    w = W.scaled(W.WORKLOADS["loop8_bf16_b1_v32768_d1024"], V=4096, d=256, B=1)
    case = GpuCase(w)
    lib = C.load_library()
    ref = out_np(case.run_step(case.state()))
    assert case.sampler.device_status() == C.DS_OK
    rc = lib.ds_sampler_selftest_wait(case.sampler.handle, 5_000_000, None)  # 5 ms
    assert rc == C.DS_OK
    assert case.sampler.device_status() == C.DS_ERR_TIMEOUT
    assert case.sampler.device_status() == C.DS_OK  # reading clears the word
    again = out_np(case.run_step(case.state()))
    for k in ref:
        assert np.array_equal(ref[k], again[k]), k
    assert lib.ds_sampler_selftest_wait(case.sampler.handle, 10, None) == C.DS_ERR_INVALID_ARG


def test_out_of_range_canvas_token_is_clamped_and_reported():
    # the stand-in reads E[canvas]: a token outside [0, V) in device memory is clamped into E
    # (rows 0 and V - 1) and reported as DS_ERR_DEVICE through the device error word; the
    # context stays usable
    w = W.scaled(W.WORKLOADS["loop48_topk64_bf16_b4_v262144_d2816"], V=4096, d=256, B=1)
    inp = W.make_inputs(w)
    case = GpuCase(w, inputs=inp)
    Wt = torch.from_numpy(inp["W"].view(np.int16)).view(torch.bfloat16).cuda()
    s_prev = torch.zeros(w.B, w.L, w.d, dtype=torch.float32, device="cuda")
    bad = inp["canvas"].copy()
    bad[0, 3], bad[0, 10] = -5, w.V + 7
    clamped = bad.copy()
    clamped[0, 3], clamped[0, 10] = 0, w.V - 1
    H_bad = torch.zeros(w.B, w.L, w.d, dtype=torch.bfloat16, device="cuda")
    H_ref = torch.zeros_like(H_bad)
    assert case.sampler.device_status() == C.DS_OK
    case.sampler.standin_hidden(Wt, s_prev, case.E, torch.from_numpy(bad).cuda(), None, H_bad)
    torch.cuda.synchronize()
    assert case.sampler.device_status() == C.DS_ERR_DEVICE
    assert case.sampler.device_status() == C.DS_OK  # reading clears the word
    case.sampler.standin_hidden(Wt, s_prev, case.E, torch.from_numpy(clamped).cuda(), None, H_ref)
    torch.cuda.synchronize()
    assert case.sampler.device_status() == C.DS_OK
    assert torch.equal(H_bad.view(torch.int16), H_ref.view(torch.int16))


def test_host_step_refuses_out_of_range_canvas_tokens():
    import ctypes
    from canvas_sampler_gb300.sampler import CanvasState, StepOutputs
    w = W.scaled(W.WORKLOADS["loop8_bf16_b1_v32768_d1024"], V=4096, d=256, B=1)
    inp = W.make_inputs(w)
    case = GpuCase(w, inputs=inp)
    lib = C.load_library()
    for tok in (-1, w.V):
        cv = inp["canvas"].copy()
        cv[0, 17] = tok
        hs = CanvasState(torch.from_numpy(cv), torch.zeros(1, w.L, dtype=torch.uint8),
                         torch.zeros(1, dtype=torch.int32), torch.zeros(1, dtype=torch.uint8))
        hout = StepOutputs.empty(1, w.L, w.d, device="cpu")
        hout.sampled.fill_(-3)
        Hh = case.H.cpu()
        a = case.sampler._step_args(Hh, case.E, case.T.cpu(), case.tau.cpu(), hs, hout,
                                    inp["seed"])
        rc = lib.ds_sampler_step_host(case.sampler.handle, ctypes.byref(a), None)
        assert rc == C.DS_ERR_INVALID_ARG
        assert torch.all(hout.sampled == -3) and int(hs.step[0]) == 0

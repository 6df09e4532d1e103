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

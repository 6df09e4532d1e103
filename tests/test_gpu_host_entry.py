"""The host-buffer entry point (ds_sampler_step_host) against the device entry point on the same
inputs: every output and every state buffer must agree bit for bit, including partial batches
(batch < max_batch), finished sequences and the entropy-budget rule's prev_argmax."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from canvas_sampler_gb300 import workloads as W
from canvas_sampler_gb300.sampler import CanvasState, Sampler, StepOutputs

from _helpers import to_torch_input

pytestmark = pytest.mark.gpu

BASE = W.WORKLOADS["step_bf16_b8_v262144_d2816"]


def _pinned(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a if dtype is None else a.astype(dtype)))
    return t.pin_memory()


@pytest.mark.parametrize("s_pinned", [True, False], ids=["s_pinned", "s_pageable"])
@pytest.mark.parametrize("rule", ["threshold", "entropy_budget"])
@pytest.mark.parametrize("batch,done", [(3, (0, 1, 0)), (4, (0, 0, 0, 0)), (1, (0,))])
def test_host_entry_matches_device(rule, batch, done, s_pinned):
    # s in page-locked memory is written by the step directly; in pageable memory it comes back
    # by a copy after the step: both must give the device step's results
    w = replace(W.scaled(BASE, V=8192, d=256, B=batch), max_steps=12)
    inp = W.make_inputs(w)
    inp["done"] = np.array(done, np.uint8)
    kw = {}
    if rule == "entropy_budget":
        kw = dict(lock_rule="entropy_budget", entropy_budget=0.1, stop_entropy=0.005,
                  t_schedule=(0.8, 0.4))
    # the sampler is sized for four sequences; the step runs `batch` of them
    sampler = Sampler(w.V, w.d, canvas_len=w.L, max_batch=4, dtype="bf16",
                      max_steps=w.max_steps, **kw)
    E = to_torch_input(inp["E"], "bf16")
    H = to_torch_input(inp["H"], "bf16")
    T = torch.from_numpy(inp["T"]).cuda()
    tau = torch.from_numpy(inp["tau"]).cuda()
    rng = np.random.default_rng(5)
    # a step in progress: some positions locked, a previous argmax for the entropy rule
    lock = (rng.random((batch, w.L)) < 0.3).astype(np.uint8)
    step = np.full(batch, 2, np.int32)
    prev = rng.integers(0, w.V, size=(batch, w.L), dtype=np.int32)
    dev_state = CanvasState.from_numpy(inp["canvas"], lock, step, inp["done"], prev_argmax=prev)
    dev_out = StepOutputs.empty(batch, w.L, w.d)
    for t in (dev_out.s, dev_out.conf, dev_out.entropy):
        t.fill_(-7.0)
    dev_out.sampled.fill_(-7)
    dev_out.argmax.fill_(-7)
    sampler.step(H, E, T, tau, dev_state, inp["seed"], out=dev_out)
    torch.cuda.synchronize()

    host_state = CanvasState(_pinned(inp["canvas"]), _pinned(lock), _pinned(step),
                             _pinned(inp["done"]), _pinned(prev))
    host_out = StepOutputs.empty(batch, w.L, w.d, pin=True)
    if not s_pinned:
        host_out.s = torch.zeros(batch, w.L, w.d, dtype=torch.float32)
        assert not host_out.s.is_pinned()
    for t in (host_out.s, host_out.conf, host_out.entropy):
        t.fill_(-7.0)
    host_out.sampled.fill_(-7)
    host_out.argmax.fill_(-7)
    sampler.step_host(H.cpu().pin_memory(), E, T.cpu().pin_memory(), tau.cpu().pin_memory(),
                      host_state, inp["seed"], host_out)
    for k, v in vars(dev_out).items():
        assert np.array_equal(v.cpu().numpy(), getattr(host_out, k).numpy()), k
    for k in ("canvas", "lock", "step", "done", "prev_argmax"):
        assert np.array_equal(getattr(dev_state, k).cpu().numpy(),
                              getattr(host_state, k).numpy()), k
    # something happened: a live sequence was sampled and its step advanced
    live = [b for b in range(batch) if not done[b]]
    assert np.all(host_out.sampled.numpy()[live] >= 0)
    assert np.all(host_state.step.numpy()[live] == 3)

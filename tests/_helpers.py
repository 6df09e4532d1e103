"""Shared helpers of the GPU parity tests: run a step through the C ABI, run the oracle on the
same inputs, and compare within the stated tolerances.

Tolerances (fp32 kernels against the fp64 oracle):
  s                  row-norm relative error ||ds|| / ||s|| <= 2e-5
  conf (probability) relative error <= 2e-5
  entropy            absolute error <= 2e-5 * max(1, H)
  sampled / argmax   identical, except positions whose top-two (perturbed) logits are within
                     1e-4 of each other (and, with top-k, where a token within 1e-4 of the k-th
                     logit could also win: see the oracle's topk_risk)
  lock / canvas      identical, except where a lock decision is ambiguous: |c - tau| <= 2e-5 tau,
                     an ambiguous sample, or (forced lock) top-two unlocked confidences within
                     2e-5 relative; those sequences are checked against the lock rule applied to
                     the GPU's own confidences instead, which must match exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from canvas_sampler_gb300 import workloads as W
from canvas_sampler_gb300.sampler import CanvasState, Sampler, StepOutputs

REL_TOL = 2e-5
MARGIN = 1e-4


def to_torch_input(arr, dtype_name):
    if dtype_name == "fp32":
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).cuda()


def exact_f64(arr, dtype_name):
    if arr is None:
        return None
    if dtype_name == "fp32":
        return np.asarray(arr, dtype=np.float64)
    return oracle.bf16_bits_to_f64(arr)


class GpuCase:
    """A workload's inputs on the device plus a sampler for it."""

    def __init__(self, w: W.Workload, impl="auto", inputs=None, max_batch=None):
        self.w = w
        self.inp = inputs if inputs is not None else W.make_inputs(w)
        self.E = to_torch_input(self.inp["E"], w.dtype)
        self.H = None if self.inp["H"] is None else to_torch_input(self.inp["H"], w.dtype)
        self.T = torch.from_numpy(self.inp["T"]).cuda()
        self.tau = torch.from_numpy(self.inp["tau"]).cuda()
        self.sampler = Sampler(w.V, w.d, canvas_len=w.L, max_batch=max_batch or w.B,
                               dtype=w.dtype, top_k=w.top_k, max_steps=w.max_steps, impl=impl)
        self._E64 = None

    @property
    def E64(self):
        if self._E64 is None:
            self._E64 = exact_f64(self.inp["E"], self.w.dtype)
        return self._E64

    def state(self):
        i = self.inp
        return CanvasState.from_numpy(i["canvas"], i["lock"], i["step"], i["done"])

    def run_step(self, state: CanvasState, H=None, seed=None):
        out = self.sampler.step(self.H if H is None else H, self.E, self.T, self.tau, state,
                                self.inp["seed"] if seed is None else seed)
        torch.cuda.synchronize()
        return out


def state_np(state: CanvasState) -> dict:
    return {"canvas": state.canvas.cpu().numpy(), "lock": state.lock.cpu().numpy(),
            "step": state.step.cpu().numpy(), "done": state.done.cpu().numpy()}


def out_np(out: StepOutputs) -> dict:
    return {"s": out.s.cpu().numpy(), "sampled": out.sampled.cpu().numpy(),
            "conf": out.conf.cpu().numpy(), "entropy": out.entropy.cpu().numpy(),
            "argmax": out.argmax.cpu().numpy()}


def compare_outputs(gpu: dict, ref: dict, active_rows, *, top_k=0):
    """Per-position checks of s, conf, entropy, argmax, sampled. Returns counts and, for the
    record, the largest elementwise relative error of s over the components that are not
    negligible (|s_k| >= 1% of the row's largest |s_k|; the asserted tolerance is the row-norm
    one)."""
    n_excl = 0
    n = 0
    s_elem = 0.0
    for b, i in active_rows:
        n += 1
        s_g, s_r = gpu["s"][b, i].astype(np.float64), ref["s"][b, i]
        err = np.linalg.norm(s_g - s_r) / max(np.linalg.norm(s_r), 1e-300)
        assert err <= REL_TOL, f"s mismatch at {(b, i)}: rel err {err:.3g}"
        big = np.abs(s_r) >= 0.01 * np.abs(s_r).max()
        if big.any():
            s_elem = max(s_elem, float(np.max(np.abs(s_g[big] - s_r[big]) / np.abs(s_r[big]))))
        H_r = ref["entropy"][b, i]
        assert abs(gpu["entropy"][b, i] - H_r) <= REL_TOL * max(1.0, abs(H_r)), (
            f"entropy at {(b, i)}: {gpu['entropy'][b, i]} vs {H_r}")
        if ref["argmax_gap"][b, i] >= MARGIN:
            assert gpu["argmax"][b, i] == ref["argmax"][b, i], f"argmax at {(b, i)}"
        ambiguous = ref["gumbel_margin"][b, i] < MARGIN or (top_k and ref["topk_risk"][b, i])
        if ambiguous:
            n_excl += 1
            continue
        assert gpu["sampled"][b, i] == ref["sampled"][b, i], (
            f"sampled at {(b, i)}: {gpu['sampled'][b, i]} vs {ref['sampled'][b, i]} "
            f"(margin {ref['gumbel_margin'][b, i]:.3g})")
        c_r = ref["conf"][b, i]
        assert abs(gpu["conf"][b, i] - c_r) <= REL_TOL * c_r + 1e-30, (
            f"conf at {(b, i)}: {gpu['conf'][b, i]} vs {c_r}")
    return {"checked": n, "excluded": n_excl, "s_elem_max": s_elem}


def check_lock_update(pre: dict, gpu_out: dict, gpu_post: dict, ref: dict | None, tau, seed, V,
                      max_steps, block=0):
    """The GPU's lock / re-noise / stop against the rule applied to the GPU's own sampled
    tokens and confidences (exact), and against the oracle where the decision is unambiguous."""
    B = pre["canvas"].shape[0]
    n_undecidable = 0
    for b in range(B):
        if pre["done"][b]:
            for k in ("canvas", "lock", "step", "done"):
                assert np.array_equal(gpu_post[k][b], pre[k][b]), f"done sequence {b} changed {k}"
            continue
        cv, lk, st, dn = oracle.lock_update(pre["canvas"][b], pre["lock"][b], gpu_out["sampled"][b],
                                            gpu_out["conf"][b].astype(np.float64), float(tau[b]),
                                            int(pre["step"][b]), seed, b + (block << 16), V,
                                            max_steps)
        assert np.array_equal(gpu_post["lock"][b], lk), f"lock rule on GPU inputs, seq {b}"
        assert np.array_equal(gpu_post["canvas"][b], cv), f"canvas rule on GPU inputs, seq {b}"
        assert gpu_post["step"][b] == st and gpu_post["done"][b] == dn
        if ref is None:
            continue
        c = ref["conf"][b]
        unl = pre["lock"][b] == 0
        amb = unl & ((np.abs(c - float(tau[b])) <= REL_TOL * float(tau[b])) |
                     (ref["gumbel_margin"][b] < MARGIN) | ref["topk_risk"][b])
        passing = unl & (c >= float(tau[b]))
        forced_amb = False
        if not passing.any() and unl.any() and int(pre["step"][b]) + 1 < max_steps:
            cu = np.sort(c[unl])[::-1]
            forced_amb = cu.shape[0] > 1 and (cu[0] - cu[1]) <= REL_TOL * cu[0]
        if amb.any() or forced_amb:
            n_undecidable += 1
            continue
        assert np.array_equal(gpu_post["lock"][b], ref["lock"][b]), f"lock vs oracle, seq {b}"
        assert np.array_equal(gpu_post["canvas"][b], ref["canvas"][b]), f"canvas vs oracle, seq {b}"
        assert gpu_post["done"][b] == ref["done"][b]
    return n_undecidable


def standin_close(got_bits, W_bits, s_prev, E64, canvas):
    """GPU stand-in H (bf16 bits) against the oracle's: within one bf16 rounding of the exact
    value plus the fp32 accumulation error of the 2d-term dot product (bounded by
    2d * 2^-24 * sum |W||u|). Returns the fraction of elements that differ at all."""
    W = oracle.bf16_bits_to_f64(W_bits)
    s_b = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(s_prev))
    u = np.concatenate([s_b, E64[np.asarray(canvas)]], axis=-1)
    x = u @ W.T
    scale = np.abs(u) @ np.abs(W).T
    exact = np.tanh(x)
    got = oracle.bf16_bits_to_f64(got_bits)
    n_terms = W.shape[1]
    bound = np.abs(exact) * 2.0 ** -8 + n_terms * 2.0 ** -24 * scale + 1e-30
    assert np.all(np.abs(got - exact) <= bound), float(np.max(np.abs(got - exact) / bound))
    want = oracle.f64_to_bf16_bits(exact)
    return float(np.mean(got_bits != want))


def oracle_step(case: GpuCase, pre: dict, H64=None, positions=None):
    w = case.w
    H64 = exact_f64(case.inp["H"], w.dtype) if H64 is None else H64
    return oracle.sampler_step(H64, case.E64, case.inp["T"].astype(np.float64),
                               case.inp["tau"].astype(np.float64), pre["canvas"], pre["lock"],
                               pre["step"], pre["done"], case.inp["seed"], top_k=w.top_k,
                               max_steps=w.max_steps, positions=positions)


def full_step_check(case: GpuCase, state: CanvasState, H=None, H64=None):
    """One GPU step against the oracle over every position; returns (gpu_out, post, report)."""
    pre = state_np(state)
    out = case.run_step(state, H=H)
    g = out_np(out)
    post = state_np(state)
    ref = oracle_step(case, pre, H64=H64)
    rows = [(b, i) for b in range(case.w.B) if not pre["done"][b] for i in range(case.w.L)]
    rep = compare_outputs(g, ref, rows, top_k=case.w.top_k)
    rep["undecidable"] = check_lock_update(pre, g, post, ref, case.inp["tau"], case.inp["seed"],
                                           case.w.V, case.w.max_steps)
    return g, post, rep

"""GPU parity of one sampler step (through the C ABI) against the fp64 oracle.

Sizes here are small enough for the oracle to finish in seconds while still spanning several
tiles, several vocabulary chunks and ragged tails. Full-size workloads are in
test_gpu_fullsize.py.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from canvas_sampler_gb300 import _lib as C
from canvas_sampler_gb300 import workloads as W
from canvas_sampler_gb300.sampler import CanvasState, Sampler, StepOutputs, philox4x32_10

from _helpers import GpuCase, compare_outputs, full_step_check, out_np, oracle_step, standin_close, state_np

pytestmark = pytest.mark.gpu

BASE_PEAKED = W.WORKLOADS["loop8_bf16_b1_v32768_d1024"]
BASE_BATCH = W.WORKLOADS["step_bf16_b8_v262144_d2816"]
BASE_TOPK = W.WORKLOADS["loop48_topk64_bf16_b4_v262144_d2816"]


def test_philox_matches_oracle():
    rng = np.random.default_rng(0)
    ctr = rng.integers(0, 2**32, size=(1 << 16, 4), dtype=np.uint64).astype(np.uint32)
    for seed in (0, 1, 0xDEADBEEF12345678):
        got = philox4x32_10(torch.from_numpy(ctr.view(np.int32)).cuda(), seed)
        got = got.cpu().numpy().view(np.uint32)
        want = oracle.philox4x32_10(ctr[:, 0], ctr[:, 1], ctr[:, 2], ctr[:, 3],
                                    oracle.philox.seed_key(seed))
        assert np.array_equal(got, want)


def test_tiny_fp32_workload_full_parity():
    case = GpuCase(W.WORKLOADS["tiny_fp32_b1_v4096_d256"])
    assert case.sampler.impl == "simt"
    _, post, rep = full_step_check(case, case.state())
    assert rep["excluded"] <= 2 and rep["undecidable"] == 0
    assert post["step"][0] == 1


CASES = [
    # (name, base recipe, B, V, d, L): several tiles, several 8192-token chunks, ragged tails;
    # B * L % 256 == 0 runs the logits GEMM as CTA pairs (256-row tiles), else one CTA per tile
    ("peaked_v16384_d512", BASE_PEAKED, 1, 16384, 512, 256),
    ("peaked_ragged_v8960_d320", BASE_PEAKED, 1, 8960, 320, 256),
    ("batched_b3_v8192_d256", BASE_BATCH, 3, 8192, 256, 256),
    # 1536 (row, chunk) items: the race's own launch takes two warps per item (8 and 4 warps per
    # item in the smaller cases, one in the larger)
    ("batched_b3_v16384_d256", BASE_BATCH, 3, 16384, 256, 256),
    ("canvas128_b3_v8192_d512", BASE_BATCH, 3, 8192, 512, 128),
    ("canvas128_b2_v8960_d256", BASE_BATCH, 2, 8960, 256, 128),
    # B * L <= 512 and d >= 2048: the row merge and the race run inside the self-conditioning
    # launch by default
    ("canvas128_b2_v8192_d2048", BASE_BATCH, 2, 8192, 2048, 128),
    ("batched_b2_v8192_d2048", BASE_BATCH, 2, 8192, 2048, 256),
]


@pytest.mark.parametrize("impl", ["tensor", "simt", "fused"])
@pytest.mark.parametrize("name,base,B,V,d,L", CASES, ids=[c[0] for c in CASES])
def test_step_parity(impl, name, base, B, V, d, L):
    if impl == "fused" and d % 256:
        pytest.skip("the fused pass takes d % 256 == 0")
    w = W.scaled(base, V=V, d=d, B=B, L=L)
    case = GpuCase(w, impl=impl)
    assert case.sampler.impl == impl
    _, _, rep = full_step_check(case, case.state())
    assert rep["excluded"] <= max(2, rep["checked"] // 100)
    assert rep["undecidable"] <= 1


@pytest.mark.parametrize("impl", ["tensor", "simt", "fused"])
@pytest.mark.parametrize("T", [0.1, 2.5])
def test_extreme_temperatures(impl, T):
    # T = 0.1 multiplies the logits by ten (peaked rows reach y - mean ~ 10 c ln V, hundreds);
    # T = 2.5 flattens them: both against the oracle on every position
    w = W.scaled(BASE_BATCH, V=16384, d=256, B=2)
    inp = W.make_inputs(w)
    inp["T"] = np.full(w.B, T, np.float32)
    case = GpuCase(w, inputs=inp, impl=impl)
    _, _, rep = full_step_check(case, case.state())
    assert rep["excluded"] <= max(2, rep["checked"] // 100)
    assert rep["undecidable"] <= 1


@pytest.mark.parametrize("k", [1, 64, 256])
def test_topk_step_parity(k):
    # the top-k recipe with fixed peaked hidden states (the stand-in loop is tested elsewhere)
    from dataclasses import replace
    w = replace(W.scaled(BASE_TOPK, V=16384, d=256, B=2), h_mode="peaked", top_k=k)
    case = GpuCase(w)
    _, _, rep = full_step_check(case, case.state())
    assert rep["excluded"] <= max(2, rep["checked"] // 100)


def _logits_ref(case, w):
    H64 = oracle.bf16_bits_to_f64(case.inp["H"]).reshape(-1, w.d)
    ref = (H64 @ case.E64.T) / float(case.inp["T"][0])
    # fp32 accumulation of exact bf16 products over d terms: at most one fp32 ulp (2^-23) of
    # the running sum per addition, whatever the rounding direction
    bound = w.d * 2.0 ** -23 * (np.abs(H64) @ np.abs(case.E64).T) + 1e-12
    return ref, bound


@pytest.mark.parametrize("impl", ["tensor", "fused"])
def test_segment_maxima_and_probabilities_match_oracle(impl):
    """Tensor-core paths without top-k: each 128-token segment's maximum is the segment maximum
    of the oracle's logits within the fp32 accumulation bound, and P_hi + P_lo = exp(y - m_ref)
    within that bound, the exp approximation (4e-6, twice on the tensor path: the tile factor) and
    the hi/lo split (2^-17), both relative; m_ref is the segment's maximum (fused pass) or the
    maximum of its 256-token tile (tensor path)."""
    w = W.scaled(BASE_PEAKED, V=8192, d=1024, B=1)
    case = GpuCase(w, impl=impl)
    case.run_step(case.state())
    R, nseg = w.B * w.L, w.V // 128
    seg = case.sampler.debug_tensor(4).cpu().numpy().view(np.float32).reshape(R, nseg, 4)
    m_g = seg[:, :, 0].astype(np.float64)
    arg = seg[:, :, 3].view(np.int32)
    ref, bound = _logits_ref(case, w)
    ref_s, bound_s = ref.reshape(R, nseg, 128), bound.reshape(R, nseg, 128)
    assert np.all(np.abs(m_g - ref_s.max(axis=2)) <= bound_s.max(axis=2))
    # the argmax is a maximum of the oracle's logits within twice the bound
    at = np.take_along_axis(ref, arg.astype(np.int64), axis=1)
    assert np.all(at >= ref_s.max(axis=2) - 2 * bound_s.max(axis=2))
    hi = oracle.bf16_bits_to_f64(case.sampler.debug_tensor(2).cpu().numpy().view(np.uint16))
    lo = oracle.bf16_bits_to_f64(case.sampler.debug_tensor(3).cpu().numpy().view(np.uint16))
    p = (hi + lo).reshape(R, nseg, 128)
    m_ref = m_g
    if impl == "tensor":
        m_ref = np.repeat(m_g.reshape(R, nseg // 2, 2).max(axis=2), 2, axis=1)
    p_ref = np.exp(ref_s - m_ref[:, :, None])
    err = np.abs(p - p_ref)
    tol = p_ref * (np.expm1(bound_s + bound_s.max(axis=2, keepdims=True)) + 8e-6 + 2.0 ** -17)
    big = p_ref > 1e-13  # y - m_g > -30, where the exp approximation keeps 4e-6
    assert np.all(err[big] <= tol[big])


@pytest.mark.parametrize("impl", ["tensor", "fused"])
def test_simt_and_tensor_agree(impl):
    w = W.scaled(BASE_PEAKED, V=8192, d=256, B=1)
    inp = W.make_inputs(w)
    a = GpuCase(w, impl=impl, inputs=inp)
    b = GpuCase(w, impl="simt", inputs=inp)
    oa, ob = out_np(a.run_step(a.state())), out_np(b.run_step(b.state()))
    rel = np.linalg.norm(oa["s"] - ob["s"], axis=-1) / np.linalg.norm(ob["s"], axis=-1)
    assert rel.max() < 4e-5
    assert (oa["sampled"] == ob["sampled"]).mean() > 0.99


def test_fused_rejects_what_it_cannot_run():
    lib = C.load_library()
    h = ctypes.c_void_p()
    for top_k, d in ((8, 256), (0, 320)):
        cfg = C.ds_sampler_config(max_batch=1, canvas_len=256, d_model=d, dtype=0, vocab=8192,
                                  top_k=top_k, max_steps=48, impl=C.DS_IMPL_FUSED)
        assert lib.ds_sampler_create(ctypes.byref(cfg), ctypes.byref(h)) == C.DS_ERR_UNSUPPORTED


def test_done_sequences_are_untouched():
    w = W.scaled(BASE_BATCH, V=8192, d=256, B=3)
    inp = W.make_inputs(w)
    inp["done"] = np.array([0, 1, 0], np.uint8)
    case = GpuCase(w, inputs=inp)
    state = case.state()
    out = StepOutputs.empty(3, w.L, w.d)
    for t in (out.s, out.conf, out.entropy):
        t.fill_(-7.0)
    out.sampled.fill_(-7)
    out.argmax.fill_(-7)
    pre = state_np(state)
    case.sampler.step(case.H, case.E, case.T, case.tau, state, inp["seed"], out=out)
    torch.cuda.synchronize()
    post = state_np(state)
    for k in pre:
        assert np.array_equal(post[k][1], pre[k][1])
    g = out_np(out)
    assert np.all(g["s"][1] == -7.0) and np.all(g["sampled"][1] == -7)
    assert np.all(g["sampled"][0] >= 0) and np.all(g["sampled"][2] >= 0)
    ref = oracle_step(case, pre)
    compare_outputs(g, ref, [(b, i) for b in (0, 2) for i in range(w.L)])


@pytest.mark.parametrize("impl", ["tensor", "simt", "fused"])
def test_all_finished_batch_is_a_no_op(impl):
    # every sequence finished on entry: the step writes nothing, and the sampler is left ready
    # for the next step (which must match the oracle: no queue counter or stale record left)
    w = W.scaled(BASE_BATCH, V=8192, d=256, B=2)
    inp = W.make_inputs(w)
    inp["done"] = np.ones(2, np.uint8)
    case = GpuCase(w, inputs=inp, impl=impl)
    state = case.state()
    out = StepOutputs.empty(2, w.L, w.d)
    for t in (out.s, out.conf, out.entropy):
        t.fill_(-7.0)
    out.sampled.fill_(-7)
    out.argmax.fill_(-7)
    pre = state_np(state)
    case.sampler.step(case.H, case.E, case.T, case.tau, state, inp["seed"], out=out)
    torch.cuda.synchronize()
    post, g = state_np(state), out_np(out)
    for k in pre:
        assert np.array_equal(post[k], pre[k]), k
    assert np.all(g["s"] == -7.0) and np.all(g["conf"] == -7.0) and np.all(g["entropy"] == -7.0)
    assert np.all(g["sampled"] == -7) and np.all(g["argmax"] == -7)
    assert case.sampler.device_status() == C.DS_OK
    inp["done"] = np.zeros(2, np.uint8)
    _, _, rep = full_step_check(case, case.state())
    assert rep["excluded"] <= 2 and rep["undecidable"] <= 1


@pytest.mark.parametrize("d", [256, 2048])
@pytest.mark.parametrize("done", [(1, 0), (0, 1)])
def test_done_sequence_inside_a_pair_tile(done, d):
    # 128-token canvases: one 256-row tile of the paired logits GEMM holds both sequences, one
    # of them finished; the live one must match the oracle and the finished one stay untouched
    # (at d = 2048 the row merge and the race run inside the self-conditioning launch)
    w = W.scaled(BASE_BATCH, V=8192, d=d, B=2, L=128)
    inp = W.make_inputs(w)
    inp["done"] = np.array(done, np.uint8)
    case = GpuCase(w, inputs=inp)
    state = case.state()
    out = StepOutputs.empty(2, w.L, w.d)
    out.s.fill_(-7.0)
    out.sampled.fill_(-7)
    pre = state_np(state)
    case.sampler.step(case.H, case.E, case.T, case.tau, state, inp["seed"], out=out)
    torch.cuda.synchronize()
    post = state_np(state)
    dead, live = (0, 1) if done[0] else (1, 0)
    for k in pre:
        assert np.array_equal(post[k][dead], pre[k][dead])
    g = out_np(out)
    assert np.all(g["s"][dead] == -7.0) and np.all(g["sampled"][dead] == -7)
    ref = oracle_step(case, pre)
    compare_outputs(g, ref, [(live, i) for i in range(w.L)])


@pytest.mark.parametrize("done", [(0, 0, 0), (0, 1, 0)])
def test_race_beside_selfcond_matches_its_own_launch(monkeypatch, done):
    # the Gumbel race on warps of the self-conditioning launch (the default) against its own
    # launch: every output and state bit for bit over three steps in a row (the race's queue
    # counters must be back at zero after each launch); the last chunk is a ragged 256 tokens
    w = W.scaled(BASE_BATCH, V=41216, d=512, B=3)
    inp = W.make_inputs(w)
    inp["done"] = np.array(done, np.uint8)
    live = [b for b in range(3) if not done[b]]
    runs = []
    for env in ("0", "1"):
        monkeypatch.setenv("DS_GUMBEL_IN_SELFCOND", env)
        case = GpuCase(w, inputs=inp)
        state = case.state()
        steps = []
        for t in range(3):
            out = case.run_step(state, seed=inp["seed"] + t)
            steps.append(({k: v[live] for k, v in out_np(out).items()}, state_np(state)))
        runs.append(steps)
    for (o0, s0), (o1, s1) in zip(*runs):
        for k in o0:
            assert np.array_equal(o0[k], o1[k]), k
        for k in s0:
            assert np.array_equal(s0[k], s1[k]), k
    assert np.all(runs[1][0][0]["sampled"] >= 0)


def test_deterministic_bits():
    w = W.scaled(BASE_PEAKED, V=8192, d=512, B=1)
    case = GpuCase(w)
    o1 = out_np(case.run_step(case.state()))
    o2 = out_np(case.run_step(case.state()))
    for k in o1:
        assert np.array_equal(o1[k], o2[k]), k


def test_uniform_logits_forced_lock_and_final_step():
    # H = 0: every logit is 0, the softmax is uniform, nobody reaches tau: exactly one forced
    # lock, at the lowest position; at the last allowed step everything is committed.
    w = W.scaled(BASE_PEAKED, V=4096, d=256, B=1)
    inp = W.make_inputs(w)
    inp["H"] = np.zeros_like(inp["H"])
    case = GpuCase(w, inputs=inp)
    state = case.state()
    g, post, rep = full_step_check(case, state)
    np.testing.assert_allclose(g["conf"], 1.0 / w.V, rtol=1e-6)
    np.testing.assert_allclose(g["entropy"], np.log(w.V), rtol=2e-6)
    assert np.array_equal(g["argmax"], np.zeros_like(g["argmax"]))
    assert post["lock"].sum() == 1 and post["lock"][0, 0] == 1
    # jump to the last step
    inp2 = dict(inp)
    inp2["step"] = np.array([w.max_steps - 1], np.int32)
    case2 = GpuCase(w, inputs=inp2)
    st2 = case2.state()
    g2, post2, _ = full_step_check(case2, st2)
    assert post2["lock"].all() and post2["done"][0] == 1
    assert np.array_equal(post2["canvas"], g2["sampled"])


def test_host_entry_point_matches_device_step():
    w = W.scaled(BASE_PEAKED, V=8192, d=256, B=1)
    case = GpuCase(w)
    dev_state = case.state()
    dev = out_np(case.run_step(dev_state))
    inp = case.inp
    host_state = CanvasState(torch.from_numpy(inp["canvas"].copy()).pin_memory(),
                             torch.from_numpy(inp["lock"].copy()).pin_memory(),
                             torch.from_numpy(inp["step"].copy()).pin_memory(),
                             torch.from_numpy(inp["done"].copy()).pin_memory())
    out = StepOutputs.empty(w.B, w.L, w.d, pin=True)
    Hh = torch.from_numpy(inp["H"].view(np.int16)).view(torch.bfloat16).pin_memory()
    case.sampler.step_host(Hh, case.E, case.T.cpu().pin_memory(), case.tau.cpu().pin_memory(),
                           host_state, inp["seed"], out)
    host = {k: v.numpy() for k, v in vars(out).items()}
    for k in dev:
        assert np.array_equal(dev[k], host[k]), k
    assert np.array_equal(host_state.canvas.numpy(), dev_state.canvas.cpu().numpy())


def test_invalid_arguments_are_rejected():
    lib = C.load_library()
    cfg = C.ds_sampler_config(max_batch=1, canvas_len=200, d_model=256, dtype=0, vocab=4096,
                              top_k=0, max_steps=48, impl=0)
    h = ctypes.c_void_p()
    assert lib.ds_sampler_create(ctypes.byref(cfg), ctypes.byref(h)) == C.DS_ERR_INVALID_ARG
    cfg.canvas_len = 256
    cfg.vocab = 4000
    assert lib.ds_sampler_create(ctypes.byref(cfg), ctypes.byref(h)) == C.DS_ERR_INVALID_ARG
    cfg.vocab = 4096
    cfg.dtype = 1
    cfg.impl = C.DS_IMPL_TENSOR
    assert lib.ds_sampler_create(ctypes.byref(cfg), ctypes.byref(h)) == C.DS_ERR_UNSUPPORTED
    w = W.scaled(BASE_PEAKED, V=4096, d=256, B=1)
    case = GpuCase(w)
    st = case.state()
    out = StepOutputs.empty(1, w.L, w.d)
    a = case.sampler._step_args(case.H, case.E, case.T, case.tau, st, out, 1)
    a.batch = 2
    assert lib.ds_sampler_step(case.sampler.handle, ctypes.byref(a), None) == C.DS_ERR_INVALID_ARG
    a.batch = 0  # an empty batch is rejected: there is no step to take
    assert lib.ds_sampler_step(case.sampler.handle, ctypes.byref(a), None) == C.DS_ERR_INVALID_ARG
    a.batch = 1
    a.conf = None
    assert lib.ds_sampler_step(case.sampler.handle, ctypes.byref(a), None) == C.DS_ERR_INVALID_ARG
    a.conf = out.conf.data_ptr()
    a.H = case.H.data_ptr() + 2
    assert lib.ds_sampler_step(case.sampler.handle, ctypes.byref(a), None) == C.DS_ERR_INVALID_ARG
    assert case.sampler.device_status() == C.DS_OK


def test_standin_hidden_matches_oracle():
    w = W.scaled(BASE_TOPK, V=4096, d=256, B=2)
    inp = W.make_inputs(w)
    case = GpuCase(w, inputs=inp)
    rng = np.random.default_rng(3)
    s_prev = (rng.standard_normal((w.B, w.L, w.d)) * 0.05).astype(np.float32)
    canvas = torch.from_numpy(inp["canvas"]).cuda()
    Wt = torch.from_numpy(inp["W"].view(np.int16)).view(torch.bfloat16).cuda()
    Hout = torch.zeros(w.B, w.L, w.d, dtype=torch.bfloat16, device="cuda")
    case.sampler.standin_hidden(Wt, torch.from_numpy(s_prev).cuda(), case.E, canvas, None, Hout)
    torch.cuda.synchronize()
    got = Hout.view(torch.int16).cpu().numpy().view(np.uint16)
    frac = standin_close(got, inp["W"], s_prev.astype(np.float64), case.E64, inp["canvas"])
    assert frac < 1e-2


def test_phase_timing_levels():
    # every phase (1) and the coarse boundaries (2) account for the same step time; the coarse
    # mode folds statistics / top-k into "convert" and finalize into "lock"
    w = W.scaled(BASE_BATCH, V=8192, d=512, B=2)
    case = GpuCase(w)
    sampler = case.sampler
    for _ in range(5):  # first launches of a fresh sampler are not representative
        case.run_step(case.state())
    # the steps here are ~0.1 ms, comparable to the host's time to enqueue one, so a host stall
    # shows up in the event times: each level keeps the least of three 20-step passes
    totals = {1: float("inf"), 2: float("inf")}
    for _ in range(3):
        for level, coarse in ((1, False), (2, True)):
            sampler.set_phase_timing(True, coarse=coarse)
            for _ in range(20):
                case.run_step(case.state())
            ph, n = sampler.phase_times()
            sampler.set_phase_timing(False)
            assert n == 20
            assert ph["logits"] > 0 and ph["selfcond"] > 0 and ph["convert"] > 0 and ph["lock"] > 0
            if coarse:
                assert ph["stats"] == 0 and ph["topk"] == 0 and ph["finalize"] == 0
            else:
                assert ph["stats"] > 0 and ph["finalize"] > 0
            totals[level] = min(totals[level], sum(ph.values()) / n)
    assert abs(totals[1] - totals[2]) <= 0.25 * min(totals[1], totals[2])
    lib = C.load_library()
    assert lib.ds_sampler_set_phase_timing(sampler.handle, 3) == C.DS_ERR_INVALID_ARG


@pytest.mark.parametrize("V,d", [(4096, 256), (264192, 64)], ids=["v4096", "v264192_fallback"])
def test_topk_uniform_logits_take_the_lowest_tokens(V, d):
    # H = 0: every logit ties, so the top 8 are tokens 0..7 (ties go to the lower token), each
    # with probability 1/8 after truncation, and the Gumbel draws decide among them exactly as in
    # the oracle. At V = 264192 the 2064 segments all reach the floor: more than the candidate
    # list holds, so the selection scans the segment maxima instead.
    from dataclasses import replace
    w = replace(W.scaled(BASE_PEAKED, V=V, d=d, B=1), top_k=8)
    inp = W.make_inputs(w)
    inp["H"] = np.zeros_like(inp["H"])
    case = GpuCase(w, inputs=inp, impl="tensor")
    state = case.state()
    pre = state_np(state)
    g = out_np(case.run_step(state))
    assert np.all((g["sampled"] >= 0) & (g["sampled"] < 8))
    np.testing.assert_allclose(g["conf"], 1.0 / 8, rtol=1e-6)
    pos = np.arange(0, w.L, 8)
    ref = oracle_step(case, pre, positions=pos)
    assert np.array_equal(g["sampled"][0, pos], ref["sampled"][0, pos])


@pytest.mark.parametrize("L", [512, 1024])
def test_long_canvases_lock_update(L):
    # canvases longer than the finalize CTA (256 threads): the lock update folded into the
    # finalize launch takes several positions a thread; the whole step against the oracle, a
    # forced lock (uniform logits) at the lowest position and the commit at the last step
    w = W.scaled(BASE_BATCH, V=4096, d=256, B=2, L=L)
    case = GpuCase(w, impl="tensor")
    _, post, rep = full_step_check(case, case.state())
    assert rep["excluded"] <= max(2, rep["checked"] // 100)
    assert post["step"].tolist() == [1, 1]
    inp = W.make_inputs(w)
    inp["H"] = np.zeros_like(inp["H"])
    case_u = GpuCase(w, inputs=inp, impl="tensor")
    _, post_u, _ = full_step_check(case_u, case_u.state())
    assert post_u["lock"].sum(axis=1).tolist() == [1, 1] and np.all(post_u["lock"][:, 0] == 1)
    inp2 = dict(inp)
    inp2["step"] = np.full(2, w.max_steps - 1, np.int32)
    case_f = GpuCase(w, inputs=inp2, impl="tensor")
    g_f, post_f, _ = full_step_check(case_f, case_f.state())
    assert post_f["lock"].all() and post_f["done"].all()
    assert np.array_equal(post_f["canvas"], g_f["sampled"])

"""Pins of the oracle's sampler step against closed forms, brute force and invariants.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a wrong sign
or index, a transposed operand, an off-by-one in the lock rule) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy import stats

from oracle import sampler as O
from oracle.philox import philox4x32_10, seed_key

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------- closed forms (golden)

@pytest.mark.parametrize("case", _golden()["softmax_cases"], ids=lambda c: c["name"])
def test_closed_form_softmax_cases(case):
    E = np.array(case["E"], dtype=np.float64)
    H = np.array(case["H"], dtype=np.float64)[None]  # B = 1
    L = H.shape[1]
    out = O.sampler_step(H, E, [case["T"]], [2.0], np.zeros((1, L), np.int64),
                         np.zeros((1, L), np.uint8), np.zeros(1, np.int64), np.zeros(1, np.uint8),
                         seed=3)
    np.testing.assert_allclose(out["s"][0, 0], case["s"], rtol=1e-13, atol=1e-15)
    assert out["entropy"][0, 0] == pytest.approx(case["entropy"], rel=1e-13, abs=1e-15)
    assert out["argmax"][0, 0] == case["argmax"]
    assert out["pmax"][0, 0] == pytest.approx(case["pmax"], rel=1e-13)
    # the confidence is the probability of whichever token was sampled
    x = out["sampled"][0, 0]
    assert out["conf"][0, 0] == pytest.approx(case["p"][x], rel=1e-13)


@pytest.mark.parametrize("case", _golden()["lock_cases"], ids=lambda c: c["name"])
def test_closed_form_lock_cases(case):
    V = 16
    cv, lk, st, dn = O.lock_update(np.array(case["canvas"]), np.array(case["lock"]),
                                   np.array(case["sampled"]), np.array(case["conf"]), case["tau"],
                                   case["step"], 77, 0, V, case["max_steps"])
    assert lk.tolist() == case["lock_after"]
    for i, tok in case["locked_tokens"].items():
        assert cv[int(i)] == tok
    expect = O.renoise_tokens(77, 0, np.array(case["renoised"], dtype=np.int64), case["step"], V)
    assert cv[case["renoised"]].tolist() == expect.tolist()
    assert (st, dn) == (case["step_after"], case["done_after"])


# ---------------------------------------------------------------- brute force, tiny V

def _brute_step_row(h, E, T, u, top_k):
    """Textbook loops with math.fsum: one position."""
    V, d = E.shape
    y = [math.fsum(h[k] * E[j, k] for k in range(d)) / T for j in range(V)]
    m = max(y)
    e = [math.exp(v - m) for v in y]
    l = math.fsum(e)
    p = [v / l for v in e]
    ent = -math.fsum(q * math.log(q) for q in p if q > 0)
    s = [math.fsum(p[j] * E[j, k] for j in range(V)) for k in range(d)]
    am = min(j for j in range(V) if y[j] == m)
    g = [-math.log(-math.log(v)) for v in u]
    if top_k:
        order = sorted(range(V), key=lambda j: (-y[j], j))[:top_k]
    else:
        order = list(range(V))
    best = max(order, key=lambda j: (y[j] + g[j], -j))
    if top_k:
        w = math.fsum(math.exp(y[j] - m) for j in order)
        c = math.exp(y[best] - m) / w
    else:
        c = p[best]
    return s, ent, am, best, c


@pytest.mark.parametrize("top_k", [0, 3])
def test_brute_force_tiny(top_k):
    rng = np.random.default_rng(2024)
    B, L, V, d = 2, 5, 7, 3
    E = rng.standard_normal((V, d))
    H = 2.0 * rng.standard_normal((B, L, d))
    T = np.array([0.8, 1.3])
    step = np.array([0, 5])
    out = O.sampler_step(H, E, T, [0.5, 0.5], np.zeros((B, L), np.int64),
                         np.zeros((B, L), np.uint8), step, np.zeros(B, np.uint8), seed=99,
                         top_k=top_k)
    for b in range(B):
        u = O.gumbel_uniforms(99, b, np.arange(L), int(step[b]), V)
        for i in range(L):
            s, ent, am, x, c = _brute_step_row(H[b, i], E, T[b], u[i], top_k)
            np.testing.assert_allclose(out["s"][b, i], s, rtol=1e-12, atol=1e-14)
            assert out["entropy"][b, i] == pytest.approx(ent, rel=1e-12, abs=1e-14)
            assert out["argmax"][b, i] == am
            assert out["sampled"][b, i] == x
            assert out["conf"][b, i] == pytest.approx(c, rel=1e-12)


def test_gumbel_uniform_mapping_matches_words():
    # u = (2 (r >> 9) + 1) / 2^24 from word (j & 3) of counter (j >> 2, i, b, 4 step)
    seed, b, i, step, V = 0x1234_5678_9ABC, 3, 17, 5, 10
    u = O.gumbel_uniforms(seed, b, [i], step, V)[0]
    for j in range(V):
        r = int(philox4x32_10(j >> 2, i, b, 4 * step, seed_key(seed))[j & 3])
        assert u[j] == (2 * (r >> 9) + 1) / 2 ** 24
    assert np.all((u > 0) & (u < 1))


def test_renoise_mapping_matches_words():
    seed, b, step, V = 9, 1, 2, 1 << 18
    pos = np.arange(8)
    tok = O.renoise_tokens(seed, b, pos, step, V)
    for i in pos:
        r = int(philox4x32_10(i >> 2, 0, b, 4 * step + 1, seed_key(seed))[i & 3])
        assert tok[i] == (r * V) >> 32


# ---------------------------------------------------------------- invariants / limits

def test_softmax_invariants():
    rng = np.random.default_rng(1)
    y = rng.standard_normal((20, 50)) * 5
    m, l, p, ent, am = O.softmax_stats(y)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-14)
    assert np.all(ent >= 0) and np.all(ent <= math.log(50) + 1e-12)
    assert np.all(am == np.argmax(y, axis=1))
    np.testing.assert_allclose(m, y.max(axis=1))


def test_self_conditioning_limit_is_the_embedding():
    # H = alpha E[j] with alpha large: s -> E[j] (E rows of unit norm, distinct)
    rng = np.random.default_rng(4)
    V, d = 40, 64
    E = rng.standard_normal((V, d))
    E /= np.linalg.norm(E, axis=1, keepdims=True)
    j = 17
    H = (300.0 * E[j])[None, None, :]
    out = O.sampler_step(H, E, [1.0], [0.5], np.zeros((1, 1), np.int64), np.zeros((1, 1), np.uint8),
                         [0], [0], seed=1)
    np.testing.assert_allclose(out["s"][0, 0], E[j], atol=1e-10)
    assert out["sampled"][0, 0] == j and out["argmax"][0, 0] == j
    assert out["entropy"][0, 0] < 1e-10


def test_zero_temperature_limit_is_argmax():
    rng = np.random.default_rng(8)
    V, d, L = 30, 8, 16
    E = rng.standard_normal((V, d))
    H = rng.standard_normal((1, L, d))
    out = O.sampler_step(H, E, [1e-7], [0.5], np.zeros((1, L), np.int64),
                         np.zeros((1, L), np.uint8), [0], [0], seed=5)
    assert np.array_equal(out["sampled"][0], out["argmax"][0])
    np.testing.assert_allclose(out["conf"][0], 1.0)


def test_uniform_logits_entropy_and_mean():
    rng = np.random.default_rng(9)
    V, d = 64, 5
    E = rng.standard_normal((V, d))
    out = O.sampler_step(np.zeros((1, 3, d)), E, [1.0], [0.5], np.zeros((1, 3), np.int64),
                         np.zeros((1, 3), np.uint8), [0], [0], seed=5)
    np.testing.assert_allclose(out["entropy"][0], math.log(V), rtol=1e-14)
    np.testing.assert_allclose(out["s"][0], np.tile(E.mean(axis=0), (3, 1)), atol=1e-14)
    assert np.all(out["argmax"][0] == 0)


def test_temperature_divides_logits():
    # y/T with T=2 equals H/2 at T=1, for every output
    rng = np.random.default_rng(10)
    V, d, L = 33, 6, 4
    E = rng.standard_normal((V, d))
    H = rng.standard_normal((1, L, d)) * 3
    a = O.sampler_step(H, E, [2.0], [0.5], np.zeros((1, L), np.int64), np.zeros((1, L), np.uint8),
                       [3], [0], seed=11)
    b = O.sampler_step(H / 2.0, E, [1.0], [0.5], np.zeros((1, L), np.int64),
                       np.zeros((1, L), np.uint8), [3], [0], seed=11)
    for k in ("s", "entropy", "conf"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-12)
    assert np.array_equal(a["sampled"], b["sampled"])


# ---------------------------------------------------------------- distributions

def test_gumbel_max_frequencies_match_softmax():
    # P(x = j) = p_j: draw one position at many step values (fresh counters each time)
    V, d = 8, 8
    E = np.eye(V)
    y_target = np.log(np.array([0.3, 0.2, 0.15, 0.1, 0.1, 0.08, 0.05, 0.02]))
    n = 40000
    counts = np.zeros(V)
    u_all = np.stack([O.gumbel_uniforms(77, 0, [0], st, V)[0] for st in range(n)])
    x = np.argmax(y_target[None, :] - np.log(-np.log(u_all)), axis=1)
    counts = np.bincount(x, minlength=V)
    p = np.exp(y_target) / np.exp(y_target).sum()
    assert stats.chisquare(counts, n * p).pvalue > 1e-4
    # and the step function agrees with this draw for a few steps
    H = y_target[None, None, :]
    for st in range(5):
        out = O.sampler_step(H, E, [1.0], [0.5], np.zeros((1, 1), np.int64),
                             np.zeros((1, 1), np.uint8), [st], [0], seed=77)
        assert out["sampled"][0, 0] == x[st]


def test_top_k_frequencies_renormalise():
    V, k = 8, 3
    y = np.log(np.array([0.3, 0.2, 0.15, 0.1, 0.1, 0.08, 0.05, 0.02]))
    n = 30000
    E = np.eye(V)
    xs = []
    for st in range(n):
        u = O.gumbel_uniforms(5, 0, [0], st, V)[0]
        v = y - np.log(-np.log(u))
        top = np.argsort(-y, kind="stable")[:k]
        xs.append(top[np.argmax(v[top])])
    counts = np.bincount(xs, minlength=V)
    assert counts[k:].sum() == 0
    q = np.exp(y[:k]) / np.exp(y[:k]).sum()
    assert stats.chisquare(counts[:k], n * q).pvalue > 1e-4
    out = O.sampler_step(y[None, None, :], E, [1.0], [0.5], np.zeros((1, 1), np.int64),
                         np.zeros((1, 1), np.uint8), [0], [0], seed=5, top_k=k)
    assert out["sampled"][0, 0] == xs[0]
    assert out["conf"][0, 0] == pytest.approx(q[xs[0]], rel=1e-12)


def test_top_k_ties_keep_lower_index():
    y = np.array([1.0, 3.0, 2.0, 3.0, 2.0, 2.0])
    assert O._top_k_set(y, 3).tolist() == [1, 2, 3]
    assert O._top_k_set(y, 4).tolist() == [1, 2, 3, 4]


def test_renoise_is_uniform():
    V = 256
    toks = np.concatenate([O.renoise_tokens(13, b, np.arange(256), st, V)
                           for b in range(4) for st in range(40)])
    assert toks.min() >= 0 and toks.max() < V
    assert stats.chisquare(np.bincount(toks, minlength=V)).pvalue > 1e-4


# ---------------------------------------------------------------- lock rule invariants

def test_lock_rule_invariants_random():
    rng = np.random.default_rng(3)
    V, L = 1000, 64
    for trial in range(200):
        lock = (rng.random(L) < rng.random()).astype(np.uint8)
        canvas = rng.integers(0, V, L)
        sampled = rng.integers(0, V, L)
        conf = rng.random(L)
        tau = rng.uniform(0.5, 1.0)
        step = int(rng.integers(0, 48))
        cv, lk, st, dn = O.lock_update(canvas, lock, sampled, conf, tau, step, 5, 2, V, 48)
        assert np.all(cv[lock == 1] == canvas[lock == 1])  # locked tokens never change
        assert np.all(lk[lock == 1] == 1)  # locks are sticky
        new = (lk == 1) & (lock == 0)
        assert np.all(cv[new] == sampled[new])
        if (lock == 0).any():
            assert new.sum() >= 1  # at least one lock per step
        if step + 1 >= 48:
            assert lk.all()
        passing = (lock == 0) & (conf >= tau)
        if passing.any() and step + 1 < 48:
            assert np.array_equal(new, passing)
        assert st == step + 1 and dn == int(lk.all())
        assert cv.min() >= 0 and cv.max() < V


def test_loop_terminates_and_resumes():
    rng = np.random.default_rng(12)
    B, L, V, d = 2, 16, 64, 8
    E = rng.standard_normal((V, d)) / math.sqrt(d)
    H = rng.standard_normal((B, L, d)) * 2
    canvas = rng.integers(0, V, (B, L))
    z = dict(lock=np.zeros((B, L), np.uint8), step=np.zeros(B, np.int64), done=np.zeros(B, np.uint8))
    full, recs = O.denoise_loop(E, [1.0, 0.8], [0.9, 0.6], canvas, seed=4, H=H, max_steps=12, **z)
    assert full["done"].all() and len(recs) <= 12
    locks = [r["lock"].sum(axis=1) for r in recs]
    for a, b in zip(locks, locks[1:]):
        assert np.all(b >= a)
    half, _ = O.denoise_loop(E, [1.0, 0.8], [0.9, 0.6], canvas, seed=4, H=H, max_steps=12,
                             max_iters=3, **z)
    rest, _ = O.denoise_loop(E, [1.0, 0.8], [0.9, 0.6], half["canvas"], half["lock"], half["step"],
                             half["done"], seed=4, H=H, max_steps=12)
    for k in ("canvas", "lock", "step", "done"):
        assert np.array_equal(rest[k], full[k])


# ---------------------------------------------------------------- number formats, stand-in

def test_bf16_rounding_matches_library_on_fp32_values():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(100000) * 10.0 ** rng.integers(-8, 8, 100000)).astype(np.float32)
    ours = O.f64_to_bf16_bits(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rounding_is_nearest_from_fp64():
    # values a hair off a bf16 midpoint, which an fp32 detour would round to the midpoint
    rng = np.random.default_rng(7)
    base = O.bf16_bits_to_f64(rng.integers(0x3F00, 0x4300, 2000).astype(np.uint16))
    ulp = 2.0 ** (np.floor(np.log2(base)) - 7)  # bf16 keeps 7 fraction bits
    mid = base + ulp / 2
    for sgn in (-1.0, 1.0):
        x = mid + sgn * ulp * 2.0 ** -30
        got = O.bf16_bits_to_f64(O.f64_to_bf16_bits(x))
        want = np.where(sgn > 0, base + ulp, base)
        np.testing.assert_array_equal(got, want)
    # exact midpoints go to the even neighbour
    got_bits = O.f64_to_bf16_bits(mid)
    assert np.all(got_bits % 2 == 0)


def test_standin_hidden_brute_force():
    rng = np.random.default_rng(21)
    B, L, V, d = 1, 3, 10, 4
    E = O.bf16_bits_to_f64(O.f64_to_bf16_bits(rng.standard_normal((V, d)) * 0.5))
    Wb = O.f64_to_bf16_bits(rng.standard_normal((d, 2 * d)) * 0.3)
    W = O.bf16_bits_to_f64(Wb)
    s_prev = rng.standard_normal((B, L, d))
    canvas = rng.integers(0, V, (B, L))
    H = O.bf16_bits_to_f64(O.standin_hidden(Wb, s_prev, E, canvas))
    for i in range(L):
        sb = O.bf16_bits_to_f64(O.f64_to_bf16_bits(s_prev[0, i]))
        u = list(sb) + list(E[canvas[0, i]])
        for k in range(d):
            v = math.tanh(math.fsum(W[k, m] * u[m] for m in range(2 * d)))
            want = O.bf16_bits_to_f64(O.f64_to_bf16_bits(np.array([v])))[0]
            assert H[0, i, k] == want


# ---------------------------------------------------------------- the pages' default sampler

@pytest.mark.parametrize("case", _golden()["entropy_budget_cases"], ids=lambda c: c["name"])
def test_closed_form_entropy_budget_cases(case):
    V = 16
    cv, lk, st, dn, pa = O.entropy_budget_update(
        np.array(case["canvas"]), np.array(case["sampled"]), np.array(case["entropy"]),
        np.array(case["argmax"]), np.array(case["prev_argmax"]), case["step"], 31, 1, V,
        case["max_steps"], case["budget"], case["stop_entropy"])
    assert lk.tolist() == case["lock_after"]
    for i, tok in case["accepted_tokens"].items():
        assert cv[int(i)] == tok
    expect = O.renoise_tokens(31, 1, np.array(case["renoised"], dtype=np.int64), case["step"], V)
    assert cv[case["renoised"]].tolist() == expect.tolist()
    assert (st, dn) == (case["step_after"], case["done_after"])
    assert pa.tolist() == case["argmax"]


def test_closed_form_temperature_schedule():
    t = _golden()["temperature_schedule"]
    for k, want in t["points"].items():
        got = O.scheduled_temperature(t["t_start"], t["t_end"], int(k), t["max_steps"])
        assert got == pytest.approx(want, rel=1e-15)


def test_entropy_budget_invariants_random():
    rng = np.random.default_rng(17)
    V, L = 500, 40
    for _ in range(300):
        H = rng.exponential(rng.choice([0.002, 0.02, 0.2]), L)
        am = rng.integers(0, V, L)
        prev = am.copy() if rng.random() < 0.5 else rng.integers(0, V, L)
        step = int(rng.integers(0, 48))
        sampled = rng.integers(0, V, L)
        cv, lk, st, dn, pa = O.entropy_budget_update(rng.integers(0, V, L), sampled, H, am, prev,
                                                     step, 3, 0, V, 48)
        acc = lk == 1
        assert acc.sum() >= 1 and st == step + 1
        if dn:
            assert np.array_equal(cv, am) and acc.all()
        else:
            assert np.array_equal(cv[acc], sampled[acc])
            # accepted = a prefix of the ascending entropies within the budget
            order = np.lexsort((np.arange(L), H))
            k = acc.sum()
            assert set(order[:k]) == set(np.nonzero(acc)[0])
            assert k == 1 or H[order[:k]].sum() <= 0.1 + 1e-12
            assert k == L or H[order[:k + 1]].sum() > 0.1


def test_entropy_budget_loop_stops_on_a_confident_stable_canvas():
    # a canvas whose logits are very peaked settles: argmax stable, entropies ~0 -> stops early
    rng = np.random.default_rng(5)
    V, d, L = 64, 16, 8
    E = rng.standard_normal((V, d))
    t = rng.integers(0, V, L)
    H = (40.0 * E[t] / np.linalg.norm(E[t], axis=1, keepdims=True))[None]
    state, recs = O.denoise_loop(E, [1.0], [0.9], rng.integers(0, V, (1, L)),
                                 np.zeros((1, L), np.uint8), np.zeros(1, np.int64),
                                 np.zeros(1, np.uint8), seed=8, H=H, max_steps=48,
                                 lock_rule=O.LOCK_ENTROPY_BUDGET, t_schedule=(0.8, 0.4))
    assert state["done"][0] == 1 and len(recs) == 2  # step 0 cannot stop; step 1 does
    assert np.array_equal(state["canvas"][0], recs[-1]["argmax"][0])


# ---------------------------------------------------------------- block-autoregressive runs

def test_block_draws_carry_the_block_in_counter_word_2():
    # Gumbel and re-noise draws of block k use counter word 2 = b + 2^16 k: the sample is the
    # argmax of y + g with g from the scalar Philox at that counter, the re-noised tokens map
    # its words; block 0 is the single-canvas draw
    rng = np.random.default_rng(31)
    B, L, V, d, seed, step = 2, 8, 24, 6, 0xABCDEF, 3
    E = rng.standard_normal((V, d)) / math.sqrt(d)
    H = rng.standard_normal((B, L, d))
    canvas = rng.integers(0, V, (B, L))
    lock = np.zeros((B, L), np.uint8)
    st = np.full(B, step, np.int64)
    done = np.zeros(B, np.uint8)
    T, tau = [1.0, 0.9], [0.99, 0.99]
    outs = {}
    for blk in (0, 1, 7):
        out = O.sampler_step(H, E, T, tau, canvas, lock, st, done, seed, max_steps=48, block=blk)
        outs[blk] = out
        for b in range(B):
            sid = b + (blk << 16)
            y = (H[b] @ E.T) / T[b]
            for i in range(L):
                u = np.array([(2 * (int(philox4x32_10(j >> 2, i, sid, 4 * step,
                                                      seed_key(seed))[j & 3]) >> 9) + 1) / 2 ** 24
                              for j in range(V)])
                assert out["sampled"][b, i] == int(np.argmax(y[i] - np.log(-np.log(u))))
            renoised = out["lock"][b] == 0
            for i in np.nonzero(renoised)[0]:
                r = int(philox4x32_10(i >> 2, 0, sid, 4 * step + 1, seed_key(seed))[i & 3])
                assert out["canvas"][b, i] == (r * V) >> 32
    default = O.sampler_step(H, E, T, tau, canvas, lock, st, done, seed, max_steps=48)
    assert np.array_equal(default["sampled"], outs[0]["sampled"])
    assert not np.array_equal(outs[1]["sampled"], outs[7]["sampled"])


def test_block_loop_chains_fresh_denoising_loops():
    rng = np.random.default_rng(32)
    n_blocks, B, L, V, d = 3, 2, 16, 64, 8
    E = rng.standard_normal((V, d)) / math.sqrt(d)
    H = rng.standard_normal((B, L, d)) * 2
    init = rng.integers(0, V, (n_blocks, B, L))
    init[2] = init[1]  # same noise, different block: different draws
    kw = dict(H=H, max_steps=12)
    tokens, steps, recs = O.block_loop(E, [1.0, 0.8], [0.9, 0.6], init, 5, **kw)
    z = dict(lock=np.zeros((B, L), np.uint8), step=np.zeros(B, np.int64),
             done=np.zeros(B, np.uint8))
    for k in range(n_blocks):
        state, _ = O.denoise_loop(E, [1.0, 0.8], [0.9, 0.6], init[k], seed=5, block=k, **kw, **z)
        assert np.array_equal(tokens[k], state["canvas"])
        assert np.array_equal(steps[k], state["step"])
        assert np.all(steps[k] <= 12) and state["done"].all()
    assert not np.array_equal(tokens[1], tokens[2])
    # first_block shifts the block indices: blocks 1..2 alone reproduce the last two blocks
    t2, s2, _ = O.block_loop(E, [1.0, 0.8], [0.9, 0.6], init[1:], 5, first_block=1, **kw)
    assert np.array_equal(t2, tokens[1:]) and np.array_equal(s2, steps[1:])

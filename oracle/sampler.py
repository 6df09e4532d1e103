"""The canvas sampler step in plain fp64 NumPy -- test infrastructure only.

One step over a batch of canvases (B sequences, L positions, vocabulary V, width d):

1. logits      z_ij = H_i . E_j                   (technical report s.6 "Sampling": the
                                                    softmax runs over the full vocabulary)
2. temperature y_ij = z_ij / T_b
3. softmax     p_ij = exp(y_ij - m_i) / l_i,  m_i = max_j y_ij,  l_i = sum_j exp(y_ij - m_i)
               entropy_i = -sum_j p_ij ln p_ij (nats); argmax_i = lowest j with y_ij = m_i
4. self-cond.  s_i = sum_j p_ij E_j               (s.6 "Sampling": "self-conditioning
                                                    embedding matmul"; s.8: fed back as z_t)
5. sample      Gumbel-max: x_i = argmax_j (y_ij + g_ij), g_ij = -ln(-ln u_ij), lowest j on
               ties; with top-k the argmax runs over the k largest y_ij only (s.6
               "Multi-user throughput": top-k applies to the sampling step). The
               confidence c_i is the probability of x_i under the distribution sampled from.
6. lock / re-noise / stop (sokufu.com "A diffusion language model refines 256 tokens in 12
               steps"; alphasignal "How text diffusion actually works"; see lock_update).

The pages print no sampler listing; the readings taken where they are silent:

* confidence threshold: a position is locked when c_i >= tau_b;
* at least one lock per step: if no unlocked position passes, the unlocked position with
  the largest c_i (lowest i on ties) is locked;
* locks are sticky: a locked position keeps its token for the rest of the canvas;
* the last allowed step (step + 1 == max_steps) locks every remaining position with x_i;
* unlocked positions are re-noised with a fresh uniform token;
* a sequence is done when every position is locked; done sequences are left untouched;
* temperature divides the logits for the softmax, the entropy, s and the sample alike;
* top-k keeps s and the entropy on the full softmax;
* the pages' own default sampler (sokufu.com, "A diffusion language model refines 256 tokens
  in 12 steps", and its Table 2) is the second lock rule, see entropy_budget_update;
* random draws come from Philox4x32-10 keyed by the seed (low, high word), with counters
    Gumbel  (j >> 2, i, sid, 4*step + 0), word j & 3, u = (2*(r >> 9) + 1) / 2**24,
    re-noise (i >> 2, 0, sid, 4*step + 1), word i & 3, token = (r * V) >> 32,
  where sid = b + 2**16 * block: the sequence, and the block of a block-autoregressive run
  (block 0 for a single canvas). u takes 2**23 values, symmetric in (0, 1) and exactly
  representable in fp32; the token map is exactly uniform when V is a power of two.
* block-autoregressive generation (the pages' "block diffusion" continuation: a finished canvas
  is committed and the next one starts from fresh noise) is block_loop: each block is one
  denoising loop from its own initial canvas with fresh state (no locks, step 0, s = 0) and its
  own draws (block index in the counters); the model's conditioning on committed blocks is out
  of scope, so the stand-in hidden state does not see them.
"""
from __future__ import annotations

import numpy as np

from .philox import philox4x32_10, seed_key

GUMBEL_STREAM = 0
RENOISE_STREAM = 1

LOCK_THRESHOLD = 0
LOCK_ENTROPY_BUDGET = 1


def scheduled_temperature(t_start: float, t_end: float, step: int, max_steps: int) -> float:
    """Linear temperature schedule over the step budget: t_start at step 0, t_end at step
    max_steps - 1 (Table 2 of the sokufu.com article: "Linear schedule from 0.8 down to 0.4";
    the pages do not say over which steps, the budget is the plainest reading)."""
    if max_steps <= 1:
        return float(t_start)
    return float(t_start) + (float(t_end) - float(t_start)) * float(step) / float(max_steps - 1)


# --------------------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------------------

def bf16_bits_to_f64(b) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16)."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16, ties to even (one rounding, from fp64).

    The fp32 conversion is exact to within half an fp32 ulp, so it can only mislead the
    bf16 rounding when it lands exactly on a bf16 midpoint; that case is decided from the
    fp64 value itself."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    low = u & np.uint64(0xFFFF)
    base = u >> np.uint64(16)
    up = (low > 0x8000) | ((low == 0x8000) & ((base & np.uint64(1)) == 1))
    f64 = f.astype(np.float64)
    midpoint_hazard = (low == 0x8000) & (f64 != x)
    up = np.where(midpoint_hazard, np.abs(x) > np.abs(f64), up)
    return (base + up.astype(np.uint64)).astype(np.uint16)


# --------------------------------------------------------------------------------------
# random draws
# --------------------------------------------------------------------------------------

def gumbel_uniforms(seed: int, b: int, positions, step: int, V: int) -> np.ndarray:
    """u_ij in (0, 1) for positions i (array) and all tokens j < V, shape [len(i), V]."""
    positions = np.asarray(positions, dtype=np.int64)
    nblk = (V + 3) // 4
    c0 = np.arange(nblk, dtype=np.uint64)[None, :]
    c1 = positions.astype(np.uint64)[:, None]
    c3 = np.uint64(4 * int(step) + GUMBEL_STREAM)
    words = philox4x32_10(c0, c1, np.uint64(b), c3, seed_key(seed))  # [n, nblk, 4]
    r = words.reshape(len(positions), 4 * nblk)[:, :V].astype(np.float64)
    return (2.0 * np.floor(r / 512.0) + 1.0) / 16777216.0


def renoise_tokens(seed: int, b: int, positions, step: int, V: int) -> np.ndarray:
    """Uniform replacement tokens for positions i of sequence b at a step."""
    positions = np.asarray(positions, dtype=np.int64)
    c0 = (positions >> 2).astype(np.uint64)
    c3 = np.uint64(4 * int(step) + RENOISE_STREAM)
    words = philox4x32_10(c0, np.uint64(0), np.uint64(b), c3, seed_key(seed))
    r = words[np.arange(len(positions)), positions & 3].astype(np.uint64)
    return ((r * np.uint64(V)) >> np.uint64(32)).astype(np.int32)


# --------------------------------------------------------------------------------------
# the step
# --------------------------------------------------------------------------------------

def softmax_stats(y: np.ndarray):
    """Row-wise softmax of y [n, V]: (m, l, p, entropy, argmax)."""
    m = y.max(axis=1)
    e = np.exp(y - m[:, None])
    l = e.sum(axis=1)
    p = e / l[:, None]
    plogp = np.where(p > 0.0, p * np.log(np.where(p > 0.0, p, 1.0)), 0.0)
    entropy = -plogp.sum(axis=1)
    argmax = y.argmax(axis=1)  # numpy returns the first (lowest j) maximum
    return m, l, p, entropy, argmax


def _top_k_set(y_row: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest values; among equal values the lower index is kept."""
    order = np.argsort(-y_row, kind="stable")
    return np.sort(order[:k])


def _sample_row(y_row, g_row, p_row, top_k, band=1e-4):
    """Gumbel-max over the row (or its top-k set).

    Returns (x, c, margin of the top two perturbed logits, top-k risk). The risk flag is a
    diagnostic for comparisons only: it is set when logits that differ by less than `band`
    could change the top-k set in a way that changes the sample."""
    risk = False
    if top_k and top_k < y_row.shape[0]:
        cand = _top_k_set(y_row, top_k)
        v = y_row[cand] + g_row[cand]
        best = int(np.argmax(v))
        x = int(cand[best])
        w = np.exp(y_row[cand] - y_row[cand].max())
        c = float(w[best] / w.sum())
        vs = np.sort(v)
        # the set is ambiguous only if a token outside it comes within `band` of its k-th
        # logit; then the sample is at risk if the winner sits in that band (it could drop
        # out) or an outside token in the band would beat it
        yk = y_row[cand].min()
        outside = np.ones(y_row.shape[0], bool)
        outside[cand] = False
        near_out = outside & (y_row > yk - band)
        if near_out.any():
            risk = bool(y_row[x] < yk + band or
                        np.any(near_out & (y_row + g_row >= v[best] - band)))
    else:
        v = y_row + g_row
        x = int(np.argmax(v))
        c = float(p_row[x])
        vs = np.partition(v, -2)[-2:] if v.shape[0] > 1 else np.array([-np.inf, v[0]])
        vs = np.sort(vs)
    margin = float(vs[-1] - vs[-2]) if vs.shape[0] > 1 else np.inf
    return x, c, margin, risk


def sampler_step(H, E, T, tau, canvas, lock, step, done, seed, *, top_k=0, max_steps=48,
                 positions=None, row_chunk=64, lock_rule=LOCK_THRESHOLD, entropy_budget=0.1,
                 stop_entropy=0.005, t_schedule=None, prev_argmax=None, block=0):
    """One sampler step over a batch, in fp64.

    H [B, L, d] and E [V, d] are the exact input values as float64 (bf16 or fp32 inputs
    convert exactly); T, tau [B]; canvas [B, L] int; lock [B, L] 0/1; step [B]; done [B].

    Returns a dict of the outputs for active sequences (done ones keep NaN / -1 outputs and
    unchanged state): s [B, L, d], sampled, conf, entropy, argmax, pmax (= 1 / l_i), and the
    updated canvas, lock, step, done, plus diagnostics used to exclude near-ties from exact
    comparisons: gumbel_margin (top-two perturbed logits), argmax_gap (top-two logits) and
    top-k boundary gaps.

    With ``positions`` set, only those positions are computed and the lock update is
    skipped (it needs the whole canvas).

    lock_rule LOCK_ENTROPY_BUDGET replaces the threshold rule by entropy_budget_update
    (prev_argmax [B, L] carries the previous step's argmax); t_schedule = (t_start, t_end)
    replaces T by the scheduled temperature of each sequence's step. ``block`` selects the draws
    of that block of a block-autoregressive run (counter word 2 = b + 2**16 block)."""
    H = np.asarray(H, dtype=np.float64)
    E = np.asarray(E, dtype=np.float64)
    B, L, d = H.shape
    V = E.shape[0]
    pos = np.arange(L) if positions is None else np.asarray(positions, dtype=np.int64)
    out = {
        "s": np.full((B, L, d), np.nan),
        "sampled": np.full((B, L), -1, np.int64),
        "conf": np.full((B, L), np.nan),
        "entropy": np.full((B, L), np.nan),
        "argmax": np.full((B, L), -1, np.int64),
        "pmax": np.full((B, L), np.nan),
        "gumbel_margin": np.full((B, L), np.inf),
        "topk_gap": np.full((B, L), np.inf),
        "argmax_gap": np.full((B, L), np.inf),
        "topk_risk": np.zeros((B, L), bool),
    }
    for b in range(B):
        if done[b]:
            continue
        for c0 in range(0, len(pos), row_chunk):
            rows = pos[c0:c0 + row_chunk]
            Tb = (float(T[b]) if t_schedule is None else
                  scheduled_temperature(t_schedule[0], t_schedule[1], int(step[b]), max_steps))
            y = (H[b, rows] @ E.T) / Tb
            m, l, p, ent, am = softmax_stats(y)
            out["s"][b, rows] = p @ E
            out["entropy"][b, rows] = ent
            out["argmax"][b, rows] = am
            out["pmax"][b, rows] = 1.0 / l
            if V > 1:
                top2 = np.partition(y, -2, axis=1)[:, -2:]
                out["argmax_gap"][b, rows] = top2[:, 1] - top2[:, 0]
            u = gumbel_uniforms(seed, b + (int(block) << 16), rows, int(step[b]), V)
            g = -np.log(-np.log(u))
            for r, i in enumerate(rows):
                x, c, margin, risk = _sample_row(y[r], g[r], p[r], top_k)
                out["topk_risk"][b, i] = risk
                out["sampled"][b, i] = x
                out["conf"][b, i] = c
                out["gumbel_margin"][b, i] = margin
                if top_k and top_k < V:
                    ys = np.sort(y[r])
                    out["topk_gap"][b, i] = ys[-top_k] - ys[-top_k - 1]
    new = {k: np.array(v, copy=True) for k, v in
           (("canvas", canvas), ("lock", lock), ("step", step), ("done", done))}
    new["prev_argmax"] = (np.full((B, L), -1, np.int64) if prev_argmax is None
                          else np.array(prev_argmax, copy=True))
    if positions is None:
        for b in range(B):
            if done[b]:
                continue
            if lock_rule == LOCK_ENTROPY_BUDGET:
                cv, lk, st, dn, pa = entropy_budget_update(
                    new["canvas"][b], out["sampled"][b], out["entropy"][b], out["argmax"][b],
                    new["prev_argmax"][b], int(step[b]), seed, b + (int(block) << 16), V,
                    max_steps, entropy_budget, stop_entropy)
                new["prev_argmax"][b] = pa
            else:
                cv, lk, st, dn = lock_update(new["canvas"][b], new["lock"][b], out["sampled"][b],
                                             out["conf"][b], float(tau[b]), int(step[b]), seed,
                                             b + (int(block) << 16), V, max_steps)
            new["canvas"][b], new["lock"][b], new["step"][b], new["done"][b] = cv, lk, st, dn
    out.update(new)
    return out


def entropy_budget_update(canvas_b, sampled_b, entropy_b, argmax_b, prev_argmax_b, step_b, seed,
                          b, V, max_steps, budget=0.1, stop_entropy=0.005):
    """The pages' default sampler step for one sequence (sokufu.com, "A diffusion language
    model refines 256 tokens in 12 steps" and Table 2).

    Tokens are accepted from the lowest to the highest entropy until the entropy budget is
    spent (the longest prefix of the ascending order whose entropies sum to at most the budget,
    and at least one position; equal entropies in position order); every other position is
    re-noised uniformly. Acceptance is decided afresh every step (tokens stay editable).
    The canvas stops when its mean entropy is below stop_entropy and the argmax predictions
    equal those of the previous step; a stopped canvas, or one at its last allowed step, takes
    the argmax predictions. Negative entropies from rounding count as zero.

    Returns (canvas, lock = accepted this step, step + 1, done, argmax for the next step)."""
    L = len(canvas_b)
    H = np.maximum(np.asarray(entropy_b, dtype=np.float64), 0.0)
    argmax_b = np.asarray(argmax_b)
    stable = step_b > 0 and np.array_equal(argmax_b, np.asarray(prev_argmax_b))
    stop = bool(H.mean() < stop_entropy and stable)
    if stop or step_b + 1 >= max_steps:
        return (argmax_b.astype(np.asarray(canvas_b).dtype), np.ones(L, np.uint8), step_b + 1, 1,
                argmax_b.copy())
    order = np.lexsort((np.arange(L), H))
    cum = np.cumsum(H[order])
    n_acc = max(1, int(np.count_nonzero(cum <= budget)))
    accepted = np.zeros(L, bool)
    accepted[order[:n_acc]] = True
    canvas = np.array(canvas_b, copy=True)
    canvas[accepted] = np.asarray(sampled_b)[accepted]
    rest = np.nonzero(~accepted)[0]
    if rest.size:
        canvas[rest] = renoise_tokens(seed, b, rest, step_b, V)
    return canvas, accepted.astype(np.uint8), step_b + 1, 0, argmax_b.copy()


def lock_update(canvas_b, lock_b, sampled_b, conf_b, tau_b, step_b, seed, b, V, max_steps):
    """Lock confident positions, re-noise the others, advance the step; one sequence.

    Returns (canvas, lock, step, done) after the step."""
    canvas_b = np.array(canvas_b, copy=True)
    lock_b = np.array(lock_b, copy=True).astype(np.uint8)
    L = lock_b.shape[0]
    unlocked = lock_b == 0
    if step_b + 1 >= max_steps:
        newly = unlocked.copy()
    else:
        newly = unlocked & (np.asarray(conf_b) >= tau_b)
        if not newly.any() and unlocked.any():
            cand = np.where(unlocked, conf_b, -np.inf)
            newly[int(np.argmax(cand))] = True  # first maximum: lowest position
    canvas_b[newly] = np.asarray(sampled_b)[newly]
    lock_b[newly] = 1
    still = np.nonzero(lock_b == 0)[0]
    if still.size:
        canvas_b[still] = renoise_tokens(seed, b, still, step_b, V)
    done = 1 if (lock_b == 1).all() else 0
    return canvas_b, lock_b, step_b + 1, done


# --------------------------------------------------------------------------------------
# the hidden-state stand-in and the loop
# --------------------------------------------------------------------------------------

def standin_hidden(W_bits, s_prev, E, canvas):
    """H = bf16(tanh(W . [bf16(s_prev); E[x]])) per position, as bf16 bits [B, L, d].

    A stand-in for the model's decoder, which the pages do not give: it feeds the
    self-conditioning vector of the previous step (report s.8, z_t) and the current canvas
    tokens back into the next step's hidden state."""
    W = bf16_bits_to_f64(W_bits)  # [d, 2d]
    s_prev = np.asarray(s_prev, dtype=np.float64)
    E = np.asarray(E, dtype=np.float64)
    s_b = bf16_bits_to_f64(f64_to_bf16_bits(s_prev))
    u = np.concatenate([s_b, E[np.asarray(canvas)]], axis=-1)  # [B, L, 2d]
    return f64_to_bf16_bits(np.tanh(u @ W.T))


def denoise_loop(E, T, tau, canvas, lock, step, done, seed, *, H=None, W_bits=None,
                 s_prev=None, top_k=0, max_steps=48, max_iters=None, lock_rule=LOCK_THRESHOLD,
                 entropy_budget=0.1, stop_entropy=0.005, t_schedule=None, prev_argmax=None,
                 block=0):
    """Run steps until every sequence is done (or max_iters); returns the per-step records.

    Fixed-H mode passes H (fp64 [B, L, d]); stand-in mode passes W_bits and recomputes H
    from the previous s (zero at the start) and the canvas before each step."""
    E = np.asarray(E, dtype=np.float64)
    B, L = np.asarray(canvas).shape
    d = E.shape[1]
    state = {"canvas": np.array(canvas), "lock": np.array(lock), "step": np.array(step),
             "done": np.array(done),
             "s": np.zeros((B, L, d)) if s_prev is None else np.array(s_prev, np.float64),
             "prev_argmax": (np.full((B, L), -1, np.int64) if prev_argmax is None
                             else np.array(prev_argmax))}
    records = []
    iters = max_steps if max_iters is None else max_iters
    for _ in range(iters):
        if state["done"].all():
            break
        Hs = H if W_bits is None else bf16_bits_to_f64(
            standin_hidden(W_bits, state["s"], E, state["canvas"]))
        out = sampler_step(Hs, E, T, tau, state["canvas"], state["lock"], state["step"],
                           state["done"], seed, top_k=top_k, max_steps=max_steps,
                           lock_rule=lock_rule, entropy_budget=entropy_budget,
                           stop_entropy=stop_entropy, t_schedule=t_schedule,
                           prev_argmax=state["prev_argmax"], block=block)
        out["H"] = Hs
        active = state["done"] == 0
        s_new = state["s"].copy()
        s_new[active] = out["s"][active]
        state = {"canvas": out["canvas"], "lock": out["lock"], "step": out["step"],
                 "done": out["done"], "s": s_new, "prev_argmax": out["prev_argmax"]}
        records.append(out)
    return state, records


def block_loop(E, T, tau, init_canvas, seed, *, first_block=0, **loop_kw):
    """Block-autoregressive generation: for k = 0 .. n_blocks - 1 run denoise_loop from
    init_canvas[k] ([n_blocks, B, L]) with fresh state (no locks, step 0, done 0, s = 0, no
    previous argmax) and block index first_block + k, then commit the canvas.

    Returns (tokens [n_blocks, B, L], steps [n_blocks, B], per-block records)."""
    init_canvas = np.asarray(init_canvas)
    n_blocks, B, L = init_canvas.shape
    tokens = np.zeros((n_blocks, B, L), np.int64)
    steps = np.zeros((n_blocks, B), np.int64)
    records = []
    for k in range(n_blocks):
        state, rec = denoise_loop(E, T, tau, init_canvas[k], np.zeros((B, L), np.uint8),
                                  np.zeros(B, np.int64), np.zeros(B, np.uint8), seed,
                                  block=first_block + k, **loop_kw)
        tokens[k] = state["canvas"]
        steps[k] = state["step"]
        records.append(rec)
    return tokens, steps, records

"""The sampler step over a vocabulary split into shards, in plain fp64 NumPy -- test
infrastructure only.

Each shard q holds a contiguous token range [a_q, b_q) of E and computes, for every row, the
softmax statistics of its own logits y_j (j in the range) and its part of s and of the sample;
the records of all shards give the full-vocabulary step exactly. The pages give no multi-GPU
sampler: this is the decomposition that the full softmax over the vocabulary (technical report
s.6 "Sampling") admits, written out term by term.

  m_q = max_j y_j,  l_q = sum_j exp(y_j - m_q),  H_q = entropy of exp(y_j - m_q) / l_q,
  O_q = sum_j exp(y_j - m_q) E_j,  (v_q, x_q) = max_j (y_j + g_j) and its token,
  with top-k: the shard's k largest y_j (its candidates).
Merge:  m = max_q m_q,  l = sum_q l_q exp(m_q - m),  s = sum_q exp(m_q - m) O_q / l,
  entropy = sum_q w_q H_q - sum_q w_q ln w_q with w_q = l_q exp(m_q - m) / l (the entropy of a
  mixture of disjointly supported distributions), argmax = the largest m_q (lowest token on
  ties), sample = the token of the largest v_q (lowest token on ties): g_j are the same
  global-token draws as in the unsharded step; with top-k the sample is the Gumbel-max over the
  k largest of the pooled candidates (lowest token on equal values).
"""
from __future__ import annotations

import numpy as np

from .sampler import _top_k_set, gumbel_uniforms, softmax_stats


def shard_partial(H, E_shard, T, token_offset, V_total, seed, step, done, *, top_k=0):
    """Records of one shard for every row of every active sequence.

    H [B, L, d] and E_shard [n, d] as float64, T [B]; token_offset = global index of the
    shard's first token. Returns a dict of arrays [B, L(, ...)]: m, l, ent, arg (global),
    O [B, L, d], v (best perturbed logit), x (its global token), yx (y at x), and with top-k
    cand_y, cand_j [B, L, k]."""
    H = np.asarray(H, dtype=np.float64)
    E_shard = np.asarray(E_shard, dtype=np.float64)
    B, L, d = H.shape
    n = E_shard.shape[0]
    out = {k: np.full((B, L), np.nan) for k in ("m", "l", "ent", "v", "yx")}
    out["arg"] = np.full((B, L), -1, np.int64)
    out["x"] = np.full((B, L), -1, np.int64)
    out["O"] = np.full((B, L, d), np.nan)
    if top_k:
        out["cand_y"] = np.full((B, L, top_k), -np.inf)
        out["cand_j"] = np.full((B, L, top_k), -1, np.int64)
    for b in range(B):
        if done[b]:
            continue
        y = (H[b] @ E_shard.T) / float(T[b])  # [L, n]
        m, l, p, ent, am = softmax_stats(y)
        out["m"][b], out["l"][b], out["ent"][b] = m, l, ent
        out["arg"][b] = am + token_offset
        out["O"][b] = (np.exp(y - m[:, None])) @ E_shard
        u = gumbel_uniforms(seed, b, np.arange(L), int(step[b]), V_total)
        g = -np.log(-np.log(u[:, token_offset:token_offset + n]))
        v = y + g
        x = v.argmax(axis=1)  # lowest token on ties
        out["v"][b] = v[np.arange(L), x]
        out["yx"][b] = y[np.arange(L), x]
        out["x"][b] = x + token_offset
        if top_k:
            kk = min(top_k, n)
            for i in range(L):
                c = _top_k_set(y[i], kk)
                out["cand_y"][b, i, :kk] = y[i, c]
                out["cand_j"][b, i, :kk] = c + token_offset
    return out


def merge_shards(parts, T, seed, step, done, V_total, *, top_k=0):
    """The step's s, sampled, conf, entropy and argmax from the records of shards given in
    token order (a list of shard_partial dicts)."""
    B, L = parts[0]["m"].shape
    d = parts[0]["O"].shape[-1]
    res = {"s": np.full((B, L, d), np.nan), "sampled": np.full((B, L), -1, np.int64),
           "conf": np.full((B, L), np.nan), "entropy": np.full((B, L), np.nan),
           "argmax": np.full((B, L), -1, np.int64)}
    for b in range(B):
        if done[b]:
            continue
        ms = np.stack([p["m"][b] for p in parts])  # [n, L]
        m = ms.max(axis=0)
        w = np.stack([p["l"][b] for p in parts]) * np.exp(ms - m)  # [n, L]
        l = w.sum(axis=0)
        wn = w / l
        ents = np.stack([p["ent"][b] for p in parts])
        res["entropy"][b] = (wn * ents).sum(axis=0) - np.where(wn > 0, wn * np.log(
            np.where(wn > 0, wn, 1.0)), 0.0).sum(axis=0)
        q_arg = ms.argmax(axis=0)  # first (lowest-token) shard with the maximum
        res["argmax"][b] = np.stack([p["arg"][b] for p in parts])[q_arg, np.arange(L)]
        res["s"][b] = sum(np.exp(p["m"][b] - m)[:, None] * p["O"][b] for p in parts) / l[:, None]
        if not top_k:
            vs = np.stack([p["v"][b] for p in parts])
            q = vs.argmax(axis=0)
            x = np.stack([p["x"][b] for p in parts])[q, np.arange(L)]
            res["sampled"][b] = x
            yx = np.stack([p["yx"][b] for p in parts])[q, np.arange(L)]
            res["conf"][b] = np.exp(yx - m) / l
        else:
            cy = np.concatenate([p["cand_y"][b] for p in parts], axis=1)  # [L, n k]
            cj = np.concatenate([p["cand_j"][b] for p in parts], axis=1)
            u = gumbel_uniforms(seed, b, np.arange(L), int(step[b]), V_total)
            for i in range(L):
                ok = cj[i] >= 0
                order = np.lexsort((cj[i][ok], -cy[i][ok]))[:top_k]  # value desc, token asc
                yy, jj = cy[i][ok][order], cj[i][ok][order]
                g = -np.log(-np.log(u[i, jj]))
                vv = yy + g
                best = np.flatnonzero(vv == vv.max())
                t = best[np.argmin(jj[best])]
                res["sampled"][b, i] = jj[t]
                wk = np.exp(yy - yy.max())
                res["conf"][b, i] = wk[t] / wk.sum()
    return res

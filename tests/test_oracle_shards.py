"""The oracle's vocabulary-shard decomposition (oracle/shards.py) against the unsharded oracle
step: the merged records of any partition of the vocabulary give the same softmax entropy,
argmax, s, sample and confidence, with and without top-k, on peaked, spread and uniform
logits. Pins the merge identities (normaliser rescaling, the mixture entropy, cross-shard
Gumbel-max with global-token draws, pooled top-k with lowest-token ties)."""
import numpy as np
import pytest

import oracle


def _case(seed, B=2, L=24, V=512, d=8, kind="mixed"):
    rng = np.random.default_rng(seed)
    E = rng.standard_normal((V, d)) / np.sqrt(d)
    if kind == "uniform":
        H = np.zeros((B, L, d))
    else:
        t = rng.integers(0, V, size=(B, L))
        c = rng.uniform(0.2, 4.0, size=(B, L, 1)) if kind == "mixed" else np.full((B, L, 1), 3.0)
        H = c * np.log(V) * E[t] * np.sqrt(d) / np.sqrt(d) + rng.standard_normal((B, L, d))
    T = rng.uniform(0.7, 1.3, size=B)
    step = rng.integers(0, 5, size=B)
    done = np.zeros(B, np.uint8)
    return H, E, T, step, done


PARTS = {"halves": [0, 256, 512], "uneven": [0, 64, 320, 512], "quarters": [0, 128, 256, 384, 512]}


@pytest.mark.parametrize("kind", ["mixed", "peaked", "uniform"])
@pytest.mark.parametrize("cuts", list(PARTS), ids=list(PARTS))
@pytest.mark.parametrize("top_k", [0, 5])
def test_merged_shards_equal_the_full_step(kind, cuts, top_k):
    H, E, T, step, done = _case(11, kind=kind)
    B, L, d = H.shape
    V = E.shape[0]
    seed = 987654321
    tau = np.full(B, 0.9)
    canvas = np.zeros((B, L), np.int64)
    full = oracle.sampler_step(H, E, T, tau, canvas, np.zeros((B, L), np.uint8), step, done, seed,
                               top_k=top_k)
    c = PARTS[cuts]
    parts = [oracle.shard_partial(H, E[a:b], T, a, V, seed, step, done, top_k=top_k)
             for a, b in zip(c[:-1], c[1:])]
    got = oracle.merge_shards(parts, T, seed, step, done, V, top_k=top_k)
    np.testing.assert_allclose(got["s"], full["s"], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(got["entropy"], full["entropy"], rtol=1e-11, atol=1e-11)
    assert np.array_equal(got["argmax"], full["argmax"])
    assert np.array_equal(got["sampled"], full["sampled"])
    np.testing.assert_allclose(got["conf"], full["conf"], rtol=1e-11)


def test_one_shard_is_the_full_step():
    H, E, T, step, done = _case(3)
    B, L, _ = H.shape
    V = E.shape[0]
    p = oracle.shard_partial(H, E, T, 0, V, 5, step, done)
    full = oracle.sampler_step(H, E, T, np.full(B, 0.9), np.zeros((B, L), np.int64),
                               np.zeros((B, L), np.uint8), step, done, 5)
    got = oracle.merge_shards([p], T, 5, step, done, V)
    assert np.array_equal(got["sampled"], full["sampled"])
    np.testing.assert_allclose(got["entropy"], full["entropy"], rtol=1e-12, atol=1e-12)


def test_mixture_entropy_closed_form():
    # two shards, each uniform over its n tokens with logits 0 and a: the merged entropy is
    # the entropy of the two-block distribution, written out by hand
    V, n, a = 8, 4, np.log(3.0)  # block 2 is three times as likely per token
    E = np.eye(V)[:, :V]
    H = np.zeros((1, 1, V))
    H[0, 0, n:] = a  # logits: 0 on tokens 0..3, a on tokens 4..7
    T = np.ones(1)
    step = np.zeros(1, np.int64)
    done = np.zeros(1, np.uint8)
    parts = [oracle.shard_partial(H, E[:n], T, 0, V, 1, step, done),
             oracle.shard_partial(H, E[n:], T, n, V, 1, step, done)]
    got = oracle.merge_shards(parts, T, 1, step, done, V)
    p_lo, p_hi = 1.0 / 16.0, 3.0 / 16.0  # 4 * (1 + 3) = 16
    want = -(4 * p_lo * np.log(p_lo) + 4 * p_hi * np.log(p_hi))
    assert abs(got["entropy"][0, 0] - want) < 1e-13
    assert got["argmax"][0, 0] == n

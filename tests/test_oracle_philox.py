"""Pins of the oracle's Philox4x32-10 against things other than its vectorised code.

The main pin is an implementation written by others: the header-only Philox4x32-10 engine that
ships with PyTorch's C++ headers (ATen/core/PhiloxRNGEngine.h, written from the same SC'11
paper), compiled here into a small driver and compared block for block with the oracle over
random and edge-case counters and keys. Planted mistakes (a swapped multiplier or Weyl
constant, permuted output words) must make that comparison fail. Beside it: a second, scalar
implementation, bijectivity (Philox is a permutation of the counter space for a fixed key),
avalanche behaviour and the uniformity / independence statistics the sampler relies on.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
from scipy import stats

import oracle.philox as ph
from oracle.philox import philox4x32_10, philox4x32_10_scalar, seed_key

# Driver around PyTorch's engine: reads "seed subsequence offset" lines, prints the four words
# of the block the engine produces there. Its counter layout: words 0-1 = offset (low, high),
# words 2-3 = subsequence (low, high); its key: (seed low, seed high).
_DRIVER = r"""
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdio>
int main() {
  unsigned long long seed, sub, off;
  while (std::scanf("%llu %llu %llu", &seed, &sub, &off) == 3) {
    at::philox_engine e(seed, sub, off);
    unsigned a = e(), b = e(), c = e(), d = e();
    std::printf("%u %u %u %u\n", a, b, c, d);
  }
  return 0;
}
"""


def _torch_include():
    try:
        import torch
    except ImportError:
        return None
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    return inc if os.path.isfile(os.path.join(inc, "ATen", "core", "PhiloxRNGEngine.h")) else None


@pytest.fixture(scope="module")
def torch_philox(tmp_path_factory):
    """Callable (counters [n, 4], keys [n, 2]) -> blocks [n, 4] from PyTorch's engine."""
    inc = _torch_include()
    cxx = shutil.which("g++") or shutil.which("c++")
    if inc is None or cxx is None:
        pytest.skip("PyTorch C++ headers or a C++ compiler not available")
    d = tmp_path_factory.mktemp("philox_driver")
    src, exe = d / "drv.cpp", d / "drv"
    src.write_text(_DRIVER)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", inc, str(src), "-o", str(exe)], check=True,
                   capture_output=True)

    def run(ctr, key):
        ctr = np.asarray(ctr, dtype=np.uint64)
        key = np.asarray(key, dtype=np.uint64)
        seed = key[:, 0] | (key[:, 1] << np.uint64(32))
        sub = ctr[:, 2] | (ctr[:, 3] << np.uint64(32))
        off = ctr[:, 0] | (ctr[:, 1] << np.uint64(32))
        text = "".join(f"{int(a)} {int(b)} {int(c)}\n" for a, b, c in zip(seed, sub, off))
        out = subprocess.run([str(exe)], input=text, capture_output=True, text=True, check=True)
        return np.array([[int(x) for x in ln.split()] for ln in out.stdout.splitlines()],
                        dtype=np.uint64)
    return run


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64)
    key = rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64)
    edge = np.array([0, 1, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF], dtype=np.uint64)
    # every word of the counter and key at an edge value in turn, the rest random
    ec, ek = [], []
    for w in range(6):
        for v in edge:
            c, k = ctr[len(ec) % n].copy(), key[len(ec) % n].copy()
            if w < 4:
                c[w] = v
            else:
                k[w - 4] = v
            ec.append(c)
            ek.append(k)
    return np.concatenate([ctr, np.array(ec)]), np.concatenate([key, np.array(ek)])


def test_matches_pytorch_engine(torch_philox):
    ctr, key = _cases(4000, 2024)
    ref = torch_philox(ctr, key)
    got = np.stack([np.asarray(philox4x32_10(c[0], c[1], c[2], c[3], (int(k[0]), int(k[1]))),
                               dtype=np.uint64) for c, k in zip(ctr, key)])
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)
    # the scalar form too
    for c, k, r in zip(ctr[:200], key[:200], ref[:200]):
        assert philox4x32_10_scalar(tuple(int(x) for x in c), (int(k[0]), int(k[1]))) == \
            tuple(int(x) for x in r)


def test_sampler_counter_layout_matches_pytorch_engine(torch_philox):
    # the sampler's Gumbel and re-noise counters (token >> 2, position, sequence, 4 step + 0/1)
    # under a 64-bit seed's key
    seed = 0xFEEDFACE12345678
    key = seed_key(seed)
    j, i, b, st = np.meshgrid(np.arange(0, 262144, 9973), [0, 77, 255], [0, 7], [0, 47],
                              indexing="ij")
    ctr = np.stack([j.ravel() >> 2, i.ravel(), b.ravel(), 4 * st.ravel() + (j.ravel() & 1)],
                   axis=1).astype(np.uint64)
    keys = np.tile(np.array(key, dtype=np.uint64), (len(ctr), 1))
    ref = torch_philox(ctr, keys)
    got = philox4x32_10(ctr[:, 0], ctr[:, 1], ctr[:, 2], ctr[:, 3], key).astype(np.uint64)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("name,value", [("_M0", 0xCD9E8D57), ("_M1", 0xD2511F53),
                                        ("_W0", 0xBB67AE85), ("_W1", 0x9E3779B9)])
def test_planted_constant_mistake_is_caught(torch_philox, monkeypatch, name, value):
    ctr, key = _cases(64, 7)
    ref = torch_philox(ctr, key)
    monkeypatch.setattr(ph, name, value)
    got = np.array([ph.philox4x32_10_scalar(tuple(int(x) for x in c), (int(k[0]), int(k[1])))
                    for c, k in zip(ctr, key)], dtype=np.uint64)
    assert not np.array_equal(got, ref)


def test_planted_word_order_mistake_is_caught(torch_philox):
    ctr, key = _cases(64, 8)
    ref = torch_philox(ctr, key)
    got = np.array([philox4x32_10_scalar(tuple(int(x) for x in c), (int(k[0]), int(k[1])))
                    for c, k in zip(ctr, key)], dtype=np.uint64)
    for perm in ([1, 0, 2, 3], [0, 1, 3, 2], [2, 3, 0, 1], [3, 2, 1, 0]):
        assert not np.array_equal(got[:, perm], ref)


def test_vectorised_matches_scalar():
    rng = np.random.default_rng(123)
    ctr = rng.integers(0, 2**32, size=(300, 4), dtype=np.uint64)
    keys = rng.integers(0, 2**32, size=(300, 2), dtype=np.uint64)
    for c, k in zip(ctr, keys):
        v = philox4x32_10(c[0], c[1], c[2], c[3], (int(k[0]), int(k[1])))
        s = philox4x32_10_scalar(tuple(int(x) for x in c), (int(k[0]), int(k[1])))
        assert tuple(int(x) for x in v) == s


def test_broadcasting_shapes():
    out = philox4x32_10(np.arange(5)[None, :], np.arange(3)[:, None], 7, 9, (1, 2))
    assert out.shape == (3, 5, 4) and out.dtype == np.uint32
    assert tuple(int(x) for x in out[2, 4]) == philox4x32_10_scalar((4, 2, 7, 9), (1, 2))


def test_seed_key_split():
    assert seed_key(0x0123456789ABCDEF) == (0x89ABCDEF, 0x01234567)
    assert seed_key(5) == (5, 0)


def test_bijective_on_a_counter_slab():
    # Distinct counters must give distinct 128-bit blocks (Philox permutes the counter space).
    c0 = np.arange(1 << 17, dtype=np.uint64)
    out = philox4x32_10(c0, 3, 0, 1, (11, 0))
    packed = out.view(np.dtype((np.void, 16)))
    assert np.unique(packed).size == c0.size


def test_bit_balance_and_uniform_words():
    out = philox4x32_10(np.arange(1 << 16, dtype=np.uint64), 0, 0, 0, (42, 7)).reshape(-1)
    bits = ((out[:, None] >> np.arange(32, dtype=np.uint32)) & 1).mean(axis=0)
    # 262144 words: each bit's frequency within 5 sigma of 1/2
    assert np.all(np.abs(bits - 0.5) < 5 * 0.5 / np.sqrt(out.size))
    hist = np.bincount(out >> np.uint32(24), minlength=256)
    assert stats.chisquare(hist).pvalue > 1e-4


def test_avalanche_on_counter_bits():
    rng = np.random.default_rng(5)
    base = rng.integers(0, 2**32, size=(2000, 4), dtype=np.uint64)
    flips = []
    for w in range(4):
        for bit in (0, 13, 31):
            alt = base.copy()
            alt[:, w] ^= np.uint64(1 << bit)
            a = philox4x32_10(base[:, 0], base[:, 1], base[:, 2], base[:, 3], (9, 9))
            b = philox4x32_10(alt[:, 0], alt[:, 1], alt[:, 2], alt[:, 3], (9, 9))
            x = (a ^ b).view(np.uint8)
            flips.append(np.unpackbits(x).reshape(2000, -1).sum(axis=1).mean())
    flips = np.array(flips)
    # a good 128-bit mixer flips half the output bits for any single input-bit change
    assert np.all(np.abs(flips - 64.0) < 1.0), flips


def test_adjacent_counters_uncorrelated():
    out = philox4x32_10(np.arange(1 << 15, dtype=np.uint64), 1, 2, 3, (5, 6))
    u = out.reshape(-1).astype(np.float64) / 2**32
    r = np.corrcoef(u[:-1], u[1:])[0, 1]
    assert abs(r) < 5.0 / np.sqrt(u.size)


@pytest.mark.parametrize("key", [(0, 0), (0xFFFFFFFF, 0xFFFFFFFF)])
def test_key_changes_everything(key):
    a = philox4x32_10(np.arange(4096, dtype=np.uint64), 0, 0, 0, key)
    b = philox4x32_10(np.arange(4096, dtype=np.uint64), 0, 0, 0, (key[0] ^ 1, key[1]))
    assert (a == b).mean() < 0.01

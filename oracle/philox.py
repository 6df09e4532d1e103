"""Philox4x32-10, written from its published definition.

Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11,
section on the Philox family: a 4-word, 32-bit counter is passed through 10 rounds; each
round multiplies words 0 and 2 by two fixed odd constants, keeps the high and low halves
of the 64-bit products, and mixes the high halves with the other two words and the two
key words; between rounds the key words are advanced by two Weyl constants.

Test infrastructure only (see the package docstring).
"""
import numpy as np

_M0 = 0xD2511F53
_M1 = 0xCD9E8D57
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = 0xFFFFFFFF


def philox4x32_10_scalar(ctr, key):
    """One block with Python integers: ctr = (c0, c1, c2, c3), key = (k0, k1)."""
    c0, c1, c2, c3 = (int(v) & _MASK for v in ctr)
    k0, k1 = (int(v) & _MASK for v in key)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        prod0 = _M0 * c0
        prod1 = _M1 * c2
        hi0, lo0 = prod0 >> 32, prod0 & _MASK
        hi1, lo1 = prod1 >> 32, prod1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return (c0, c1, c2, c3)


def philox4x32_10(c0, c1, c2, c3, key):
    """Vectorised blocks: c0..c3 broadcastable integer arrays, key = (k0, k1) ints.

    Returns a uint32 array of shape broadcast(c0..c3) + (4,)."""
    c0, c1, c2, c3 = np.broadcast_arrays(*(np.asarray(c, dtype=np.uint64) & np.uint64(_MASK)
                                           for c in (c0, c1, c2, c3)))
    k0 = np.uint64(int(key[0]) & _MASK)
    k1 = np.uint64(int(key[1]) & _MASK)
    mask = np.uint64(_MASK)
    sh = np.uint64(32)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + np.uint64(_W0)) & mask
            k1 = (k1 + np.uint64(_W1)) & mask
        prod0 = c0 * np.uint64(_M0)
        prod1 = c2 * np.uint64(_M1)
        c0, c1, c2, c3 = ((prod1 >> sh) ^ c1 ^ k0, prod1 & mask,
                          (prod0 >> sh) ^ c3 ^ k1, prod0 & mask)
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def seed_key(seed: int):
    """The generator key of a 64-bit sampler seed: (low word, high word)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return (seed & _MASK, seed >> 32)

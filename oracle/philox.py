"""Philox4x32-10 and the uniform position sampler.  TEST INFRASTRUCTURE ONLY.

Philox4x32-10 follows its published definition (Salmon, Moraes, Dror, Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC'11): a 4x32-bit counter
and a 2x32-bit key; each of 10 rounds multiplies words 0 and 2 by the round
multipliers 0xD2511F53 and 0xCD9E8D57, forms the new counter from the
high/low halves xor'ed with the other words and the round key, and the key
is bumped by the Weyl constants 0x9E3779B9 and 0xBB67AE85 between rounds.
Pinned by the generator's published known-answer vectors.

Sampling (Prof-K section 3, stage 1: S uniform positions of [N]).  Reading
used by the engine: draws are independent (with replacement).  Draw j of row
r for call counter c and seed s uses counter (j // 2, r, c_lo, c_hi) and key
(s_lo, s_hi); the even draw takes the 64-bit word (w1 << 32 | w0), the odd
draw (w3 << 32 | w2); the position is floor(u * N / 2^64).
"""
from __future__ import annotations

import numpy as np

_MASK = np.uint64(0xFFFFFFFF)
_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10.  Inputs are 32-bit values (any int arrays); outputs uint64 arrays."""
    c0, c1, c2, c3 = (np.asarray(v, dtype=np.uint64) & _MASK for v in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK
    for _ in range(10):
        p0 = _M0 * c0          # < 2^64, exact in uint64
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + _W0) & _MASK
        k1 = (k1 + _W1) & _MASK
    return c0, c1, c2, c3


def sample_positions(n: int, s: int, seed: int, counter: int, row: int = 0) -> np.ndarray:
    """The S sampled positions of one row (int64), in draw order."""
    j = np.arange(s, dtype=np.uint64)
    pair = j >> np.uint64(1)
    w0, w1, w2, w3 = philox4x32_10(pair, row, counter & 0xFFFFFFFF, counter >> 32,
                                   seed & 0xFFFFFFFF, seed >> 32)
    even = (j & np.uint64(1)) == 0
    u = np.where(even, (w1 << np.uint64(32)) | w0, (w3 << np.uint64(32)) | w2)
    # floor(u * n / 2^64) with exact integers
    pos = [(int(v) * n) >> 64 for v in u.tolist()]
    return np.asarray(pos, dtype=np.int64)

"""Philox4x32-10 counter-based generator and the dropout keep-mask built on it.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and
its Python binding) may import this module; only ``tests/``, the package's
``smoke()`` self-check and the CPU-baseline leg of ``bench.py`` use it.

Source of the method: the dropout section of "Lecture 7 — Backward Pass and
Validation" (§Dropout) says the kernel draws its Bernoulli mask from a Philox
generator keyed by (seed, offset), and that a reference must use the same
generator with the same (seed, offset) to reproduce the mask. The pages do not
fix the word layout, so this project fixes its own convention (written out in
``keep_mask`` below). The generator itself is Philox-4x32 with 10 rounds as
published by Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy
as 1, 2, 3" (SC'11): two 32x32->64 multiplies per round, a Weyl-sequence key
schedule, and the word permutation of that paper. This file is written from
that definition in numpy; it shares nothing with the CUDA implementation.
"""
from __future__ import annotations

import numpy as np

_MASK32 = np.uint64(0xFFFFFFFF)
# Round multipliers and key-schedule increments of Philox-4x32 (Salmon et al.).
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten Philox-4x32 rounds over broadcastable uint32 counter words.

    Returns the four 32-bit output words as ``np.uint32`` arrays.
    Each round maps (c0, c1, c2, c3) with key (k0, k1) to
    (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0));
    the key is advanced by the Weyl increments (W0, W1) between rounds.
    """
    c0, c1, c2, c3 = (np.asarray(x, dtype=np.uint64) & _MASK32 for x in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK32
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK32
    for rnd in range(10):
        if rnd:
            k0 = (k0 + PHILOX_W0) & _MASK32
            k1 = (k1 + PHILOX_W1) & _MASK32
        p0 = PHILOX_M0 * c0  # < 2**64: exact in uint64
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))


def drop_threshold(p: float) -> int:
    """16-bit threshold T = floor(p * 2**16): a 16-bit value u is kept iff u >= T."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must lie in [0, 1)")
    return int(np.floor(np.float64(p) * 65536.0))


def keep_mask(b: int, h: int, H: int, N: int, rows, seed: int, offset: int, p: float):
    """Boolean keep-mask Z[i, j] for query rows ``rows`` and all N keys of head (b, h).

    Convention of this project (the pages leave it open). One Philox call
    serves eight consecutive keys of one query, each taking a 16-bit half of
    an output word:
      * key     = (lo32(seed), hi32(seed))
      * group   g = ((b*H + h)*N + i) * ceil(N/8) + floor(j/8)
      * counter = (lo32(g), hi32(g), lo32(offset), hi32(offset))
      * the value for key j is half (j mod 2) of output word ((j mod 8) div 2):
        the low 16 bits for even j, the high 16 bits for odd j
      * keep  <=>  value >= floor(p * 2**16)
    With p == 0 every entry is kept.
    """
    rows = np.asarray(rows, dtype=np.int64)
    if p == 0.0:
        return np.ones((rows.size, N), dtype=bool)
    T = np.uint32(drop_threshold(p))
    n8 = (N + 7) // 8
    grp = np.arange(n8, dtype=np.uint64)
    g = ((np.uint64(b * H + h) * np.uint64(N) + rows.astype(np.uint64))[:, None]
         * np.uint64(n8) + grp[None, :])
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    offset = int(offset) & 0xFFFFFFFFFFFFFFFF
    words = philox4x32_10(g & _MASK32, g >> np.uint64(32),
                          np.uint64(offset & 0xFFFFFFFF), np.uint64(offset >> 32),
                          np.uint64(seed & 0xFFFFFFFF), np.uint64(seed >> 32))
    # key 8q + 2w + half takes half `half` of words[w][r, q]
    w4 = np.stack(words, axis=-1)                                  # [rows, n8, 4]
    halves = np.stack([w4 & np.uint32(0xFFFF), w4 >> np.uint32(16)], axis=-1)  # [rows, n8, 4, 2]
    full = halves.reshape(rows.size, 8 * n8)[:, :N]
    return full >= T

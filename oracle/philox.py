"""Philox4x32-10 and the dropout keep mask, for the fp64 oracle.

TEST INFRASTRUCTURE ONLY. This module is part of the CPU oracle: only the
test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it. The CUDA path has
its own Philox and never calls this one.

Sources
-------
* Counter-based generator: Salmon, Moraes, Dror, Shaw, "Parallel Random
  Numbers: As Easy as 1, 2, 3" (SC'11), the Philox-4x32 bijection with
  R = 10 rounds. Each round multiplies counter words 0 and 2 by two fixed
  32-bit constants, takes the high and low halves of the 64-bit products,
  XORs the high halves with the other two counter words and the round key,
  and permutes the four words. The key is bumped by two Weyl constants
  between rounds.
* What the random numbers are for: "REDO of dropout support for mem eff
  #102038" (pytorch PR 103704), Summary: the RNG state (seed, offset) is
  passed from forward to backward so the backward regenerates the same
  mask, and the RNG is indexed by the *absolute* element index so the mask
  does not depend on how the kernel tiles the problem.

Counter mapping (a reading of that page; it fixes only "absolute index")
-----------------------------------------------------------------------
For element (b, h, i, j) of a [B, H, Sq, Sk] attention matrix::

    n    = ((b*H + h)*Sq + i)*Sk + j
    ctr  = (lo32(n >> 2), hi32(n >> 2), lo32(offset), hi32(offset))
    key  = (lo32(seed), hi32(seed))
    u    = Philox4x32_10(ctr, key)[n & 3]
    keep = u >= T,   T = floor(p * 2**32)

so one Philox call yields the draws of four consecutive elements, and the
keep decision is an integer compare (bit-exact on any hardware).
"""

import numpy as np

# Philox-4x32 multipliers and Weyl key increments (Salmon et al., SC'11).
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
PHILOX_ROUNDS = 10

_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr, key):
    """Philox-4x32-10 of a batch of 128-bit counters under one 64-bit key.

    ctr: array-like of shape (4, N) (or (4,)) holding uint32 counter words
         c0..c3. key: pair (k0, k1) of python ints < 2**32.
    Returns a uint32 array of the same shape with the four output words.
    """
    c = np.asarray(ctr, dtype=np.uint64)
    squeeze = c.ndim == 1
    if squeeze:
        c = c[:, None]
    c0, c1, c2, c3 = (c[w].copy() for w in range(4))
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    for _ in range(PHILOX_ROUNDS):
        p0 = PHILOX_M0 * c0  # exact: both factors < 2**32
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1,
                          hi0 ^ c3 ^ np.uint64(k1), lo0)
        k0 = (k0 + PHILOX_W0) & 0xFFFFFFFF
        k1 = (k1 + PHILOX_W1) & 0xFFFFFFFF
    out = np.stack([c0, c1, c2, c3]).astype(np.uint32)
    return out[:, 0] if squeeze else out


def keep_threshold(p):
    """Integer threshold T = floor(p * 2**32) for a drop probability p in [0, 1)."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must lie in [0, 1)")
    return int(np.floor(np.float64(p) * 4294967296.0))


def uniform_words(n_first, count, seed, offset):
    """The 32-bit draws u(n) for the absolute indices n_first .. n_first+count-1."""
    if count == 0:
        return np.zeros(0, dtype=np.uint32)
    g_first = n_first >> 2
    g_last = (n_first + count - 1) >> 2
    g = np.arange(g_first, g_last + 1, dtype=np.uint64)
    ctr = np.stack([
        g & _MASK32,
        g >> np.uint64(32),
        np.full_like(g, offset & 0xFFFFFFFF),
        np.full_like(g, (offset >> 32) & 0xFFFFFFFF),
    ])
    words = philox4x32_10(ctr, (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    stream = words.T.reshape(-1)  # word w of group g sits at 4*(g - g_first) + w
    start = n_first - 4 * g_first
    return stream[start:start + count]


def keep_mask_head(b, h, H, Sq, Sk, p, seed, offset):
    """Boolean keep mask [Sq, Sk] of attention head (b, h); True = kept."""
    if p == 0.0:
        return np.ones((Sq, Sk), dtype=bool)
    n_first = ((b * H + h) * Sq) * Sk
    u = uniform_words(n_first, Sq * Sk, seed, offset).reshape(Sq, Sk)
    return u >= np.uint32(keep_threshold(p))


def keep_mask(B, H, Sq, Sk, p, seed, offset):
    """Boolean keep mask [B, H, Sq, Sk] for the whole problem."""
    m = np.empty((B, H, Sq, Sk), dtype=bool)
    for b in range(B):
        for h in range(H):
            m[b, h] = keep_mask_head(b, h, H, Sq, Sk, p, seed, offset)
    return m

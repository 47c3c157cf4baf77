"""Philox4x32-10 counter-based generator (oracle side; test infrastructure only).

Written from its published definition: J. K. Salmon, M. A. Moraes,
R. O. Dror, D. E. Shaw, "Parallel random numbers: as easy as 1, 2, 3"
(SC'11).  Ten rounds; each round multiplies counter words 0 and 2 by the
two Philox multipliers, mixes the high halves with words 1/3 and the key,
and the key advances by the two Weyl increments between rounds.

The pages name no generator; the rejection rule needs uniforms, drawn here
per decision from a counter so that the CUDA path (which implements the same
published generator separately) draws the identical numbers:

* accept draw for child node c of sequence b at step t:
  counter (c, 0, b, t), key (seed_lo, seed_hi), word 0;
* race draw for token x when sampling at stop node v:
  counter (x div 4, 256 + v, b, t), same key, word x mod 4 (one call of
  the generator serves four consecutive tokens).

A 32-bit word w maps to u = (w >> 8) * 2^-24 in [0, 1) (exact in float32);
for the race the open-interval form u' = ((w >> 9) + 0.5) * 2^-23 is used
(exact in float32, never 0 or 1).
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Vectorised over numpy uint arrays: ctr = (c0,c1,c2,c3), key = (k0,k1).
    Returns four uint32 arrays."""
    c0, c1, c2, c3 = (np.asarray(c, np.uint64) & MASK32 for c in ctr)
    k0, k1 = (np.asarray(k, np.uint64) & MASK32 for k in key)
    for r in range(10):
        if r:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = np.uint64(M0) * c0
        p1 = np.uint64(M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return tuple(np.asarray(c, np.uint64).astype(np.uint32) for c in (c0, c1, c2, c3))


def _key(seed: int):
    return (seed & MASK32, (seed >> 32) & MASK32)


def uniform_accept(seed: int, b: int, step: int, child):
    """u in [0,1) for the accept test of child node(s) ``child``."""
    w = philox4x32_10((child, 0, b, step), _key(seed))[0]
    return (w >> np.uint32(8)).astype(np.float64) * 2.0 ** -24


def uniform_race(seed: int, b: int, step: int, node: int, tokens):
    """u' in (0,1) for the sampling race over ``tokens`` at stop node ``node``."""
    t = np.asarray(tokens, np.int64)
    words = philox4x32_10((t >> 2, 256 + node, b, step), _key(seed))
    w = np.choose(t & 3, words)
    return ((w >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23

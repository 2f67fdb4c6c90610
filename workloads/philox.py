"""Philox4x32-10 counter-based generator, written from its published description.

Source: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3", SC'11 -- the Philox-4x32 bijection with ten
rounds.  Each round multiplies counter words 0 and 2 by two fixed odd 32-bit
multipliers, keeps the 64-bit products' high and low halves, and permutes and
xors them with the other counter words and the round key; the two-word key is
bumped by two Weyl constants between rounds.

This module is input synthesis only: it turns a seed into the uniforms that the
verify-and-sample epilogue consumes as data.  It holds none of the epilogue's
arithmetic.  The pages fix that sampling is seeded (mlx-dspark changelog v0.1.0
"OpenAI-compatible API server": a ``seed`` request parameter) but not the
generator; Philox keyed by seed, request and position is this library's choice.
"""
from __future__ import annotations

import numpy as np

PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter, key):
    """Apply the 10-round Philox-4x32 bijection.

    counter: uint32-valued array of shape [..., 4]; key: [..., 2] (broadcastable).
    Returns uint32 array [..., 4].
    """
    c = np.asarray(counter, dtype=np.uint64) & _MASK32
    k = np.asarray(key, dtype=np.uint64) & _MASK32
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0 = np.broadcast_to(k[..., 0], c0.shape).copy()
    k1 = np.broadcast_to(k[..., 1], c0.shape).copy()
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + PHILOX_W0) & _MASK32
            k1 = (k1 + PHILOX_W1) & _MASK32
        p0 = PHILOX_M0 * c0          # < 2^64, exact in uint64
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniforms_from_words(words):
    """Map 32-bit words to float32 uniforms in [0, 1): top 24 bits times 2^-24 (exact in fp32)."""
    w = np.asarray(words, dtype=np.uint32)
    return ((w >> np.uint32(8)).astype(np.float64) * (2.0 ** -24)).astype(np.float32)


def epilogue_uniforms(seed: int, B: int, K_max: int) -> np.ndarray:
    """Uniforms [B, K_max+1, 2] float32 for the verify-and-sample epilogue.

    Key = (seed low 32 bits, seed high 32 bits); counter = (position j, request b, 0, 0).
    Word 0 of the output is the accept draw at position j, word 1 the
    resample / bonus draw at position j.
    """
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint64)
    j = np.arange(K_max + 1, dtype=np.uint64)
    b = np.arange(B, dtype=np.uint64)
    ctr = np.zeros((B, K_max + 1, 4), dtype=np.uint64)
    ctr[..., 0] = j[None, :]
    ctr[..., 1] = b[:, None]
    words = philox4x32_10(ctr, key)
    return uniforms_from_words(words[..., :2])

"""Oracle token selection: greedy argmax, top-k with temperature, Philox4x32-10 draws.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the product path.

[LM4] "Temperature and top-k": keep the k best logits (the k-th largest value is the
threshold and every logit below it becomes -inf, so ties with it are kept), take the
temperature softmax, and draw from the result. The page's random source (.NET Random)
and the body of its sampling call are not shown; the reading used here is:

* the uniform u in [0, 1) for step s and batch row b is the first 32-bit word of
  Philox4x32-10 (Salmon, Moraes, Dror & Shaw, "Parallel random numbers: as easy as
  1, 2, 3", SC'11) with key = (seed low word, seed high word) and counter
  (s, b, 0, 0), shifted right by 8 and scaled by 2^-24;
* the pick is the first kept index, in ascending index order, whose running float64 sum of
  exp((l - max) / temperature) exceeds u times the total.

Greedy decoding is top-1: the lowest index among the largest logits.
"""
from __future__ import annotations

import numpy as np

_MASK32 = 0xFFFFFFFF
# Philox4x32 multipliers and Weyl key increments, as published by Salmon et al.
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds on a 4-word counter and a 2-word key (Python ints).

    Each round multiplies words 0 and 2 by the two constants into 64-bit products, then
    the new words are (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0));
    the key is bumped by the Weyl constants between rounds.
    """
    c0, c1, c2, c3 = (int(x) & _MASK32 for x in counter)
    k0, k1 = (int(x) & _MASK32 for x in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + PHILOX_W0) & _MASK32
            k1 = (k1 + PHILOX_W1) & _MASK32
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & _MASK32, p1 & _MASK32, \
                         ((p0 >> 32) ^ c3 ^ k1) & _MASK32, p0 & _MASK32
    return c0, c1, c2, c3


def uniform(seed: int, step: int, row: int) -> float:
    """u in [0, 1) for decode step `step` and batch row `row` (24-bit resolution)."""
    x0 = philox4x32_10((step, row, 0, 0), (seed & _MASK32, (seed >> 32) & _MASK32))[0]
    return (x0 >> 8) * (2.0 ** -24)


def greedy(logits) -> np.ndarray:
    """Index of the largest logit per row; ties go to the lowest index."""
    return np.argmax(np.asarray(logits), axis=-1).astype(np.int32)


def topk_keep(row, k: int) -> np.ndarray:
    """Boolean mask of kept logits: l >= the k-th largest value (ties kept).

    k <= 0 or k >= len(row) keeps everything, as on the page.
    """
    row = np.asarray(row)
    if k <= 0 or k >= row.size:
        return np.ones(row.size, dtype=bool)
    kth = np.sort(row)[::-1][k - 1]
    return row >= kth


def topk_sample(row, k: int, temperature: float, u: float) -> int:
    """The sampled index of one logits row (see the module docstring for the reading)."""
    row = np.asarray(row, dtype=np.float64)
    keep = topk_keep(row, k)
    mx = row[keep].max()
    w = np.where(keep, np.exp((row - mx) / temperature), 0.0)
    total = w.sum()
    csum = 0.0
    for i in np.flatnonzero(keep):
        csum += w[i]
        if csum > u * total:
            return int(i)
    return int(np.flatnonzero(keep)[-1])

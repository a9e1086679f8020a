"""Limited-width accumulation model for FP8 tensor-core sums.  TEST INFRASTRUCTURE ONLY.

The pages report that the FP8 GEMM accumulation of the H800 tensor cores keeps
only about 14 bits, which motivates promoting partial sums to FP32 every 128
elements of K (page 2, inprokorea.com free #735329, accumulation-precision
passage and Figure 6).  They give no mechanism beyond the bit count, so this
model is a reading: products arrive in groups (one MMA instruction's share of
K); each group's exact sum is added to the running accumulator after both
terms are aligned to the larger of their exponents and truncated toward zero
to `bits` significant bits at that exponent.  bits = 53 with any group size
reproduces an exact float64 sum of exactly representable terms.

Parity unpinned: the pages' "about 2% maximum relative error at K = 4096" is
context, not a value this model is fitted to.
"""

from __future__ import annotations

import math

import numpy as np


def _trunc_to(x: float, ulp: float) -> float:
    return math.trunc(x / ulp) * ulp


def aligned_sum(terms, bits: int, group: int = 32) -> float:
    """Sum `terms` (float64, in order) with a `bits`-bit aligned accumulator."""
    acc = 0.0
    t = np.asarray(terms, dtype=np.float64)
    for i in range(0, t.shape[0], group):
        s = float(np.sum(t[i:i + group], dtype=np.float64))   # exact for E4M3 products
        big = max(abs(acc), abs(s))
        if big == 0.0:
            continue
        e = math.frexp(big)[1] - 1                              # floor(log2 big)
        ulp = math.ldexp(1.0, e - bits + 1)
        acc = _trunc_to(acc, ulp) + _trunc_to(s, ulp)
    return acc


def aligned_dot_rows(A, B, bits: int, group: int = 32) -> np.ndarray:
    """C[m, n] = aligned_sum over k of A[m, k] * B[n, k] (A [M, K], B [N, K] float64)."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    out = np.empty((A.shape[0], B.shape[0]))
    for m in range(A.shape[0]):
        prods = A[m][None, :] * B                               # [N, K], exact products
        for n in range(B.shape[0]):
            out[m, n] = aligned_sum(prods[n], bits, group)
    return out

"""Block-scaled FP8 GEMM with per-128-K promotion.  TEST INFRASTRUCTURE ONLY.

Definition (page 2, inprokorea.com free #735329: the promotion passage and
Figure 6, and the per-group-scaling passage): the K dimension is cut into
groups of 128; each group's partial product of the E4M3 operands is formed,
multiplied by that group's activation-tile scale and weight-block scale, and
added into a full-precision accumulator:

    C[m, n] = sum_kb  P_kb[m, n] * sa[m, kb] * sb(n, kb),
    P_kb[m, n] = sum_{k in group kb} decode(A[m, k]) * decode(B[n, k])

with sb(n, kb) = sb[n // 128, kb] for 128x128 weight blocks, or sb[n, kb] when
B also carries 1x128 tiles (the Wgrad case, both operands quantised along the
token dimension; page 5, inprokorea.com free #890463, backward-pass passage).

Exactness: every E4M3 value is an integer multiple of 2^-9 below 2^9 in
magnitude, so 2^18 * P_kb is an integer below 2^43 and any float64 summation
order (BLAS included) gives P_kb exactly.  sa*sb is exact in float64 (24+24
bits).  The only roundings are the float64 products with P_kb and the float64
sum over groups.  Output dtype rounding (BF16 / FP32) is the caller's.
"""

from __future__ import annotations

import numpy as np

from .e4m3 import decode

TILE = 128


def slice_partials(qa, qb) -> np.ndarray:
    """All P_kb at once: float64 [K/128, M, N] (exact)."""
    A = decode(qa)
    B = decode(qb)
    K = A.shape[1]
    nkb = K // TILE
    out = np.empty((nkb, A.shape[0], B.shape[0]), dtype=np.float64)
    for kb in range(nkb):
        sl = slice(kb * TILE, (kb + 1) * TILE)
        out[kb] = A[:, sl] @ B[:, sl].T
    return out


def _b_scale(sb, n_rows: int, kb: int, b_tile: bool) -> np.ndarray:
    sb = np.asarray(sb, dtype=np.float64)
    if b_tile:
        return sb[:, kb]
    return np.repeat(sb[:, kb], TILE)[:n_rows]


def gemm(qa, sa, qb, sb, b_tile: bool = False) -> np.ndarray:
    """float64 C[M, N] for A codes [M, K], B codes [N, K] (both K-major).

    sa: float32 [M, K/128]; sb: float32 [N/128, K/128] (blocks) or [N, K/128]
    (b_tile=True).
    """
    qa = np.asarray(qa)
    qb = np.asarray(qb)
    M, K = qa.shape
    N, Kb = qb.shape
    if K != Kb or K % TILE:
        raise ValueError("bad K")
    A = decode(qa)
    B = decode(qb)
    sa = np.asarray(sa, dtype=np.float64)
    C = np.zeros((M, N), dtype=np.float64)
    for kb in range(K // TILE):
        sl = slice(kb * TILE, (kb + 1) * TILE)
        P = A[:, sl] @ B[:, sl].T
        C += P * (sa[:, kb][:, None] * _b_scale(sb, N, kb, b_tile)[None, :])
    return C


def grouped_gemm(qa, sa, offsets, qb, sb) -> np.ndarray:
    """Per-expert gemm over contiguous row groups.

    qa [T, K], sa [T, K/128]; offsets int [E+1] (non-decreasing, 0..T);
    qb [E, N, K]; sb [E, N/128, K/128].  Rows of expert e are
    offsets[e]..offsets[e+1]-1 and use B[e] only.
    """
    qa = np.asarray(qa)
    off = np.asarray(offsets, dtype=np.int64)
    E = off.shape[0] - 1
    N = qb.shape[1]
    C = np.zeros((qa.shape[0], N), dtype=np.float64)
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            C[r0:r1] = gemm(qa[r0:r1], np.asarray(sa)[r0:r1], qb[e], sb[e])
    return C


def gemm_quant(qa, sa, qb, sb, b_tile: bool = False, pow2: bool = False):
    """The GEMM's FP32 result quantised into 1x128 E4M3 tiles along N.

    This is the output an FP8 producer hands to the next FP8 GEMM: the pages
    cache the inputs of the following Linear as FP8 with per-1x128-tile
    scales (page 2, inprokorea.com free #735329, fine-grained quantisation
    passage; power-of-2 scales for the inputs the page names, pages 1 and 2).
    Reading: the tile is quantised from the float32 rounding of the promoted
    sum C (no BF16 step in between), with the same amax, scale and multiplier
    rules as the activation quantiser.

    Returns (q uint8 [M, N], s float32 [M, N/128], x float32 [M, N]) where x is
    the float32 C that was quantised.
    """
    from .quant import act_quant

    C = gemm(qa, sa, qb, sb, b_tile)
    if C.shape[1] % TILE:
        raise ValueError("N must be a multiple of 128 for 1x128 output tiles")
    x = C.astype(np.float32)                         # RNE from float64
    q, s = act_quant(x, pow2)
    return q, s, x


def silu(g):
    """g * sigmoid(g) = g / (1 + exp(-g)) in float64."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def grouped_swiglu_quant(qa, sa, offsets, qb, sb, pow2: bool = True):
    """Routed up-projection followed by SwiGLU, quantised as the down-projection input.

    qb [E, 2I, K] holds each expert's gate rows (0..I-1) then up rows (I..2I-1);
    with C = grouped_gemm(...) [T, 2I], g = C[:, :I], u = C[:, I:]:
        h = silu(g) * u                      (float64 from the exact sums)
    then h rounded to float32 and quantised into 1x128 tiles along I with
    power-of-2 scales: the down-projection input, which page 2 (inprokorea.com
    free #735329, power-of-2 passage) and page 1 name among the activations
    cached in FP8 with integral power-of-2 scales.  The SwiGLU form and the
    gate/up row order are readings (the pages name neither).

    Returns (q uint8 [T, I], s float32 [T, I/128], h float32 [T, I]).
    """
    from .quant import act_quant

    qb = np.asarray(qb)
    if qb.shape[1] % 256:
        raise ValueError("2I must be a multiple of 256")
    C = grouped_gemm(qa, sa, offsets, qb, sb)
    I = qb.shape[1] // 2
    h = (silu(C[:, :I]) * C[:, I:]).astype(np.float32)
    q, s = act_quant(h, pow2)
    return q, s, h

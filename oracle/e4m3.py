"""E4M3 codec from the bit-field definition.  TEST INFRASTRUCTURE ONLY.

The pages fix the format only as "E4M3 (4-bit exponent and 3-bit mantissa)" on
all tensors (page 2, inprokorea.com free #735329, passage contrasting the
hybrid E4M3/E5M2 format).  Reading used here (the FN variant): 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits; no infinities; the only NaN
codes are S.1111.111, so the largest finite magnitude is 1.75 * 2^8 = 448;
subnormals are m * 2^-9.  Encoding rounds to nearest, ties to even, and
saturates magnitudes beyond 448 to 448 (sign kept, -0 -> 0x80).
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6       # smallest normal binade: 2^-6
_MANT_BITS = 3


def decode(codes) -> np.ndarray:
    """Codes (uint8 array) -> float64 values; NaN codes give NaN."""
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m.astype(np.float64) * 2.0 ** (_MIN_NORMAL_EXP - _MANT_BITS)
    norm = (1.0 + m / 8.0) * np.ldexp(1.0, e - 7)
    val = np.where(e == 0, sub, norm)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return np.where(sign == 1, -val, val)


def encode(x) -> np.ndarray:
    """float32 values -> uint8 codes (RNE, satfinite, sign of zero kept).

    The input is first taken as float32 (the only width the path rounds from);
    the rounding itself is done exactly in float64: the value is divided by the
    quantum of its binade (a power of two, so exact), rounded half-to-even to an
    integer, and multiplied back.
    """
    x = np.asarray(x, dtype=np.float32)
    neg = np.signbit(x)
    a = np.abs(x).astype(np.float64)
    nan = np.isnan(a)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(np.where(np.isfinite(a), a, 1.0))
        binade = np.maximum(e - 1, _MIN_NORMAL_EXP)          # floor(log2 a), clamped
        quantum = np.ldexp(1.0, binade - _MANT_BITS)
        r = np.rint(np.where(np.isfinite(a), a, 0.0) / quantum)  # ties to even
        v = r * quantum
        v = np.where(np.isinf(a), E4M3_MAX, v)
        v = np.minimum(v, E4M3_MAX)                            # satfinite
    sub = v < 2.0 ** _MIN_NORMAL_EXP
    code_sub = np.rint(v / 2.0 ** (_MIN_NORMAL_EXP - _MANT_BITS)).astype(np.int64)
    mv, ev = np.frexp(np.where(sub, 1.0, v))                  # v = mv * 2^ev, mv in [0.5,1)
    mant = np.rint((mv * 2.0 - 1.0) * 8.0).astype(np.int64)
    code_norm = ((ev - 1 + 7) << 3) | mant
    code = np.where(sub, code_sub, code_norm) | (neg.astype(np.int64) << 7)
    code = np.where(nan, 0x7F | (neg.astype(np.int64) << 7), code)
    return code.astype(np.uint8)

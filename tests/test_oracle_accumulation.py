"""Pins for the limited-width accumulation model (CPU only).

The model (oracle/accumulation.py) reads the pages' "about 14 bits" statement
(page 2, inprokorea.com free #735329, accumulation-precision passage) as
aligned truncation per MMA group.  Pinned by closed forms: full width is an
exact sum; terms below the accumulator's last kept bit vanish; terms at it are
kept; the error never exceeds one truncation step per group.
"""

import math

import numpy as np
import pytest

from oracle import accumulation as acc
from oracle import e4m3


def test_full_width_is_exact_for_e4m3_products():
    g = np.random.default_rng(0)
    a = e4m3.decode(g.integers(0, 0x7E, 4096).astype(np.uint8))
    b = e4m3.decode(g.integers(0, 0x7E, 4096).astype(np.uint8))
    p = a * b                                       # exact in float64
    exact = sum(int(round(x * 2 ** 18)) for x in p) / 2 ** 18
    for group in (1, 4, 32):
        assert acc.aligned_sum(p, bits=53, group=group) == exact


@pytest.mark.parametrize("bits", [8, 14, 22])
def test_terms_below_the_kept_bit_vanish(bits):
    # accumulator 1.0 keeps bits down to 2^(1-bits); adding 2^-bits n times (one
    # term per group) changes nothing, while 2^(1-bits) terms are all kept
    tiny = [1.0] + [2.0 ** -bits] * 1000
    assert acc.aligned_sum(tiny, bits=bits, group=1) == 1.0
    kept = [1.0] + [2.0 ** (1 - bits)] * 10
    assert acc.aligned_sum(kept, bits=bits, group=1) == 1.0 + 10 * 2.0 ** (1 - bits)


def test_group_sums_are_exact_before_alignment():
    # within one group the small terms add up exactly and survive together
    bits = 8
    terms = [1.0] + [2.0 ** -bits] * 31
    assert acc.aligned_sum(terms, bits=bits, group=32) == 1.0 + 31 * 2.0 ** -bits - (
        (31 * 2.0 ** -bits) % 2.0 ** (1 - bits))


@pytest.mark.parametrize("bits", [10, 14, 18])
def test_error_bounded_by_one_step_per_group(bits):
    g = np.random.default_rng(bits)
    p = g.standard_normal(4096)
    exact = math.fsum(p)
    got = acc.aligned_sum(p, bits=bits, group=32)
    # each of the 128 additions truncates both terms by less than one ulp of the
    # larger magnitude seen so far
    big = max(abs(math.fsum(p[:i])) for i in range(32, 4097, 32))
    big = max(big, max(abs(math.fsum(p[i:i + 32])) for i in range(0, 4096, 32)))
    assert abs(got - exact) <= 128 * 2 * 2.0 ** (math.frexp(big)[1] - bits)


def test_fewer_bits_give_larger_error():
    g = np.random.default_rng(5)
    A = e4m3.decode(g.integers(0, 0x7E, (4, 2048)).astype(np.uint8)) * np.where(
        g.random((4, 2048)) < 0.5, -1, 1)
    B = e4m3.decode(g.integers(0, 0x7E, (4, 2048)).astype(np.uint8))
    exact = A @ B.T
    errs = [np.abs(acc.aligned_dot_rows(A, B, bits) - exact).max() for bits in (10, 14, 20, 53)]
    assert errs[0] >= errs[1] >= errs[2] >= errs[3] == 0.0
    assert errs[0] > errs[2]

"""Pins for the oracle's E4M3 codec (CPU only).

The format facts come from the E4M3 definition (4 exponent bits, bias 7,
3 mantissa bits, FN variant: no infinities, NaN = S.1111.111), which the
pages name for every tensor (page 2, inprokorea.com free #735329, passage
contrasting the hybrid E4M3/E5M2 format).  The rounding facts are checked
against two independent library casts.
"""

import ml_dtypes
import numpy as np
import pytest
import torch

from oracle import e4m3

ALL = np.arange(256, dtype=np.uint8)
FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def test_decode_fixed_points():
    # (code, value) pairs written from the bit-field definition by hand
    table = {
        0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
        0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x78: 256.0,
        0x7E: 448.0, 0x81: -(2.0 ** -9), 0xB8: -1.0, 0xFE: -448.0,
    }
    for c, v in table.items():
        assert e4m3.decode(np.uint8(c)) == v, hex(c)
    assert np.signbit(e4m3.decode(np.uint8(0x80)))
    assert np.isnan(e4m3.decode(np.uint8(0x7F))) and np.isnan(e4m3.decode(np.uint8(0xFF)))
    assert np.nanmax(e4m3.decode(ALL)) == e4m3.E4M3_MAX == 448.0
    assert np.sum(np.isnan(e4m3.decode(ALL))) == 2


def test_decode_matches_library_on_all_codes():
    ours = e4m3.decode(ALL)
    lib = ALL.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(ours[ok], lib[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(lib[ok]))
    tl = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(ours[ok], tl[ok])


def test_roundtrip_every_finite_code():
    assert np.array_equal(e4m3.encode(e4m3.decode(FINITE).astype(np.float32)), FINITE)


def test_monotone():
    pos = np.arange(0, 0x7F, dtype=np.uint8)
    v = e4m3.decode(pos)
    assert np.all(np.diff(v) > 0)


def test_midpoints_tie_to_even_and_neighbours_round_to_nearest():
    pos = np.arange(0, 0x7E, dtype=np.uint8)           # pairs (c, c+1), c+1 <= 0x7E
    lo = e4m3.decode(pos)
    hi = e4m3.decode(pos + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)   # exact in float32
    got = e4m3.encode(mid)
    even = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    assert np.array_equal(got, even)
    below = np.nextafter(mid, np.float32(0))
    above = np.nextafter(mid, np.float32(np.inf))
    assert np.array_equal(e4m3.encode(below), pos)
    assert np.array_equal(e4m3.encode(above), (pos + 1).astype(np.uint8))
    assert np.array_equal(e4m3.encode(-mid), even | 0x80)


def test_saturation_and_specials():
    big = np.array([448.0, 448.5, 463.9, 464.0, 480.0, 1e6, 3.0e38, np.inf], np.float32)
    assert np.all(e4m3.encode(big) == 0x7E)
    assert np.all(e4m3.encode(-big) == 0xFE)
    assert e4m3.encode(np.float32(-0.0)) == 0x80
    assert e4m3.encode(np.float32(0.0)) == 0x00
    assert (e4m3.encode(np.float32(np.nan)) & 0x7F) == 0x7F
    # below half the smallest subnormal -> zero; exactly half -> ties to even (zero)
    assert e4m3.encode(np.float32(2.0 ** -10)) == 0x00
    assert e4m3.encode(np.float32(np.nextafter(np.float32(2.0 ** -10), np.float32(1)))) == 0x01
    assert e4m3.encode(np.float32(3 * 2.0 ** -10)) == 0x02        # 1.5 ulp -> 2 (even)


def _sweep_patterns():
    """Every float32 whose upper 20 bits vary, with 6 choices of the low 12 bits.

    The E4M3 rounding bit of a normal result is float32 mantissa bit 19 and
    every lower bit is sticky, so this covers ties, sticky cases and every
    binade (float32 subnormals through the saturation range).
    """
    hi = np.arange(1 << 20, dtype=np.uint32) << 12
    lows = np.array([0x000, 0x001, 0x7FF, 0x800, 0x801, 0xFFF], np.uint32)
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    return np.clip(x, -448.0, 448.0).astype(np.float32)   # library casts do not saturate


def test_sweep_against_ml_dtypes():
    x = _sweep_patterns()
    ours = e4m3.encode(x)
    lib = x.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    bad = np.nonzero(ours != lib)[0]
    assert bad.size == 0, (x[bad[:5]], ours[bad[:5]], lib[bad[:5]])


def test_sweep_against_torch():
    x = _sweep_patterns()
    ours = e4m3.encode(x)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)


@pytest.mark.parametrize("seed", [0, 1])
def test_random_values_against_library(seed):
    g = np.random.default_rng(seed)
    x = (g.standard_normal(200_000) * np.exp(g.uniform(-25, 8, 200_000))).astype(np.float32)
    x = np.clip(x, -448, 448).astype(np.float32)
    assert np.array_equal(e4m3.encode(x), x.astype(ml_dtypes.float8_e4m3fn).view(np.uint8))

"""Pins for the oracle's fine-grained quantisers (CPU only).

What the pages fix: 1x128 activation tiles and 128x128 weight blocks
(page 1, xn--9g3bo1gtkw0l8ubf92bgle.kr qna #85187, Figure 7 (a)); an online
amax per tile/block and per-group scales (page 2, inprokorea.com free
#735329); power-of-2 scales for some activations (pages 1 and 2); 128x1 tiles
for the backward re-quantisation (page 5, inprokorea.com free #890463).
What mathematics fixes: the tile amax lands on the E4M3 maximum; the
round-trip error is at most half an E4M3 step times the scale.
"""

import os

import numpy as np
import pytest

import oracle
from oracle import e4m3
from oracle import quant as oq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "act_tile_worked.txt")


def _rand(shape, seed, heavy=True):
    g = np.random.default_rng(seed)
    x = g.standard_normal(shape).astype(np.float32)
    if heavy:
        x *= np.exp(g.uniform(-30, 30, shape)).astype(np.float32)
        x[g.random(shape) < 0.01] = 0.0
    return x.astype(np.float32)


def _f32_bits(v):
    return int(np.array([v], np.float32).view(np.uint32)[0])


def test_worked_tile_fixture():
    x = np.arange(128, dtype=np.float32)
    x[127] = -256.0
    scales, codes = {}, []
    for line in open(GOLDEN):
        p = line.split("#")[0].split()
        if not p:
            continue
        if p[0] == "scale":
            scales[p[1]] = int(p[2], 16)
        elif p[0] == "code":
            codes.append((p[1], int(p[2]), int(p[3], 16)))
    for mode, pow2 in (("default", False), ("pow2", True)):
        q, s = oracle.act_quant(x[None, :], pow2=pow2)
        assert _f32_bits(s[0, 0]) == scales[mode]
        for m, i, c in codes:
            if m == mode:
                assert q[0, i] == c, (mode, i, hex(q[0, i]), hex(c))
    assert len(codes) >= 20


def test_amax_maps_to_e4m3_max():
    x = _rand((37, 1024), 1)
    q, s = oracle.act_quant(x)
    d = np.abs(e4m3.decode(q)).reshape(37, 8, 128).max(axis=2)
    nz = np.abs(x).reshape(37, 8, 128).max(axis=2) > 0
    assert np.all(d[nz] == 448.0)
    assert np.all(d[~nz] == 0.0)


def test_scale_is_amax_over_448_in_float32():
    x = _rand((9, 512), 2)
    _, s = oracle.act_quant(x)
    amax = np.abs(x).reshape(9, 4, 128).max(axis=2)
    expect = (np.maximum(amax, np.float32(2.0 ** -64)) / np.float32(448)).astype(np.float32)
    assert np.array_equal(s, expect)


def test_pow2_rule():
    x = _rand((21, 768), 3)
    q, s = oracle.act_quant(x, pow2=True)
    mant, _ = np.frexp(s.astype(np.float64))
    assert np.all(mant == 0.5)                               # exact powers of two
    amax = np.abs(x).reshape(21, 6, 128).max(axis=2).astype(np.float64)
    a = np.maximum(amax, 2.0 ** -64)
    # smallest power of two that is >= fl32(a/448)
    t = (a.astype(np.float32) / np.float32(448)).astype(np.float64)
    assert np.all(s >= t) and np.all(s < 2 * t)
    nz = amax > 0
    y = a / s                                  # the tile amax after scaling, exact
    assert np.all(y[nz] > 224.0) and np.all(y[nz] <= 448.0 * (1 + 2.0 ** -22))
    # after E4M3 rounding (step 16 in [128, 256)) the top code lies in [224, 448]
    d = np.abs(e4m3.decode(q)).reshape(21, 6, 128).max(axis=2)
    assert np.all(d[nz] >= 224.0) and np.all(d[nz] <= 448.0)


def _check_error_bound(x, xhat, s_full):
    err = np.abs(x.astype(np.float64) - xhat)
    bound = (2.0 ** -4 * np.abs(x.astype(np.float64)) + 2.0 ** -10 * s_full) * (1 + 2.0 ** -16)
    assert np.all(err <= bound)
    # coarse form: one half E4M3 step of the top binade (16) times the scale
    assert np.all(err <= 16.0 * s_full * (1 + 2.0 ** -16))


@pytest.mark.parametrize("pow2", [False, True])
def test_act_roundtrip_error_bound(pow2):
    x = _rand((33, 640), 4)
    q, s = oracle.act_quant(x, pow2=pow2)
    xhat = oracle.dequant_tiles(q, s)
    sf = np.repeat(s.astype(np.float64), 128, axis=1)
    _check_error_bound(x, xhat, sf)
    amax = np.repeat(np.abs(x).reshape(33, 5, 128).max(axis=2), 128, axis=1).astype(np.float64)
    if not pow2:   # tile amax / 28 is the familiar "E4M3 ulp x amax" form
        assert np.all(np.abs(x - xhat) <= amax / 28 * (1 + 2.0 ** -16))


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_roundtrip_error_bound(pow2):
    w = _rand((256, 384), 5)
    q, s = oracle.weight_quant(w, pow2=pow2)
    assert s.shape == (2, 3)
    xhat = oracle.dequant_blocks(q, s)
    sf = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)
    _check_error_bound(w, xhat, sf)


def test_weight_block_amax_and_transpose():
    w = _rand((384, 256), 6)
    q, s, qt, st = oracle.weight_quant(w, transposed=True)
    blk = np.abs(w).reshape(3, 128, 2, 128).max(axis=(1, 3))
    assert np.array_equal(s, (np.maximum(blk, np.float32(2.0 ** -64)) / np.float32(448)).astype(np.float32))
    assert np.array_equal(qt, q.T) and np.array_equal(st, s.T)
    d = np.abs(e4m3.decode(q)).reshape(3, 128, 2, 128).max(axis=(1, 3))
    assert np.all(d[blk > 0] == 448.0)


def test_weight_block_is_not_row_tiles():
    # a block shares one scale across its 128 rows: a row of small values in a
    # block with a large outlier must get the outlier's scale
    w = np.full((128, 128), 0.5, np.float32)
    w[7, 9] = 1000.0
    q, s = oracle.weight_quant(w)
    assert s.shape == (1, 1) and s[0, 0] == np.float32(1000.0) / np.float32(448)
    qa, sa = oracle.act_quant(w)
    assert sa[0, 0] == np.float32(0.5) / np.float32(448)
    assert not np.array_equal(q, qa)


@pytest.mark.parametrize("pow2", [False, True])
def test_transposed_mode_equals_quantising_the_transpose(pow2):
    x = _rand((256, 384), 7)
    qt, st = oracle.act_quant_t(x, pow2=pow2)
    q2, s2 = oracle.act_quant(np.ascontiguousarray(x.T), pow2=pow2)
    assert qt.shape == (384, 256) and st.shape == (384, 2)
    assert np.array_equal(qt, q2) and np.array_equal(st, s2)


def test_pow2_idempotent():
    x = _rand((5, 256), 8, heavy=False)
    q, s = oracle.act_quant(x, pow2=True)
    xhat = oracle.dequant_tiles(q, s).astype(np.float32)     # exact: codes x 2^k
    q2, s2 = oracle.act_quant(xhat, pow2=True)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)


def test_zero_and_signed_zero_tiles():
    x = np.zeros((2, 128), np.float32)
    x[1] = -0.0
    q, s = oracle.act_quant(x)
    assert np.all(q[0] == 0x00) and np.all(q[1] == 0x80)
    # floor 2^-64: s = fl32(2^-64/448) = fl32(2^-70 / 7); 8/7 mantissa 0x124925, exponent -73
    assert _f32_bits(s[0, 0]) == 0x1B124925


def test_ragged_rows():
    for M in (1, 3, 129):
        x = _rand((M, 256), 9 + M)
        q, s = oracle.act_quant(x)
        assert q.shape == (M, 256) and s.shape == (M, 2)
        q1, s1 = oracle.act_quant(x[-1:])
        assert np.array_equal(q[-1:], q1) and np.array_equal(s[-1:], s1)


def test_bad_shapes_rejected():
    with pytest.raises(ValueError):
        oracle.act_quant(np.zeros((2, 100), np.float32))
    with pytest.raises(ValueError):
        oracle.act_quant_t(np.zeros((100, 128), np.float32))
    with pytest.raises(ValueError):
        oracle.weight_quant(np.zeros((100, 128), np.float32))


def test_planted_mistakes_are_caught(monkeypatch):
    """A wrong quantum or a dropped floor in the oracle must trip a pin above."""
    x = np.arange(128, dtype=np.float32)
    x[127] = -256.0
    real = oq.scale_from_amax

    def off_by_one(amax, pow2=False):      # 447 instead of 448
        a = np.maximum(np.asarray(amax, np.float32), oq.AMAX_FLOOR)
        return (a / np.float32(447)).astype(np.float32), (np.float32(447) / a).astype(np.float32)

    monkeypatch.setattr(oq, "scale_from_amax", off_by_one)
    with pytest.raises(AssertionError):
        test_worked_tile_fixture()
    monkeypatch.setattr(oq, "scale_from_amax", real)

    def pow2_round_down(amax, pow2=False):
        s, m = real(amax, pow2=False)
        mt, et = np.frexp(s.astype(np.float64))
        return np.ldexp(1.0, et - 1).astype(np.float32), np.ldexp(1.0, 1 - et).astype(np.float32)

    monkeypatch.setattr(oq, "scale_from_amax", lambda a, pow2=False: pow2_round_down(a) if pow2 else real(a))
    with pytest.raises(AssertionError):
        test_pow2_rule()


# ---------------------------------------------------------------- backward re-quantisation
REQUANT_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "requant_t_worked.txt")


def _requant_fixture_input():
    q = np.empty((128, 256), np.uint8)
    q[:, :128] = 0x38
    q[:, 128::2] = 0x3C
    q[:, 129::2] = 0xBC
    s = np.empty((128, 2), np.float32)
    s[:, 0] = 2.0 ** (np.arange(128) % 8)
    s[:, 1] = 0.25
    return q, s


def test_requant_worked_block():
    q, s = _requant_fixture_input()
    scales, codes = {}, {}
    for line in open(REQUANT_GOLDEN):
        f = line.split("#")[0].split()
        if not f:
            continue
        if f[0] == "scale":
            scales[(f[1], int(f[2]))] = int(f[3], 16)
        else:
            codes[(f[1], int(f[2]), int(f[3]))] = int(f[4], 16)
    for mode in ("default", "pow2"):
        qt, st = oracle.requant_t(q, s, pow2=(mode == "pow2"))
        assert qt.shape == (256, 128) and st.shape == (256, 1)
        stb = st.view(np.uint32)
        assert (stb[:128, 0] == scales[(mode, 0)]).all()
        assert (stb[128:, 0] == scales[(mode, 1)]).all()
        for r in range(128):
            assert (qt[:128, r] == codes[(mode, 0, r % 8)]).all(), (mode, r)
        assert (qt[128::2, :] == codes[(mode, 1, 0)]).all()
        assert (qt[129::2, :] == codes[(mode, 1, 1)]).all()


@pytest.mark.parametrize("pow2", [False, True])
def test_requant_two_step_error_bound(pow2):
    # quantise 1x128, then re-quantise 128x1: each step is within half an E4M3
    # step of its input (relative 2^-4 for normal codes, 2^-10 * s below 2^-6),
    # so the composition is within the sum of the two bounds
    x = _rand((256, 384), 21, heavy=False)
    q, s = oracle.act_quant(x)
    qt, st = oracle.requant_t(q, s, pow2=pow2)
    x1 = oracle.dequant_tiles(q, s)                       # after the first step
    x2 = (e4m3.decode(qt) * np.repeat(st.astype(np.float64), 128, axis=1)).T
    s1 = np.repeat(s.astype(np.float64), 128, axis=1)
    s2 = np.repeat(st.astype(np.float64), 128, axis=1).T
    b1 = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s1) * (1 + 2.0 ** -20)
    b2 = np.maximum(2.0 ** -4 * np.abs(x1), 2.0 ** -10 * s2) * (1 + 2.0 ** -20)
    assert (np.abs(x2 - x) <= b1 + b2).all()


def test_requant_uses_the_right_row_scale():
    # every row has its own scale: a transposed or shared scale index would
    # give a different column amax and different codes
    g = np.random.default_rng(4)
    q = e4m3.encode(g.standard_normal((256, 128)).astype(np.float32) * 40)
    s = np.exp(g.uniform(-5, 5, (256, 1))).astype(np.float32)
    qt, st = oracle.requant_t(q, s)
    x = (e4m3.decode(q) * s.astype(np.float64)).astype(np.float32)
    # the 128x1 tile amax of column k over rows 0..127 is max_r |x[r, k]|
    amax = np.max(np.abs(x[:128]), axis=0).astype(np.float32)
    assert np.array_equal(st[:, 0], (amax / np.float32(448)).astype(np.float32))


def test_requant_rejects_ragged_rows():
    with pytest.raises(ValueError):
        oracle.requant_t(np.zeros((100, 128), np.uint8), np.ones((100, 1), np.float32))

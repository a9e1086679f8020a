"""Pins for the oracle's block-scaled GEMM and grouped GEMM (CPU only).

The definition (page 2, inprokorea.com free #735329, promotion passage and
Figure 6; per-group scaling passage): partial products over each 128-wide K
group are scaled by that group's activation and weight scales and accumulated
at full precision.  Pinned here by exact rational brute force, by an int64
restatement of the partial sums, and by special cases that reduce to a
library matmul.
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import e4m3
from oracle import scaled_gemm as og

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def _codes(shape, g):
    return g.choice(FINITE, size=shape)


def _scales(shape, g):
    return np.exp(g.uniform(-20, 20, shape)).astype(np.float32)


def _exact(qa, sa, qb, sb, b_tile):
    """C as exact rationals: sum over groups of (sum of products) * sa * sb."""
    M, K = qa.shape
    N = qb.shape[0]
    A = [[Fraction(float(v)) for v in row] for row in e4m3.decode(qa)]
    B = [[Fraction(float(v)) for v in row] for row in e4m3.decode(qb)]
    C = [[Fraction(0)] * N for _ in range(M)]
    mag = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            tot = 0.0
            for kb in range(K // 128):
                p = sum(A[m][k] * B[n][k] for k in range(kb * 128, kb * 128 + 128))
                sbv = sb[n, kb] if b_tile else sb[n // 128, kb]
                term = p * Fraction(float(sa[m, kb])) * Fraction(float(sbv))
                acc += term
                tot += abs(float(term))
            C[m][n] = acc
            mag[m, n] = tot
    return C, mag


@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (2, 3, 128), (3, 2, 256), (3, 3, 384)])
@pytest.mark.parametrize("b_tile", [False, True])
def test_bruteforce_rational(M, N, K, b_tile):
    g = np.random.default_rng(M * 100 + N * 10 + K + b_tile)
    qa, qb = _codes((M, K), g), _codes((N, K), g)
    sa = _scales((M, K // 128), g)
    sb = _scales((N, K // 128) if b_tile else ((N + 127) // 128, K // 128), g)
    C = oracle.gemm(qa, sa, qb, sb, b_tile=b_tile)
    exact, mag = _exact(qa, sa, qb, sb, b_tile)
    for m in range(M):
        for n in range(N):
            err = abs(Fraction(float(C[m, n])) - exact[m][n])
            assert float(err) <= 2.0 ** -50 * mag[m, n], (m, n)


def test_slice_partials_are_exact_integers():
    g = np.random.default_rng(11)
    qa, qb = _codes((17, 512), g), _codes((9, 512), g)
    P = og.slice_partials(qa, qb)
    ia = np.rint(e4m3.decode(qa) * 512).astype(np.int64)      # codes are multiples of 2^-9
    ib = np.rint(e4m3.decode(qb) * 512).astype(np.int64)
    for kb in range(4):
        sl = slice(kb * 128, kb * 128 + 128)
        ref = ia[:, sl] @ ib[:, sl].T                          # int64, |.| < 2^43
        assert np.array_equal(P[kb] * 2.0 ** 18, ref.astype(np.float64))
        assert np.all(np.abs(ref) < 2 ** 43)


def test_unit_scales_small_integers_reduce_to_int_matmul():
    g = np.random.default_rng(12)
    ints = g.integers(-16, 17, size=(40, 384))
    intsb = g.integers(-16, 17, size=(256, 384))
    qa = e4m3.encode(ints.astype(np.float32))                  # |i| <= 16 is exact in E4M3
    qb = e4m3.encode(intsb.astype(np.float32))
    assert np.array_equal(e4m3.decode(qa), ints)
    C = oracle.gemm(qa, np.ones((40, 3), np.float32), qb, np.ones((2, 3), np.float32))
    assert np.array_equal(C, (ints @ intsb.T).astype(np.float64))


def test_single_group_equals_dequantised_matmul():
    g = np.random.default_rng(13)
    x = g.standard_normal((50, 128)).astype(np.float32)
    w = (g.standard_normal((256, 128)) * 0.02).astype(np.float32)
    qa, sa = oracle.act_quant(x)
    qb, sb = oracle.weight_quant(w)
    C = oracle.gemm(qa, sa, qb, sb)
    ref = oracle.dequant_tiles(qa, sa) @ oracle.dequant_blocks(qb, sb).T
    np.testing.assert_allclose(C, ref, rtol=1e-13, atol=1e-13 * np.abs(ref).max())


def test_multi_group_equals_dequantised_matmul_to_rounding():
    g = np.random.default_rng(14)
    x = g.standard_normal((64, 1024)).astype(np.float32)
    w = g.standard_normal((128, 1024)).astype(np.float32)
    qa, sa = oracle.act_quant(x)
    qb, sb = oracle.weight_quant(w)
    C = oracle.gemm(qa, sa, qb, sb)
    ref = oracle.dequant_tiles(qa, sa) @ oracle.dequant_blocks(qb, sb).T
    assert np.linalg.norm(C - ref) <= 1e-13 * np.linalg.norm(ref)
    # and the quantised product tracks the unquantised one at E4M3 accuracy
    full = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.linalg.norm(C - full) / np.linalg.norm(full) < 0.05


def test_power_of_two_scale_is_linear_and_exact():
    g = np.random.default_rng(15)
    qa, qb = _codes((6, 256), g), _codes((128, 256), g)
    sa, sb = _scales((6, 2), g), _scales((1, 2), g)
    C = oracle.gemm(qa, sa, qb, sb)
    sa2 = sa.copy()
    sa2[3] *= 2
    C2 = oracle.gemm(qa, sa2, qb, sb)
    assert np.array_equal(C2[3], 2 * C[3])
    assert np.array_equal(np.delete(C2, 3, 0), np.delete(C, 3, 0))


def test_block_mode_equals_tile_mode_with_repeated_scales():
    g = np.random.default_rng(16)
    qa, qb = _codes((5, 384), g), _codes((256, 384), g)
    sa, sb = _scales((5, 3), g), _scales((2, 3), g)
    Cb = oracle.gemm(qa, sa, qb, sb)
    Ct = oracle.gemm(qa, sa, qb, np.repeat(sb, 128, axis=0), b_tile=True)
    assert np.array_equal(Cb, Ct)


def test_wgrad_transpose_identity():
    # tile x tile scaling is symmetric: (A B^T)^T == B A^T exactly
    g = np.random.default_rng(17)
    qa, qb = _codes((7, 256), g), _codes((11, 256), g)
    sa, sb = _scales((7, 2), g), _scales((11, 2), g)
    assert np.array_equal(oracle.gemm(qa, sa, qb, sb, b_tile=True).T,
                          oracle.gemm(qb, sb, qa, sa, b_tile=True))


def test_dgrad_via_transposed_weight_codes():
    # Dgrad uses W^T's codes/scales (exact transposes of the block quantisation)
    g = np.random.default_rng(18)
    dy = g.standard_normal((8, 256)).astype(np.float32)
    w = g.standard_normal((256, 384)).astype(np.float32)       # [N_out, K_in]
    qw, sw, qwt, swt = oracle.weight_quant(w, transposed=True)
    qd, sd = oracle.act_quant(dy)
    C = oracle.gemm(qd, sd, qwt, swt)                         # dX = dY . W  ([8, 384])
    ref = oracle.dequant_tiles(qd, sd) @ oracle.dequant_blocks(qw, sw)
    assert np.linalg.norm(C - ref) <= 1e-13 * np.linalg.norm(ref)


def test_grouped_single_expert_equals_dense():
    g = np.random.default_rng(19)
    qa, qb = _codes((40, 256), g), _codes((1, 128, 256), g)
    sa, sb = _scales((40, 2), g), _scales((1, 1, 2), g)
    C = oracle.grouped_gemm(qa, sa, np.array([0, 40]), qb, sb)
    assert np.array_equal(C, oracle.gemm(qa, sa, qb[0], sb[0]))


def test_grouped_empty_experts_and_relabelling():
    g = np.random.default_rng(20)
    sizes = [3, 0, 5, 0, 1]
    off = np.concatenate([[0], np.cumsum(sizes)])
    T = off[-1]
    qa, sa = _codes((T, 256), g), _scales((T, 2), g)
    qb, sb = _codes((5, 128, 256), g), _scales((5, 1, 2), g)
    C = oracle.grouped_gemm(qa, sa, off, qb, sb)
    for e in range(5):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            assert np.array_equal(C[r0:r1], oracle.gemm(qa[r0:r1], sa[r0:r1], qb[e], sb[e]))
    # relabel experts: reverse their order and move their rows with them
    perm = [4, 3, 2, 1, 0]
    rows = np.concatenate([np.arange(off[e], off[e + 1]) for e in perm]).astype(int)
    off2 = np.concatenate([[0], np.cumsum([sizes[e] for e in perm])])
    C2 = oracle.grouped_gemm(qa[rows], sa[rows], off2, qb[perm], sb[perm])
    assert np.array_equal(C2, C[rows])


def test_grouped_bruteforce_rational():
    g = np.random.default_rng(21)
    off = np.array([0, 2, 2, 3])
    qa, sa = _codes((3, 128), g), _scales((3, 1), g)
    qb, sb = _codes((3, 2, 128), g), _scales((3, 1, 1), g)
    C = oracle.grouped_gemm(qa, sa, off, qb, sb)
    for e in range(3):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        ex, mag = _exact(qa[r0:r1], sa[r0:r1], qb[e], sb[e], False)
        for i in range(r1 - r0):
            for n in range(2):
                assert float(abs(Fraction(float(C[r0 + i, n])) - ex[i][n])) <= 2.0 ** -50 * mag[i, n]


def test_planted_mistakes_are_caught(monkeypatch):
    """A wrong scale index or a transposed operand in the oracle trips the brute force."""
    real = og._b_scale

    def wrong_group(sb, n_rows, kb, b_tile):           # uses the next group's scale
        nkb = np.asarray(sb).shape[1]
        return real(sb, n_rows, (kb + 1) % nkb, b_tile)

    monkeypatch.setattr(og, "_b_scale", wrong_group)
    with pytest.raises(AssertionError):
        test_bruteforce_rational(3, 2, 256, False)
    monkeypatch.setattr(og, "_b_scale", real)

    real_decode = og.decode
    monkeypatch.setattr(og, "decode", lambda c: -real_decode(c) if np.asarray(c).shape[0] == 2 else real_decode(c))
    with pytest.raises(AssertionError):
        test_bruteforce_rational(3, 2, 256, True)


# --------------------------------------------------------------------------
# The GEMM result quantised into 1x128 E4M3 tiles (the FP8 producer output).

def _exact_e4m3_rows(M, N, g):
    """A = 1.0 at k=0 only, B row n carries code c_n at k=0: C[m, n] = value(c_n)."""
    K = 128
    qa = np.zeros((M, K), np.uint8)
    qa[:, 0] = 0x38                                   # 1.0
    codes = g.choice(FINITE, size=N).astype(np.uint8)
    for t in range(N // 128):
        codes[128 * t + int(g.integers(0, 128))] = 0x7E  # each tile holds +448
    qb = np.zeros((N, K), np.uint8)
    qb[:, 0] = codes
    return qa, qb, codes


@pytest.mark.parametrize("pow2", [False, True])
def test_gemm_quant_returns_exact_e4m3_products_unchanged(pow2):
    # every C value is an E4M3 value and each tile's amax is 448, so the scale
    # is exactly 1 and every code comes back (negative zero sums to +0)
    g = np.random.default_rng(11)
    qa, qb, codes = _exact_e4m3_rows(3, 384, g)
    sa = np.ones((3, 1), np.float32)
    sb = np.ones((3, 1), np.float32)
    q, s, x = og.gemm_quant(qa, sa, qb, sb, pow2=pow2)
    want = np.where(codes == 0x80, 0x00, codes).astype(np.uint8)
    assert np.all(s == 1.0)
    for m in range(3):
        assert np.array_equal(q[m], want)


@pytest.mark.parametrize("pow2", [False, True])
def test_gemm_quant_scale_direction(pow2):
    # sa = 2^3, sb = 2^-5: C = value * 2^-2, tile amax 112, dequant scale 1/4
    g = np.random.default_rng(12)
    qa, qb, codes = _exact_e4m3_rows(2, 256, g)
    sa = np.full((2, 1), 8.0, np.float32)
    sb = np.full((2, 1), 2.0 ** -5, np.float32)
    q, s, x = og.gemm_quant(qa, sa, qb, sb, pow2=pow2)
    assert np.all(s == 0.25)
    want = np.where(codes == 0x80, 0x00, codes).astype(np.uint8)
    assert np.array_equal(q[1], want)
    assert np.array_equal(e4m3.decode(q[0]) * 0.25, x[0].astype(np.float64))


def test_gemm_quant_tile_bound_and_amax_code():
    # random operands: the tile amax takes code +-448 (non-pow2) and every
    # element is within half an E4M3 step of x / s
    g = np.random.default_rng(13)
    M, N, K = 5, 256, 384
    qa, qb = _codes((M, K), g), _codes((N, K), g)
    sa, sb = _scales((M, K // 128), g), _scales((N // 128, K // 128), g)
    q, s, x = og.gemm_quant(qa, sa, qb, sb)
    C = og.gemm(qa, sa, qb, sb)
    assert np.array_equal(x, C.astype(np.float32))
    for m in range(M):
        for t in range(N // 128):
            xt = x[m, 128 * t:128 * (t + 1)].astype(np.float64)
            qt = q[m, 128 * t:128 * (t + 1)]
            st = float(s[m, t])
            i = int(np.argmax(np.abs(xt)))
            assert e4m3.decode(qt[i:i + 1])[0] == np.copysign(448.0, xt[i])
            y = xt / st
            # E4M3 spacing: 2^(e-3) for |y| in [2^e, 2^(e+1)), 2^-9 below 2^-6
            step = np.where(np.abs(y) < 2.0 ** -6, 2.0 ** -9,
                            2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6))) - 3))
            assert np.all(np.abs(e4m3.decode(qt) - y) <= 0.5 * step * (1 + 1e-6))


def test_gemm_quant_zero_tile_and_ragged_n():
    qa = np.zeros((1, 128), np.uint8)
    qb = np.zeros((128, 128), np.uint8)
    q, s, _ = og.gemm_quant(qa, np.ones((1, 1), np.float32), qb, np.ones((1, 1), np.float32))
    assert np.all(q == 0) and s[0, 0] == np.float32(2.0 ** -64) / np.float32(448)
    with pytest.raises(ValueError):
        og.gemm_quant(np.zeros((1, 128), np.uint8), np.ones((1, 1), np.float32),
                      np.zeros((144, 128), np.uint8), np.ones((144, 1), np.float32), b_tile=True)


# --------------------------------------------------------------------------
# Routed up-projection + SwiGLU, quantised as the down-projection input.

def test_silu_against_library_logistic_and_odd_identity():
    from scipy.special import expit
    x = np.concatenate([np.linspace(-40, 40, 801), [0.0, 1e-30, -1e-30, 700.0, -700.0]])
    assert np.allclose(og.silu(x), x * expit(x), rtol=1e-14, atol=0)
    # sigmoid(x) + sigmoid(-x) = 1  =>  silu(x) - silu(-x) = x
    assert np.allclose(og.silu(x) - og.silu(-x), x, rtol=1e-14, atol=1e-300)
    assert og.silu(0.0) == 0.0 and og.silu(64.0) == 64.0


def _swiglu_case(rows_per_expert, I, g):
    """Gate = 64 exactly for every row, up = E4M3 values: h = 64 * value(up code)."""
    E = len(rows_per_expert)
    T = int(sum(rows_per_expert))
    K = 128
    qa = np.zeros((T, K), np.uint8)
    qa[:, 0] = 0x38                                    # 1.0
    qb = np.zeros((E, 2 * I, K), np.uint8)
    ups = []
    for e in range(E):
        codes = g.choice(FINITE, size=I).astype(np.uint8)
        for t in range(I // 128):
            codes[128 * t + int(g.integers(0, 128))] = 0x7E   # 448 in every tile
        qb[e, :I, 0] = 0x68                            # gate row value 64
        qb[e, I:, 0] = codes                           # up row values
        ups.append(codes)
    off = np.concatenate([[0], np.cumsum(rows_per_expert)]).astype(np.int64)
    sa = np.ones((T, 1), np.float32)
    sb = np.ones((E, 2 * I // 128, 1), np.float32)
    return qa, sa, off, qb, sb, ups


def test_swiglu_quant_worked_exact_case():
    # silu(64) = 64 exactly in float64, so h = 64 * up; every tile's amax is
    # 64 * 448 and its power-of-2 scale 64: the up codes come back unchanged
    g = np.random.default_rng(21)
    qa, sa, off, qb, sb, ups = _swiglu_case([3, 0, 5], 256, g)
    q, s, h = og.grouped_swiglu_quant(qa, sa, off, qb, sb)
    assert np.all(s == 64.0)
    for e, (r0, r1) in enumerate(zip(off[:-1], off[1:])):
        want = np.where(ups[e] == 0x80, 0, ups[e]).astype(np.uint8)
        for r in range(r0, r1):
            assert np.array_equal(q[r], want)
            assert np.array_equal(h[r], (64.0 * e4m3.decode(want)).astype(np.float32))


def test_swiglu_quant_gate_up_order_matters():
    # swapping the gate and up halves gives silu(up) * 64, not 64 * up
    g = np.random.default_rng(22)
    qa, sa, off, qb, sb, ups = _swiglu_case([4], 128, g)
    swapped = np.concatenate([qb[:, 128:], qb[:, :128]], axis=1)
    _, _, h = og.grouped_swiglu_quant(qa, sa, off, qb, sb)
    _, _, h2 = og.grouped_swiglu_quant(qa, sa, off, swapped, sb)
    assert not np.allclose(h, h2)
    up = e4m3.decode(ups[0]).astype(np.float64)
    assert np.allclose(h2[0], (og.silu(up) * 64.0).astype(np.float32))


def test_swiglu_quant_random_tiles_bound():
    # random operands: power-of-2 scales, every element within half an E4M3
    # step of h / s, and each tile's largest magnitude at most 448 after scaling
    g = np.random.default_rng(23)
    sizes = [7, 0, 130, 2]
    T, I, K = sum(sizes), 256, 256
    qa = _codes((T, K), g)
    qb = _codes((len(sizes), 2 * I, K), g)
    sa = _scales((T, K // 128), g) * 1e-6
    sb = (_scales((len(sizes), 2 * I // 128, K // 128), g) * 1e-6).astype(np.float32)
    off = np.concatenate([[0], np.cumsum(sizes)])
    q, s, h = og.grouped_swiglu_quant(qa, sa.astype(np.float32), off, qb, sb)
    C = og.grouped_gemm(qa, sa.astype(np.float32), off, qb, sb)
    assert np.array_equal(h, (og.silu(C[:, :I]) * C[:, I:]).astype(np.float32))
    assert np.all(np.log2(s) == np.round(np.log2(s)))
    y = h.astype(np.float64).reshape(T, I // 128, 128) / s[:, :, None]
    assert np.all(np.abs(y) <= 448.0)
    dec = e4m3.decode(q).reshape(T, I // 128, 128)
    step = np.where(np.abs(y) < 2.0 ** -6, 2.0 ** -9,
                    2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6))) - 3))
    assert np.all(np.abs(dec - y) <= 0.5 * step * (1 + 1e-9))

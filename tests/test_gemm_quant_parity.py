"""GPU block-scaled GEMM with E4M3 output tiles vs the oracle.

The fused epilogue quantises the kernel's FP32 accumulator into 1x128 tiles
along N with the activation quantiser's rules (oracle.gemm_quant; page 2,
inprokorea.com free #735329, fine-grained quantisation passage).

Two checks:
  * bit-exact against fp8_act_quant applied to the same kernel's FP32 output
    (both quantise the identical FP32 accumulator);
  * against the oracle, which quantises fl32 of the exact sum.  The GPU sum
    carries FP32 rounding: each of the nkb promoted FMAs errs by at most 2^-24
    of the running magnitude, so |C32 - C| <= nkb * 2^-24 * sum_kb |P_kb sa sb|
    (=: E).  A code must then equal the oracle's unless the oracle's x*m lies
    within E*m (plus a 2^-22 relative margin for the multiplier) of an E4M3
    rounding midpoint, where either neighbouring code is correct; scales agree
    within the amax's share of E (non-power-of-2) or exactly unless the
    tile's amax/448 lies that close to a power of two.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import e4m3
from tests import helpers as H

pytestmark = pytest.mark.gpu

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def _operands(M, N, K, seed, b_tile):
    g = np.random.default_rng(seed)
    qa = e4m3.encode((g.standard_normal((M, K)) * 40).astype(np.float32))
    qb = e4m3.encode((g.standard_normal((N, K)) * 40).astype(np.float32))
    sa = np.exp(g.uniform(-3, 3, (M, K // 128))).astype(np.float32)
    sb = np.exp(g.uniform(-3, 3, (N, K // 128) if b_tile else (N // 128, K // 128))).astype(np.float32)
    return qa, sa, qb, sb


def _abs_sum(qa, sa, qb, sb, b_tile):
    """sum_kb |P_kb| * sa * sb in float64 (the magnitude the FP32 sum rounds against)."""
    P = np.abs(oracle.slice_partials(qa, qb))
    out = np.zeros(P.shape[1:], np.float64)
    for kb in range(P.shape[0]):
        sbk = sb[:, kb] if b_tile else np.repeat(sb[:, kb], 128)[:qb.shape[0]]
        out += P[kb] * sa[:, kb].astype(np.float64)[:, None] * sbk.astype(np.float64)[None, :]
    return out


def _check_against_oracle(q_gpu, s_gpu, qa, sa, qb, sb, b_tile, pow2, rows=None):
    if rows is not None:
        qa, sa = qa[rows], sa[rows]
    _, _, x_o = oracle.gemm_quant(qa, sa, qb, sb, b_tile=b_tile, pow2=pow2)
    nkb = qa.shape[1] // 128
    err = (nkb + 1) * 2.0 ** -24 * _abs_sum(qa, sa, qb, sb, b_tile)     # bound on |C32 - C|
    return H.check_quant_decisions(q_gpu, s_gpu, x_o, err, pow2)


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("M,N,K,b_tile", [(300, 384, 640, False), (128, 256, 128, False),
                                          (257, 512, 512, True), (1, 128, 256, True)])
def test_fused_equals_act_quant_of_fp32_output(cuda_lib, M, N, K, b_tile, pow2):
    qa, sa, qb, sb = _operands(M, N, K, M + N + K, b_tile)
    d = [H.to_dev(v) for v in (qa, sa, qb, sb)]
    c32 = cuda_lib.gemm(*d, out_dtype=torch.float32, b_tile=b_tile)
    q_ref, s_ref = cuda_lib.act_quant(c32, pow2=pow2)
    raw_q, q = H.guarded_empty((M, N), torch.uint8)
    raw_s, s = H.guarded_empty((M, N // 128), torch.float32)
    cuda_lib.gemm_quant(*d, b_tile=b_tile, pow2=pow2, out=q, out_scales=s)
    torch.cuda.synchronize()
    assert H.guards_intact(raw_q) and H.guards_intact(raw_s), "write outside the outputs"
    assert torch.equal(q, q_ref) and torch.equal(s, s_ref)


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("M,N,K,b_tile", [(300, 384, 640, False), (257, 512, 512, True)])
def test_fused_vs_oracle(cuda_lib, M, N, K, b_tile, pow2):
    qa, sa, qb, sb = _operands(M, N, K, 7 * M + N, b_tile)
    q, s = cuda_lib.gemm_quant(*[H.to_dev(v) for v in (qa, sa, qb, sb)], b_tile=b_tile, pow2=pow2)
    decided = _check_against_oracle(q.cpu().numpy(), s.cpu().numpy(), qa, sa, qb, sb, b_tile, pow2)
    assert decided > 0.99


def test_exact_products_come_back_unchanged(cuda_lib):
    # every C value is an E4M3 value and every tile holds 448: scale 1, same codes
    g = np.random.default_rng(5)
    M, N, K = 130, 384, 128
    qa = np.zeros((M, K), np.uint8)
    qa[:, 0] = 0x38
    codes = g.choice(FINITE, size=N).astype(np.uint8)
    codes[[3, 200, 300]] = 0x7E
    qb = np.zeros((N, K), np.uint8)
    qb[:, 0] = codes
    ones_a = np.ones((M, 1), np.float32)
    ones_b = np.ones((N // 128, 1), np.float32)
    for pow2 in (False, True):
        q, s = cuda_lib.gemm_quant(*[H.to_dev(v) for v in (qa, ones_a, qb, ones_b)], pow2=pow2)
        want = np.where(codes == 0x80, 0, codes).astype(np.uint8)
        assert np.all(s.cpu().numpy() == 1.0)
        assert np.array_equal(q.cpu().numpy(), np.broadcast_to(want, (M, N)))


def test_fprop_full_size_sampled(cuda_lib):
    """X[4096,7168] . W[18432,7168]^T quantised into 1x128 tiles; sampled rows vs the oracle."""
    case = synth.dense_case("fprop")
    x, w = case.x(), case.w()
    qa, sa = cuda_lib.act_quant(x.cuda())
    qb, sb = cuda_lib.weight_quant(w.cuda())
    q, s = cuda_lib.gemm_quant(qa, sa, qb, sb)
    c32 = cuda_lib.gemm(qa, sa, qb, sb, out_dtype=torch.float32)
    q_ref, s_ref = cuda_lib.act_quant(c32)
    assert torch.equal(q, q_ref) and torch.equal(s, s_ref)
    rows = np.unique(np.concatenate([np.arange(4), np.arange(case.M - 4, case.M), [1000, 2500]]))
    decided = _check_against_oracle(q.cpu().numpy()[rows], s.cpu().numpy()[rows],
                                    qa.cpu().numpy(), sa.cpu().numpy(), qb.cpu().numpy(),
                                    sb.cpu().numpy(), False, False, rows=rows)
    assert decided > 0.99

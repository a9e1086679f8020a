"""The per-element GEMM error bound the parity tests use (CPU only).

tests/helpers.py, gemm_error_bound, bounds |C32 - C| for the promoted FP32 sum
of page 2 (inprokorea.com free #735329, promotion passage and Figure 6).  Here
a float32 emulation of that sum must satisfy the bound on random operands:
each 128-K group is accumulated in four K=32 steps with an FP32 rounding after
each, its scale product is rounded to FP32, and it is added into an FP32
accumulator.  Plausible kernel mistakes (a dropped group, a wrong scale, one
wrong element, a group counted twice) must break it.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import e4m3
from tests import helpers as H


def _operands(M, N, K, seed, b_tile=False):
    g = np.random.default_rng(seed)
    qa = e4m3.encode((g.standard_normal((M, K)) * 60).astype(np.float32))
    qb = e4m3.encode((g.standard_normal((N, K)) * 60).astype(np.float32))
    sa = np.exp(g.uniform(-4, 4, (M, K // 128))).astype(np.float32)
    sb = np.exp(g.uniform(-4, 4, (N, K // 128) if b_tile else (N // 128, K // 128))).astype(np.float32)
    return qa, sa, qb, sb


def _emulate_fp32(qa, sa, qb, sb, b_tile=False, drop=None, scale_bug=None):
    """Promoted sum in float32 arithmetic (with optional planted mistakes)."""
    A = e4m3.decode(qa).astype(np.float64)
    B = e4m3.decode(qb).astype(np.float64)
    M, K = A.shape
    N = B.shape[0]
    acc = np.zeros((M, N), np.float32)
    for kb in range(K // 128):
        if kb == drop:
            continue
        t = np.zeros((M, N), np.float32)
        for c in range(4):                                   # four K=32 tensor-core steps
            sl = slice(128 * kb + 32 * c, 128 * kb + 32 * c + 32)
            t = (t.astype(np.float64) + A[:, sl] @ B[:, sl].T).astype(np.float32)
        sbk = sb[:, kb] if b_tile else np.repeat(sb[:, kb], 128)[:N]
        s = (sa[:, kb][:, None] * sbk[None, :]).astype(np.float32)   # FP32 product
        if scale_bug is not None and kb == scale_bug:
            s = (s * np.float32(1.001)).astype(np.float32)
        acc = (acc.astype(np.float64) + t.astype(np.float64) * s.astype(np.float64)).astype(np.float32)
    return acc


@pytest.mark.parametrize("b_tile", [False, True])
@pytest.mark.parametrize("M,N,K", [(64, 128, 512), (33, 256, 1024)])
def test_fp32_emulation_within_bound(M, N, K, b_tile):
    qa, sa, qb, sb = _operands(M, N, K, M + N + K, b_tile)
    ref = oracle.gemm(qa, sa, qb, sb, b_tile=b_tile)
    bound = H.gemm_error_bound(qa, sa, qb, sb, b_tile=b_tile)
    c32 = _emulate_fp32(qa, sa, qb, sb, b_tile)
    worst = H.assert_elementwise(c32, ref, bound, "fp32 emulation")
    assert worst < 1.0
    # BF16 output: one RNE rounding of the FP32 value on top
    cb = torch.from_numpy(c32).to(torch.bfloat16)
    H.assert_elementwise(cb, ref, bound, "bf16 emulation")


def test_bound_is_tight_enough_to_matter():
    # the bound is far below the normwise tolerance's per-element scale ...
    qa, sa, qb, sb = _operands(48, 128, 1024, 3)
    ref = oracle.gemm(qa, sa, qb, sb)
    bound = H.gemm_error_bound(qa, sa, qb, sb)
    assert np.median(bound / np.abs(ref)) < 1e-4


@pytest.mark.parametrize("mistake", ["drop_group", "scale", "one_element", "double_group"])
def test_planted_mistakes_break_the_bound(mistake):
    qa, sa, qb, sb = _operands(64, 128, 512, 11)
    ref = oracle.gemm(qa, sa, qb, sb)
    bound = H.gemm_error_bound(qa, sa, qb, sb)
    if mistake == "drop_group":
        bad = _emulate_fp32(qa, sa, qb, sb, drop=2)
    elif mistake == "scale":
        bad = _emulate_fp32(qa, sa, qb, sb, scale_bug=1)
    elif mistake == "one_element":
        bad = _emulate_fp32(qa, sa, qb, sb)
        bad[5, 77] = np.float32(bad[5, 77] * np.float32(1.0 + 2.0 ** -10))
    else:
        qa2 = qa.copy()
        qa2[:, 128:256] = qa[:, 0:128]                  # group 0's codes where group 1's belong
        bad = _emulate_fp32(qa2, sa, qb, sb)
    with pytest.raises(AssertionError):
        H.assert_elementwise(bad, ref, bound, mistake)

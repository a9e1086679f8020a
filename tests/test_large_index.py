"""Tensors of more than 2^31 elements (each dimension below 2^31, the ABI's rule).

A kernel that formed an element offset in 32 bits would read or write the
wrong place past element 2^31.  Each kernel here runs once on such a tensor,
and samples of its output are compared with the oracle: the first and last
rows, columns or blocks, and those around element 2^31.  Quantiser codes and
scales must match bit for bit; the GEMMs must stay within the per-element
bound of tests/helpers.py.  Inputs are drawn on the GPU (seeded) and only the
sampled parts travel to the host.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu

BIG = 1 << 31


def _gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def _f32(t):
    return synth.bf16_to_f32(t.cpu()) if t.dtype == torch.bfloat16 else t.cpu().numpy()


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_act_quant_rows_past_2_31(cuda_lib):
    M, K = (1 << 18) + 64, 8192
    assert M * K > BIG
    x = torch.randn((M, K), generator=_gen(1), device="cuda").to(torch.bfloat16)
    q, s = cuda_lib.act_quant(x)
    edge = BIG // K
    for r0, r1 in ((0, 64), (edge - 32, edge + 32), (M - 64, M)):
        qr, sr = oracle.act_quant(_f32(x[r0:r1]))
        assert np.array_equal(q[r0:r1].cpu().numpy(), qr), f"codes, rows {r0}..{r1}"
        assert np.array_equal(s[r0:r1].cpu().numpy().view(np.int32), sr.view(np.int32)), f"scales, rows {r0}..{r1}"


def test_act_quant_transposed_past_2_31(cuda_lib):
    M, K = (1 << 18) + 128, 8192
    assert M * K > BIG and M % 128 == 0
    x = torch.randn((M, K), generator=_gen(2), device="cuda").to(torch.bfloat16)
    qt, st = cuda_lib.act_quant(x, transpose=True)          # [K, M], [K, M/128]
    cols = [0, 1, K // 2, K - 2, K - 1]
    xc = _f32(x[:, cols].contiguous())                       # every row of the sampled columns
    qr, sr = oracle.act_quant_t(xc)                          # [len(cols), M]
    assert np.array_equal(qt[cols].cpu().numpy(), qr)
    assert np.array_equal(st[cols].cpu().numpy().view(np.int32), sr.view(np.int32))


def test_weight_quant_with_transpose_past_2_31(cuda_lib):
    N, K = 16384 + 128, 131072
    assert N * K > BIG
    w = (torch.randn((N, K), generator=_gen(3), device="cuda") * 0.02).to(torch.bfloat16)
    q, s, qt, st = cuda_lib.weight_quant(w, transposed=True)
    edge_row = (BIG // K) // 128 * 128
    for r0 in (0, edge_row, N - 128):
        for c0 in (0, K - 1024):
            blk = _f32(w[r0:r0 + 128, c0:c0 + 1024])
            qr, sr = oracle.weight_quant(blk)
            assert np.array_equal(q[r0:r0 + 128, c0:c0 + 1024].cpu().numpy(), qr), (r0, c0)
            assert np.array_equal(qt[c0:c0 + 1024, r0:r0 + 128].cpu().numpy(), qr.T), (r0, c0)
            got = s[r0 // 128, c0 // 128:c0 // 128 + 8].cpu().numpy()
            assert np.array_equal(got.view(np.int32), sr[0].view(np.int32)), (r0, c0)
            got_t = st[c0 // 128:c0 // 128 + 8, r0 // 128].cpu().numpy()
            assert np.array_equal(got_t.view(np.int32), sr[0].view(np.int32)), (r0, c0)


def test_requant_transpose_past_2_31(cuda_lib):
    M, K = (1 << 18) + 128, 8192
    x = torch.randn((M, K), generator=_gen(4), device="cuda").to(torch.bfloat16)
    q, s = cuda_lib.act_quant(x)
    del x
    qt, st = cuda_lib.requant_transpose(q, s)                # [K, M], [K, M/128]
    for grp in (0, K // 128 - 1):                            # whole 128-column groups, every row
        c0 = grp * 128
        qr, sr = oracle.requant_t(q[:, c0:c0 + 128].cpu().numpy(), s[:, grp:grp + 1].cpu().numpy())
        assert np.array_equal(qt[c0:c0 + 128].cpu().numpy(), qr), grp
        assert np.array_equal(st[c0:c0 + 128].cpu().numpy().view(np.int32), sr.view(np.int32)), grp


def _codes(shape, gen):
    mag = torch.randint(0, 0x7E, shape, generator=gen, device="cuda", dtype=torch.int32)
    sgn = torch.randint(0, 2, shape, generator=gen, device="cuda", dtype=torch.int32) * 0x80
    return (mag | sgn).to(torch.uint8)


def test_gemm_output_past_2_31(cuda_lib):
    M, N, K = 65536, 32768 + 256, 128
    assert M * N > BIG
    g = _gen(5)
    a, b = _codes((M, K), g), _codes((N, K), g)
    sa = torch.exp(torch.rand((M, 1), generator=g, device="cuda") * 4 - 2)
    sb = torch.exp(torch.rand((N // 128, 1), generator=g, device="cuda") * 4 - 2)
    c = cuda_lib.gemm(a, sa, b, sb, out_dtype=torch.bfloat16)
    qb, sbn = b.cpu().numpy(), sb.cpu().numpy()
    edge = BIG // N
    for r0, r1 in ((0, 4), (edge - 2, edge + 2), (M - 4, M)):
        qa, san = a[r0:r1].cpu().numpy(), sa[r0:r1].cpu().numpy()
        ref = oracle.gemm(qa, san, qb, sbn)
        H.assert_elementwise(c[r0:r1], ref, H.gemm_error_bound(qa, san, qb, sbn), f"rows {r0}..{r1}")


def test_grouped_gemm_output_past_2_31(cuda_lib):
    T, N, K, E = 65536, 32768 + 256, 128, 2
    g = _gen(6)
    a, b = _codes((T, K), g), _codes((E, N, K), g)
    sa = torch.exp(torch.rand((T, 1), generator=g, device="cuda") * 4 - 2)
    sb = torch.exp(torch.rand((E, N // 128, 1), generator=g, device="cuda") * 4 - 2)
    off = torch.tensor([0, 40000, T], dtype=torch.int32, device="cuda")
    c = cuda_lib.grouped_gemm(a, sa, off, b, sb, out_dtype=torch.bfloat16)
    edge = BIG // N
    for r0, r1, e in ((0, 4, 0), (39998, 40000, 0), (40000, 40002, 1), (edge - 2, edge + 2, 1), (T - 4, T, 1)):
        qa, san = a[r0:r1].cpu().numpy(), sa[r0:r1].cpu().numpy()
        qb, sbn = b[e].cpu().numpy(), sb[e].cpu().numpy()
        ref = oracle.gemm(qa, san, qb, sbn)
        H.assert_elementwise(c[r0:r1], ref, H.gemm_error_bound(qa, san, qb, sbn), f"rows {r0}..{r1}")

"""Data-parallel sharding of the FFN step, emulated on one GPU.

The path shards over tokens: a data-parallel rank holds a contiguous block of
rows of X and dY and the whole weight W.
- Fprop (X W^T) and Dgrad (dY W) rows depend only on the rank's own rows, and
  1x128 activation tiles never span rows (page 1, xn--9g3bo1gtkw0l8ubf92bgle.kr
  qna #85187, Figure 7 (a)).  Each shard's outputs must therefore equal the
  unsharded outputs' rows bit for bit.
- Wgrad (dY^T X) contracts over tokens.  Each rank quantises its own dY^T and
  re-quantises its stored X into 128x1 tiles (page 5, inprokorea.com free
  #890463, backward-pass passage).  Shards are multiples of 128 tokens, so no
  tile crosses a shard and the ranks hold exactly the unsharded codes.  Each
  rank's partial dW covers its own 128-token groups, and the ranks' partials
  are summed in FP32: the gradient all-reduce of data parallelism.  The sum
  differs from the unsharded Wgrad only in the order of FP32 additions, so both
  stay within the per-element bound widened by one addition per extra rank.
"""

import pytest
import torch

import fp8_fine_grained_19_b300 as fp8
import oracle
from tests import helpers as TH

pytestmark = pytest.mark.gpu

TOKENS, HIDDEN, FFN = 512, 1024, 768


def _step(xs, dys, qw, sw, qwt, swt):
    qx, sx = fp8.act_quant(xs)
    y = fp8.gemm(qx, sx, qw, sw, out_dtype=torch.bfloat16, stream_k=False)        # Fprop [t, FFN]
    qd, sd = fp8.act_quant(dys)
    dx = fp8.gemm(qd, sd, qwt, swt, out_dtype=torch.bfloat16, stream_k=False)     # Dgrad [t, HIDDEN]
    qdt, sdt = fp8.act_quant(dys, transpose=True)                                # dY^T [FFN, t]
    qxt, sxt = fp8.requant_transpose(qx, sx)                                     # X^T [HIDDEN, t]
    dw = fp8.gemm(qdt, sdt, qxt, sxt, out_dtype=torch.float32, b_tile=True,      # Wgrad [FFN, HIDDEN]
                  stream_k=False)
    return y, dx, dw, (qdt, sdt, qxt, sxt)


@pytest.mark.parametrize("shards", [2, 4])
def test_token_shards_reproduce_the_unsharded_step(cuda_lib, shards):
    g = torch.Generator().manual_seed(19 + shards)
    x = torch.randn((TOKENS, HIDDEN), generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn((FFN, HIDDEN), generator=g) * 0.02).to(torch.bfloat16).cuda()
    dy = (torch.randn((TOKENS, FFN), generator=g) * 1e-3).to(torch.bfloat16).cuda()
    qw, sw, qwt, swt = fp8.weight_quant(w, transposed=True)

    y, dx, dw, full = _step(x, dy, qw, sw, qwt, swt)
    rows = TOKENS // shards
    assert rows % 128 == 0
    dw_sum = torch.zeros_like(dw)
    for r in range(shards):
        sl = slice(r * rows, (r + 1) * rows)
        y_r, dx_r, dw_r, ops_r = _step(x[sl].contiguous(), dy[sl].contiguous(), qw, sw, qwt, swt)
        assert torch.equal(y_r, y[sl]), f"Fprop rows of shard {r}"
        assert torch.equal(dx_r, dx[sl]), f"Dgrad rows of shard {r}"
        # the shard's 128x1 codes and scales are the unsharded ones of its tokens
        qdt_r, sdt_r, qxt_r, sxt_r = ops_r
        g0, g1 = r * rows // 128, (r + 1) * rows // 128
        assert torch.equal(qdt_r, full[0][:, sl]) and torch.equal(sdt_r, full[1][:, g0:g1])
        assert torch.equal(qxt_r, full[2][:, sl]) and torch.equal(sxt_r, full[3][:, g0:g1])
        dw_sum += dw_r                                   # the all-reduce, in rank order
    torch.cuda.synchronize()
    assert fp8.device_status() == fp8.OK

    qdt, sdt, qxt, sxt = (t.cpu().numpy() for t in full)
    ref = oracle.gemm(qdt, sdt, qxt, sxt, b_tile=True)
    bound = TH.gemm_error_bound(qdt, sdt, qxt, sxt, b_tile=True, extra_adds=shards - 1)
    TH.assert_elementwise(dw, ref, bound, "unsharded Wgrad")
    TH.assert_elementwise(dw_sum, ref, bound, "summed Wgrad partials")
    assert TH.normwise_rel_err(dw_sum, ref) <= 1e-5

"""Stream-K split of the dense block-scaled GEMM vs the oracle and vs the whole-tile path.

fp8_blockscaled_gemm_ws keeps the full waves of output tiles whole and shares
each leftover tile among its own group of CTAs, which divide its 128-K groups
evenly; a shared tile is summed from the group's FP32 partial sums by a second
kernel, in a fixed order.  The result is the promoted
sum of page 2 (inprokorea.com free #735329, promotion passage and Figure 6) with
one more FP32 addition per extra part, so the per-element bound gains that many
terms (tests/helpers.py, gemm_error_bound, extra_adds).  Forced splits on small
ragged shapes put up to one group per CTA, so a tile may have as many parts as
groups; the Dgrad shape (896 tiles on 148 SMs) splits on its own.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import e4m3
from tests import helpers as H

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 4e-3}


def _operands(M, N, K, seed, b_tile=False):
    g = np.random.default_rng(seed)
    qa = e4m3.encode((g.standard_normal((M, K)) * 60).astype(np.float32))
    qb = e4m3.encode((g.standard_normal((N, K)) * 60).astype(np.float32))
    sa = np.exp(g.uniform(-4, 4, (M, K // 128))).astype(np.float32)
    sb = np.exp(g.uniform(-4, 4, (N, K // 128) if b_tile else (N // 128, K // 128))).astype(np.float32)
    return qa, sa, qb, sb


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K,b_tile", [(300, 768, 1280, False), (129, 400, 2048, True),
                                          (1, 128, 6144, False), (520, 1024, 384, False),
                                          (700, 2304, 1024, True)])
def test_forced_split_vs_oracle(cuda_lib, M, N, K, b_tile, dtype):
    qa, sa, qb, sb = _operands(M, N, K, M + 3 * N + K, b_tile)
    assert cuda_lib.gemm_workspace_bytes(M, N, K, b_tile, stream_k=True) > 0
    d = [H.to_dev(v) for v in (qa, sa, qb, sb)]
    raw, out = H.guarded_empty((M, N), dtype)
    cuda_lib.gemm(*d, b_tile=b_tile, out=out, stream_k=True)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == cuda_lib.OK
    assert H.guards_intact(raw), "write outside the output"
    ref = oracle.gemm(qa, sa, qb, sb, b_tile=b_tile)
    assert H.normwise_rel_err(out, ref) <= TOL[dtype]
    nkb = K // 128
    H.assert_elementwise(out, ref, H.gemm_error_bound(qa, sa, qb, sb, b_tile, extra_adds=nkb),
                         f"stream-K {M}x{N}x{K}")
    # the same result on every run (the parts are added in a fixed order)
    again = cuda_lib.gemm(*d, b_tile=b_tile, out_dtype=dtype, stream_k=True)
    assert torch.equal(out, again)
    # and the whole-tile path agrees within both bounds
    whole = cuda_lib.gemm(*d, b_tile=b_tile, out_dtype=dtype, stream_k=False)
    H.assert_elementwise(whole, ref, H.gemm_error_bound(qa, sa, qb, sb, b_tile), "whole tiles")


def test_split_with_caller_workspace_and_reuse(cuda_lib):
    # a caller-owned workspace, reused by two different shapes in a row: its
    # contents on entry do not matter
    M, N, K = 300, 768, 1280
    qa, sa, qb, sb = _operands(M, N, K, 5)
    need = cuda_lib.gemm_workspace_bytes(M, N, K, stream_k=True)
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device="cuda")
    d = [H.to_dev(v) for v in (qa, sa, qb, sb)]
    a = cuda_lib.gemm(*d, out_dtype=torch.float32, stream_k=True, workspace=ws)
    qa2, sa2, qb2, sb2 = _operands(129, 384, 2048, 6, True)
    cuda_lib.gemm(*[H.to_dev(v) for v in (qa2, sa2, qb2, sb2)], b_tile=True, out_dtype=torch.float32,
                  stream_k=True, workspace=ws)
    b = cuda_lib.gemm(*d, out_dtype=torch.float32, stream_k=True, workspace=ws)
    assert torch.equal(a, b)
    ref = oracle.gemm(qa, sa, qb, sb)
    H.assert_elementwise(b, ref, H.gemm_error_bound(qa, sa, qb, sb, extra_adds=K // 128), "reuse")


def test_workspace_too_small_is_rejected(cuda_lib):
    M, N, K = 300, 768, 1280
    qa, sa, qb, sb = [H.to_dev(v) for v in _operands(M, N, K, 7)]
    need = cuda_lib.gemm_workspace_bytes(M, N, K, stream_k=True)
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.Fp8Error) as e:
        cuda_lib.gemm(qa, sa, qb, sb, stream_k=True, workspace=small)
    assert e.value.status == cuda_lib.ERR_INVALID_ARG


def test_auto_split_on_the_dgrad_shape(cuda_lib):
    # 896 output tiles on the SMs: the last wave would leave most SMs idle for
    # most of the 144 groups, so the automatic choice splits
    assert cuda_lib.gemm_workspace_bytes(4096, 7168, 18432) > 0
    # the Fprop shape's last wave is nearly full: no split
    assert cuda_lib.gemm_workspace_bytes(4096, 18432, 7168) == 0


def test_split_inside_a_cuda_graph(cuda_lib):
    # 160 output tiles on 148 SMs: a whole-tile launch and a split launch (the
    # second queued with programmatic stream serialisation), then the fix-up.
    # In one captured graph: act_quant produces A, the GEMM consumes it, and a
    # torch op reads C right after; every replay must equal the eager run.
    M, N, K = 2048, 2560, 1280
    lib = cuda_lib.load()
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    x = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    _, _, qb_np, sb_np = _operands(M, N, K, 12)
    qb, sb = H.to_dev(qb_np), H.to_dev(sb_np)
    qa = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
    need = cuda_lib.gemm_workspace_bytes(M, N, K, stream_k=True)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y = torch.empty_like(c)

    def body():
        sp = torch.cuda.current_stream().cuda_stream
        assert lib.fp8_act_quant(x.data_ptr(), cuda_lib.BF16, M, K, qa.data_ptr(), sa.data_ptr(), 0,
                                 sp) == cuda_lib.OK
        assert lib.fp8_blockscaled_gemm_ws(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(),
                                           c.data_ptr(), cuda_lib.F32, M, N, K, cuda_lib.STREAM_K,
                                           ws.data_ptr(), need, sp) == cuda_lib.OK
        torch.mul(c, 2.0, out=y)

    body()
    torch.cuda.synchronize()
    c_eager, y_eager = c.clone(), y.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()
    for _ in range(2):
        c.fill_(float("nan"))
        y.fill_(float("nan"))
        qa.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(c, c_eager) and torch.equal(y, y_eager)
    assert cuda_lib.device_status() == cuda_lib.OK
    qa_np, sa_np = qa.cpu().numpy(), sa.cpu().numpy()
    ref = oracle.gemm(qa_np, sa_np, qb_np, sb_np)
    H.assert_elementwise(c_eager, ref, H.gemm_error_bound(qa_np, sa_np, qb_np, sb_np, extra_adds=K // 128),
                         "split in a graph")

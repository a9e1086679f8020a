"""GPU grouped (per-expert) block-scaled GEMM vs the oracle.

Covers ragged expert groups (empty, 1-row, 129-row, >256-row experts, empty
first/last experts), a small routed MoE layer compared in full, the
full-size routed layer (256 experts, top-8, 8192 tokens, hidden 7168, expert
hidden 2048) on sampled experts, and device-side rejection of bad offsets.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import e4m3
from tests import helpers as H

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 4e-3}


def _operands(sizes, N, K, seed):
    g = np.random.default_rng(seed)
    off = synth.ragged_offsets(sizes)
    T, E = int(off[-1]), len(sizes)
    qa = e4m3.encode((g.standard_normal((T, K)) * 50).astype(np.float32))
    sa = np.exp(g.uniform(-3, 3, (T, K // 128))).astype(np.float32)
    qb = e4m3.encode((g.standard_normal((E, N, K)) * 50).astype(np.float32))
    sb = np.exp(g.uniform(-3, 3, (E, N // 128, K // 128))).astype(np.float32)
    return off, qa, sa, qb, sb


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("sizes", [[0, 1, 129, 0, 300, 2], [5], [0, 0, 260, 0],
                                   [128, 128, 1, 255, 0, 3, 64, 0]])
def test_ragged_groups(cuda_lib, sizes, dtype):
    N, K = 384, 384
    off, qa, sa, qb, sb = _operands(sizes, N, K, sum(sizes) + len(sizes))
    T = int(off[-1])
    raw, out = H.guarded_empty((T, N), dtype)
    cuda_lib.grouped_gemm(H.to_dev(qa), H.to_dev(sa), H.to_dev(off), H.to_dev(qb), H.to_dev(sb),
                          out=out)
    assert cuda_lib.device_status() == cuda_lib.OK
    assert H.guards_intact(raw)
    ref = oracle.grouped_gemm(qa, sa, off, qb, sb)
    assert H.normwise_rel_err(out, ref) <= TOL[dtype]
    H.assert_elementwise(out, ref, H.grouped_error_bound(qa, sa, off, qb, sb), f"ragged {sizes}")


def test_single_expert_matches_dense_kernel(cuda_lib):
    off, qa, sa, qb, sb = _operands([333], 256, 512, 7)
    g = cuda_lib.grouped_gemm(H.to_dev(qa), H.to_dev(sa), H.to_dev(off), H.to_dev(qb),
                              H.to_dev(sb), out_dtype=torch.float32)
    d = cuda_lib.gemm(H.to_dev(qa), H.to_dev(sa), H.to_dev(qb[0]), H.to_dev(sb[0]),
                      out_dtype=torch.float32)
    assert torch.equal(g, d)


@pytest.mark.parametrize("bad", ["decreasing", "last_not_total", "first_not_zero"])
def test_bad_offsets_rejected_on_device(cuda_lib, bad):
    off, qa, sa, qb, sb = _operands([100, 50, 80], 256, 256, 3)
    if bad == "decreasing":
        off[1], off[2] = 120, 100
    elif bad == "last_not_total":
        off[3] = 229
    else:
        off[0] = 4
    T = qa.shape[0]
    raw, out = H.guarded_empty((T, 256), torch.float32, fill_byte=0x5A)
    cuda_lib.grouped_gemm(H.to_dev(qa), H.to_dev(sa), H.to_dev(off.astype(np.int32)),
                          H.to_dev(qb), H.to_dev(sb), out=out)
    assert cuda_lib.device_status() == cuda_lib.ERR_BAD_OFFSETS
    assert bool((raw == 0x5A).all().item()), "output written despite bad offsets"
    assert cuda_lib.device_status() == cuda_lib.OK          # read-and-clear
    # and the library keeps working afterwards
    off2, qa2, sa2, qb2, sb2 = _operands([10, 20], 256, 256, 4)
    out2 = cuda_lib.grouped_gemm(H.to_dev(qa2), H.to_dev(sa2), H.to_dev(off2), H.to_dev(qb2),
                                 H.to_dev(sb2), out_dtype=torch.float32)
    assert H.normwise_rel_err(out2, oracle.grouped_gemm(qa2, sa2, off2, qb2, sb2)) <= 1e-5


def _routed_rows(case):
    tok = case.tokens()
    r = synth.moe_route(H.f32(tok), case.router(), case.bias(), case.topk)
    return tok, r


def test_small_routed_layer_full(cuda_lib):
    """Routed MoE layer with the full-size structure at a size the oracle finishes quickly."""
    case = synth.MOE_SMALL
    tok, r = _routed_rows(case)
    off = r["offsets"]
    # tokens quantised once on power-of-2 scales, then gathered into expert order
    qx, sx = cuda_lib.act_quant(tok.cuda(), pow2=True)
    qx_r, sx_r = oracle.act_quant(H.f32(tok), pow2=True)
    assert np.array_equal(qx.cpu().numpy(), qx_r)
    idx = torch.from_numpy(r["token_of_row"]).cuda()
    qa, sa = qx.index_select(0, idx).contiguous(), sx.index_select(0, idx).contiguous()
    qa_r, sa_r = qx_r[r["token_of_row"]], sx_r[r["token_of_row"]]
    wu = torch.stack([synth.expert_weight(case, e, "up") for e in range(case.E)])
    wd = torch.stack([synth.expert_weight(case, e, "down") for e in range(case.E)])
    qu, su = cuda_lib.weight_quant(wu.reshape(-1, case.H).cuda())
    qu_r, su_r = oracle.weight_quant(H.f32(wu.reshape(-1, case.H)))
    assert np.array_equal(qu.cpu().numpy(), qu_r)
    qu = qu.view(case.E, 2 * case.I, case.H)
    su = su.view(case.E, 2 * case.I // 128, case.H // 128)
    qu_r = qu_r.reshape(case.E, 2 * case.I, case.H)
    su_r = su_r.reshape(case.E, 2 * case.I // 128, case.H // 128)
    dev_off = H.to_dev(off)
    ref = oracle.grouped_gemm(qa_r, sa_r, off, qu_r, su_r)
    bound = H.grouped_error_bound(qa_r, sa_r, off, qu_r, su_r)
    for dtype in (torch.bfloat16, torch.float32):
        up = cuda_lib.grouped_gemm(qa, sa, dev_off, qu, su, out_dtype=dtype)
        assert H.normwise_rel_err(up, ref) <= TOL[dtype]
        H.assert_elementwise(up, ref, bound, f"small routed up {dtype}")
    # down projection from a drawn h (power-of-2 scales)
    h = synth.swiglu_like_bf16((case.rows, case.I), case.seed)
    qh, sh = cuda_lib.act_quant(h.cuda(), pow2=True)
    qh_r, sh_r = oracle.act_quant(H.f32(h), pow2=True)
    assert np.array_equal(qh.cpu().numpy(), qh_r)
    qd, sd = cuda_lib.weight_quant(wd.reshape(-1, case.I).cuda())
    qd_r, sd_r = oracle.weight_quant(H.f32(wd.reshape(-1, case.I)))
    assert np.array_equal(qd.cpu().numpy(), qd_r)
    down = cuda_lib.grouped_gemm(qh, sh, dev_off, qd.view(case.E, case.H, case.I),
                                 sd.view(case.E, case.H // 128, case.I // 128),
                                 out_dtype=torch.float32)
    qd3 = qd_r.reshape(case.E, case.H, case.I)
    sd3 = sd_r.reshape(case.E, case.H // 128, case.I // 128)
    ref = oracle.grouped_gemm(qh_r, sh_r, off, qd3, sd3)
    assert H.normwise_rel_err(down, ref) <= TOL[torch.float32]
    H.assert_elementwise(down, ref, H.grouped_error_bound(qh_r, sh_r, off, qd3, sd3), "small routed down")


def test_full_routed_layer_sampled_experts(cuda_lib):
    """256 experts, top-8 of 8192 tokens: every expert runs, a few are checked in full."""
    case = synth.MOE_FULL
    tok, r = _routed_rows(case)
    off, counts = r["offsets"], r["counts"]
    qx, sx = cuda_lib.act_quant(tok.cuda(), pow2=True)
    idx = torch.from_numpy(r["token_of_row"]).cuda()
    qa, sa = qx.index_select(0, idx).contiguous(), sx.index_select(0, idx).contiguous()
    # expert weights drawn on the device, quantised there
    qu = torch.empty((case.E, 2 * case.I, case.H), dtype=torch.uint8, device="cuda")
    su = torch.empty((case.E, 2 * case.I // 128, case.H // 128), dtype=torch.float32, device="cuda")
    for e in range(case.E):
        q_e, s_e = cuda_lib.weight_quant(synth.expert_weight(case, e, "up", "cuda"))
        qu[e].copy_(q_e)
        su[e].copy_(s_e)
    up = cuda_lib.grouped_gemm(qa, sa, H.to_dev(off), qu, su, out_dtype=torch.bfloat16)
    assert cuda_lib.device_status() == cuda_lib.OK
    nz = np.nonzero(counts)[0]
    check = sorted({int(nz[0]), int(nz[-1]), int(np.argmax(counts)), int(nz[np.argmin(counts[nz])]),
                    int(nz[len(nz) // 2])})
    qx_r, sx_r = H.oracle_act_quant_rows(H.f32(tok), pow2=True)
    assert np.array_equal(qx.cpu().numpy(), qx_r)
    for e in check:
        w_e = synth.expert_weight(case, e, "up", "cuda").cpu()
        qe_r, se_r = oracle.weight_quant(H.f32(w_e))
        assert np.array_equal(qu[e].cpu().numpy(), qe_r) and \
            np.array_equal(su[e].cpu().numpy(), se_r)
        rows = slice(int(off[e]), int(off[e + 1]))
        toks = r["token_of_row"][rows]
        ref = oracle.gemm(qx_r[toks], sx_r[toks], qe_r, se_r)
        assert H.normwise_rel_err(up[rows], ref) <= TOL[torch.bfloat16], e
        H.assert_elementwise(up[rows], ref, H.gemm_error_bound(qx_r[toks], sx_r[toks], qe_r, se_r),
                             f"full routed up, expert {e}")

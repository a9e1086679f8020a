"""GPU quantisers vs the oracle: E4M3 codes and FP32 scales must match bit for bit.

Covers the 1x128 row tiles, the 128x1 transposed tiles and the 128x128 weight
blocks, BF16 and FP32 sources, power-of-2 scales, crafted edge tiles (zeros,
signed zeros, outliers, exact E4M3 midpoints and their neighbours, subnormal
codes, FP32 subnormal and huge inputs, power-of-2 boundaries), ragged row
counts, the workloads' full sizes, and canary guards around every output.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import e4m3
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu().contiguous()
    return a.view(torch.int32).numpy() if a.dtype == torch.float32 else a.numpy()


def _assert_same(q_gpu, s_gpu, q_ref, s_ref):
    qg = q_gpu.cpu().numpy()
    if not np.array_equal(qg, q_ref):
        bad = np.argwhere(qg != q_ref)
        raise AssertionError(f"{len(bad)} code mismatches, first at {bad[:3].tolist()}: "
                             f"gpu {qg[tuple(bad[0])]:#x} ref {q_ref[tuple(bad[0])]:#x}")
    sg = s_gpu.cpu().numpy()
    assert np.array_equal(sg.view(np.int32), np.asarray(s_ref, np.float32).view(np.int32)), \
        "scale mismatch"


def edge_tiles() -> np.ndarray:
    """float32 [3, 1536]: 12 tiles per row with crafted contents."""
    g = np.random.default_rng(5)
    rows = []
    codes = np.arange(0, 0x7E, dtype=np.uint8)
    lo, hi = e4m3.decode(codes), e4m3.decode(codes + 1)
    mids = ((lo + hi) / 2).astype(np.float32)                  # 126 midpoints (exact)
    for r in range(3):
        t = []
        t.append(np.zeros(128, np.float32))                     # all zero
        t.append(np.full(128, -0.0, np.float32))                # negative zeros
        z = g.standard_normal(128).astype(np.float32)
        z[17] = 1e4
        t.append(z)                                             # one outlier
        m = np.concatenate([mids, [448.0, -448.0]]).astype(np.float32)
        t.append(m * (1 if r == 0 else -1))                     # midpoints, amax 448 -> m == 1
        away = (np.sign(m) * np.inf).astype(np.float32)
        nb = np.nextafter(m, np.float32(0)) if r != 2 else np.nextafter(m, away)
        nb[-2:] = [448.0, -448.0]
        t.append(nb.astype(np.float32))                         # midpoint neighbours
        sub = g.uniform(2.0 ** -11, 2.0 ** -6, 128).astype(np.float32)
        sub[0] = 448.0
        t.append(sub * np.float32(2.0 ** (r - 1)))              # E4M3 subnormal codes
        t.append((g.standard_normal(128) * 1e-40).astype(np.float32))  # FP32 subnormals
        t.append((g.standard_normal(128) * 1e-30).astype(np.float32))  # below the amax floor
        t.append((g.standard_normal(128) * 1e37).astype(np.float32))   # near FP32 max
        p2 = (g.uniform(-1, 1, 128) * 56).astype(np.float32)
        p2[3] = 56.0                                            # amax/448 == 2^-3 exactly
        t.append(p2)
        p3 = p2.copy()
        p3[3] = np.nextafter(np.float32(56.0), np.float32(100))  # just above a power of two
        t.append(p3)
        t.append(g.standard_normal(128).astype(np.float32) * np.float32(10.0 ** (r - 1)))
        rows.append(np.concatenate(t))
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("pow2", [False, True])
def test_edge_tiles_f32_source(cuda_lib, pow2):
    x = edge_tiles()
    q, s = cuda_lib.act_quant(H.to_dev(x), pow2=pow2)
    _assert_same(q, s, *oracle.act_quant(x, pow2=pow2))


@pytest.mark.parametrize("pow2", [False, True])
def test_edge_tiles_bf16_source(cuda_lib, pow2):
    xb = synth.f32_to_bf16(edge_tiles())
    q, s = cuda_lib.act_quant(xb.cuda(), pow2=pow2)
    _assert_same(q, s, *oracle.act_quant(H.f32(xb), pow2=pow2))


@pytest.mark.parametrize("M", [1, 3, 129, 1000])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ragged_rows(cuda_lib, M, dtype):
    z = synth.normal_f32((M, 640), 1.0, 7, M, outlier_p=0.02, outlier_mult=30.0)
    x = torch.from_numpy(z).to(dtype)
    q, s = cuda_lib.act_quant(x.cuda())
    _assert_same(q, s, *oracle.act_quant(x.float().numpy()))


def test_tiny_workload_and_guards(cuda_lib):
    case = synth.dense_case("tiny")
    for t in (case.x(), case.w()):
        x = t.cuda()
        M, K = x.shape
        raw_q, q = H.guarded_empty((M, K), torch.uint8)
        raw_s, s = H.guarded_empty((M, K // 128), torch.float32)
        st = cuda_lib.load().fp8_act_quant(x.data_ptr(), 0, M, K, q.data_ptr(), s.data_ptr(), 0,
                                           torch.cuda.current_stream().cuda_stream)
        assert st == 0
        torch.cuda.synchronize()
        assert H.guards_intact(raw_q) and H.guards_intact(raw_s)
        _assert_same(q, s, *oracle.act_quant(H.f32(t)))


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_transposed_mode(cuda_lib, pow2, dtype):
    z = synth.normal_f32((384, 640), 1.0, 3, 9, outlier_p=0.01, outlier_mult=40.0)
    x = torch.from_numpy(z).to(dtype)
    qt, st = cuda_lib.act_quant(x.cuda(), pow2=pow2, transpose=True)
    assert qt.shape == (640, 384) and st.shape == (640, 3)
    _assert_same(qt, st, *oracle.act_quant_t(x.float().numpy(), pow2=pow2))


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_weight_blocks_with_transpose(cuda_lib, pow2, dtype):
    z = synth.normal_f32((384, 640), 0.02, 4, 11, outlier_p=0.001, outlier_mult=100.0)
    w = torch.from_numpy(z).to(dtype)
    N, K = w.shape
    d = w.cuda()
    raws = [H.guarded_empty(shp, dt) for shp, dt in (((N, K), torch.uint8),
                                                     ((N // 128, K // 128), torch.float32),
                                                     ((K, N), torch.uint8),
                                                     ((K // 128, N // 128), torch.float32))]
    q, s, qt, st = (b for _, b in raws)
    rc = cuda_lib.load().fp8_weight_quant(d.data_ptr(), 0 if dtype == torch.bfloat16 else 1, N, K,
                                          q.data_ptr(), s.data_ptr(), qt.data_ptr(), st.data_ptr(),
                                          1 if pow2 else 0,
                                          torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert all(H.guards_intact(r) for r, _ in raws)
    q_ref, s_ref, qt_ref, st_ref = oracle.weight_quant(w.float().numpy(), pow2=pow2, transposed=True)
    _assert_same(q, s, q_ref, s_ref)
    _assert_same(qt, st, qt_ref, st_ref)


def test_fprop_workload_full_size(cuda_lib):
    """X 4096x7168 (1x128) and W 18432x7168 (128x128), every code and scale."""
    case = synth.dense_case("fprop")
    x, w = case.x(), case.w()
    q, s = cuda_lib.act_quant(x.cuda())
    _assert_same(q, s, *H.oracle_act_quant_rows(H.f32(x)))
    qw, sw, qwt, swt = cuda_lib.weight_quant(w.cuda(), transposed=True)
    q_ref, s_ref = H.oracle_weight_quant(H.f32(w))
    _assert_same(qw, sw, q_ref, s_ref)
    _assert_same(qwt, swt, np.ascontiguousarray(q_ref.T), np.ascontiguousarray(s_ref.T))


def test_backward_workload_full_size(cuda_lib):
    """dY 4096x18432: 1x128 rows for Dgrad, 128x1 columns for Wgrad; X^T for Wgrad."""
    dy = synth.dy_bf16()
    q, s = cuda_lib.act_quant(dy.cuda())
    _assert_same(q, s, *H.oracle_act_quant_rows(H.f32(dy)))
    qt, st = cuda_lib.act_quant(dy.cuda(), transpose=True)
    _assert_same(qt, st, *H.oracle_act_quant_cols(H.f32(dy)))
    x = synth.dense_case("fprop").x()
    qt, st = cuda_lib.act_quant(x.cuda(), transpose=True)
    _assert_same(qt, st, *H.oracle_act_quant_cols(H.f32(x)))


def test_moe_inputs_pow2_full_size(cuda_lib):
    """Routed-expert inputs on power-of-2 scales: tokens 8192x7168 and h 65536x2048."""
    case = synth.MOE_FULL
    tok = case.tokens()
    q, s = cuda_lib.act_quant(tok.cuda(), pow2=True)
    _assert_same(q, s, *H.oracle_act_quant_rows(H.f32(tok), pow2=True))
    h = synth.swiglu_like_bf16((case.rows, case.I), case.seed)
    q, s = cuda_lib.act_quant(h.cuda(), pow2=True)
    _assert_same(q, s, *H.oracle_act_quant_rows(H.f32(h), pow2=True))


# ------------------------------------------------- backward re-quantisation (128x1 from FP8)
def _stored_codes(M, K, seed, pow2=False):
    z = synth.normal_f32((M, K), 1.0, seed, 77, outlier_p=0.01, outlier_mult=60.0)
    return oracle.act_quant(z, pow2=pow2)


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("M,K", [(128, 128), (384, 640), (256, 1152)])
def test_requant_transpose(cuda_lib, M, K, pow2):
    q, s = _stored_codes(M, K, M + K)
    raws = [H.guarded_empty(shp, dt) for shp, dt in (((K, M), torch.uint8),
                                                     ((K, M // 128), torch.float32))]
    qt, st = (b for _, b in raws)
    q_d, s_d = H.to_dev(q), H.to_dev(s)          # keep the inputs alive across the launch
    rc = cuda_lib.load().fp8_requant_transpose(q_d.data_ptr(), s_d.data_ptr(), M, K,
                                               qt.data_ptr(), st.data_ptr(), 1 if pow2 else 0,
                                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert all(H.guards_intact(r) for r, _ in raws)
    _assert_same(qt, st, *oracle.requant_t(q, s, pow2=pow2))


def test_requant_transpose_worked_block(cuda_lib):
    # the hand-worked block of tests/golden/requant_t_worked.txt
    q = np.empty((128, 256), np.uint8)
    q[:, :128] = 0x38
    q[:, 128::2] = 0x3C
    q[:, 129::2] = 0xBC
    s = np.empty((128, 2), np.float32)
    s[:, 0] = 2.0 ** (np.arange(128) % 8)
    s[:, 1] = 0.25
    for pow2 in (False, True):
        qt, st = cuda_lib.requant_transpose(H.to_dev(q), H.to_dev(s), pow2=pow2)
        _assert_same(qt, st, *oracle.requant_t(q, s, pow2=pow2))


def test_requant_transpose_edge_codes(cuda_lib):
    # every finite code (signed zeros, subnormal codes, +-448) with widely
    # different row scales, including scales that make the products subnormal
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]                       # drop the NaN codes
    g = np.random.default_rng(8)
    q = codes[g.integers(0, codes.size, (256, 256))].astype(np.uint8)
    s = np.exp2(g.integers(-140, 60, (256, 2))).astype(np.float32)
    s[5] = 0.0
    qt, st = cuda_lib.requant_transpose(H.to_dev(q), H.to_dev(s))
    _assert_same(qt, st, *oracle.requant_t(q, s))


def test_requant_transpose_full_size(cuda_lib):
    """The stored Fprop input X 4096x7168 (1x128) re-quantised for the Wgrad GEMM."""
    x = synth.dense_case("fprop").x()
    q, s = cuda_lib.act_quant(x.cuda())
    qt, st = cuda_lib.requant_transpose(q, s)
    q_r, s_r = H.oracle_act_quant_rows(H.f32(x))
    assert np.array_equal(q.cpu().numpy(), q_r)
    qt_r = np.empty((7168, 4096), np.uint8)
    st_r = np.empty((7168, 32), np.float32)
    for c in range(0, 7168, 1024):       # column groups of the oracle (tiles never cross columns)
        qt_r[c:c + 1024], st_r[c:c + 1024] = oracle.requant_t(q_r[:, c:c + 1024], s_r[:, c // 128:(c + 1024) // 128])
    _assert_same(qt, st, qt_r, st_r)

"""How much does the promotion buy on B300?  (page 2, inprokorea.com free #735329:
accumulation-precision passage and Figure 6; next-row study.)

Operands of the K-sweep workload (2048 x 2048 x K, N(0,1) with Student-t
outliers) are quantised with ONE scale per tensor, so that the promoted GEMM
(every 128-K partial scaled and added in FP32) and the study mode without
promotion (all of K inside the tensor core, FP8FG_WHOLE_K) compute the same
mathematical sum; the oracle gives it exactly on sampled rows.  The 14-bit
aligned-accumulation model of the pages' H800 statement runs on a smaller
sample for comparison.  The test prints one line per K (run with -s) and
asserts only what must hold: the promoted result within the FP32 tolerance,
and both errors finite and below 5 %.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import accumulation, e4m3
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _per_tensor(x):
    a = np.float32(np.abs(x).max())
    s = np.float32(a / np.float32(448.0))
    m = np.float32(np.float32(448.0) / a)
    return e4m3.encode((x * m).astype(np.float32)), s


@pytest.mark.parametrize("K", [4096, 8192, 16384])
def test_whole_k_accumulation_error(cuda_lib, K):
    case = synth.dense_case(f"ksweep{K}")
    x, w = H.f32(case.x()), H.f32(case.w())
    qa, s_a = _per_tensor(x)
    qb, s_b = _per_tensor(w)
    M, N = qa.shape[0], qb.shape[0]
    sa = np.full((M, K // 128), s_a, np.float32)
    sb = np.full((N // 128, K // 128), s_b, np.float32)
    d = [H.to_dev(v) for v in (qa, sa, qb, sb)]
    promoted = cuda_lib.gemm(*d, out_dtype=torch.float32).cpu().numpy()
    whole = cuda_lib.gemm(*d, out_dtype=torch.float32, whole_k=True).cpu().numpy()
    rows = np.array([0, 1, 517, 1024, 2047])
    ref = oracle.gemm(qa[rows], sa[rows], qb, sb)
    scale = np.abs(ref).max()

    def errs(c):
        e = c.astype(np.float64) - ref
        return np.linalg.norm(e) / np.linalg.norm(ref), np.abs(e).max() / scale

    p_norm, p_max = errs(promoted[rows])
    w_norm, w_max = errs(whole[rows])
    # the aligned-accumulation model on 2 rows x 64 columns: 14 bits (the
    # pages' H800 statement) and the width whose error is closest to B300's
    A = e4m3.decode(qa[rows[:2]]) * np.float64(s_a)
    B = e4m3.decode(qb[:64]) * np.float64(s_b)
    r_s = ref[:2, :64]
    w_s = np.linalg.norm(whole[rows[:2], :64].astype(np.float64) - r_s) / np.linalg.norm(r_s)

    def model_err(bits):
        m = accumulation.aligned_dot_rows(A, B, bits=bits, group=32)
        return np.linalg.norm(m - r_s) / np.linalg.norm(r_s), np.abs(m - r_s).max() / np.abs(r_s).max()

    e14, e14_max = model_err(14)
    fits = {b: model_err(b)[0] for b in range(18, 27)}
    best = min(fits, key=lambda b: abs(np.log(max(fits[b], 1e-30)) - np.log(max(w_s, 1e-30))))
    print(f"\nK={K}: promoted normwise {p_norm:.2e} max/|C|max {p_max:.2e}; "
          f"whole-K (B300 tensor core) normwise {w_norm:.2e} max/|C|max {w_max:.2e}; "
          f"14-bit model normwise {e14:.2e} max/|C|max {e14_max:.2e}; "
          f"on the model's sample B300 whole-K {w_s:.2e} is closest to {best} bits "
          f"({', '.join(f'{b}:{e:.1e}' for b, e in fits.items())})")
    assert p_norm <= 1e-5
    assert np.isfinite(w_norm) and w_norm < 0.05 and w_max < 0.05


@pytest.mark.parametrize("M,N,K", [(1, 128, 256), (129, 384, 640), (300, 256, 1152)])
def test_whole_k_mode_small_ragged_shapes(cuda_lib, M, N, K):
    # the study mode on ragged shapes: one scale per tensor (only sa[0, 0] and
    # sb[0, 0] are read), rows past M untouched, result within FP32-level
    # accumulation error of the exact sum
    g = np.random.default_rng(M + N + K)
    qa = e4m3.encode((g.standard_normal((M, K)) * 50).astype(np.float32))
    qb = e4m3.encode((g.standard_normal((N, K)) * 50).astype(np.float32))
    s_a, s_b = np.float32(0.0123), np.float32(3.5)
    sa = np.full((M, K // 128), s_a, np.float32)
    sb = np.full((N // 128, K // 128), s_b, np.float32)
    sa_dev = H.to_dev(sa.copy())
    sa_dev.view(-1)[1:] = 7.0                      # only the first scale may be read
    sb_dev = H.to_dev(sb.copy())
    sb_dev.view(-1)[1:] = 7.0
    raw, out = H.guarded_empty((M, N), torch.float32)
    cuda_lib.gemm(H.to_dev(qa), sa_dev, H.to_dev(qb), sb_dev, out_dtype=torch.float32,
                  whole_k=True, out=out)
    torch.cuda.synchronize()
    assert H.guards_intact(raw), "write outside the output"
    ref = oracle.gemm(qa, sa, qb, sb)
    assert H.normwise_rel_err(out, ref) <= 1e-5

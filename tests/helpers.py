"""Shared helpers for the parity tests (oracle side on the CPU, library side on the GPU)."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

GUARD = 4096      # bytes of canary on each side of a guarded output


def oracle_act_quant_rows(x_f32: np.ndarray, pow2=False, rows_per_chunk=2048):
    """oracle.act_quant over row chunks (tiles never cross rows, so this is exact)."""
    M, K = x_f32.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, K // 128), np.float32)
    for r in range(0, M, rows_per_chunk):
        q[r:r + rows_per_chunk], s[r:r + rows_per_chunk] = oracle.act_quant(
            x_f32[r:r + rows_per_chunk], pow2=pow2)
    return q, s


def oracle_act_quant_cols(x_f32: np.ndarray, pow2=False, cols_per_chunk=1024):
    """oracle.act_quant_t over column chunks (tiles never cross columns)."""
    M, K = x_f32.shape
    qt = np.empty((K, M), np.uint8)
    st = np.empty((K, M // 128), np.float32)
    for c in range(0, K, cols_per_chunk):
        qt[c:c + cols_per_chunk], st[c:c + cols_per_chunk] = oracle.act_quant_t(
            np.ascontiguousarray(x_f32[:, c:c + cols_per_chunk]), pow2=pow2)
    return qt, st


def oracle_weight_quant(w_f32: np.ndarray, pow2=False, rows_per_chunk=1024):
    """oracle.weight_quant over strips of whole 128-row blocks."""
    N, K = w_f32.shape
    q = np.empty((N, K), np.uint8)
    s = np.empty((N // 128, K // 128), np.float32)
    for r in range(0, N, rows_per_chunk):
        q[r:r + rows_per_chunk], s[r // 128:(r + rows_per_chunk) // 128] = oracle.weight_quant(
            w_f32[r:r + rows_per_chunk], pow2=pow2)
    return q, s


def normwise_rel_err(c_gpu, c_ref: np.ndarray) -> float:
    g = c_gpu.detach().float().cpu().numpy().astype(np.float64) if isinstance(c_gpu, torch.Tensor) \
        else np.asarray(c_gpu, np.float64)
    return float(np.linalg.norm(g - c_ref) / np.linalg.norm(c_ref))


def to_dev(a, dev="cuda"):
    if isinstance(a, torch.Tensor):
        return a.to(dev).contiguous()
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def guarded_empty(shape, dtype, fill_byte=0xA5, dev="cuda"):
    """An output tensor with canary bytes before and after it in one allocation."""
    nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((GUARD + nbytes + GUARD,), fill_byte, dtype=torch.uint8, device=dev)
    body = raw[GUARD:GUARD + nbytes].view(dtype).view(shape)
    return raw, body


def guards_intact(raw: torch.Tensor, fill_byte=0xA5) -> bool:
    head = raw[:GUARD]
    tail = raw[-GUARD:]
    return bool((head == fill_byte).all().item() and (tail == fill_byte).all().item())


def f32(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_to_f32(t)


def oracle_gemm_chunked(qa, sa, qb, sb, b_tile=False, chunk=2048) -> np.ndarray:
    """oracle.gemm over column chunks of B (output columns are independent)."""
    N = qb.shape[0]
    parts = []
    for c0 in range(0, N, chunk):
        c1 = min(N, c0 + chunk)
        sbc = sb[c0:c1] if b_tile else sb[c0 // 128:(c1 + 127) // 128]
        parts.append(oracle.gemm(qa, sa, qb[c0:c1], sbc, b_tile=b_tile))
    return np.concatenate(parts, axis=1)


_E4M3_MAGS = None


def check_quant_decisions(q_gpu, s_gpu, x_ref, err, pow2):
    """Compare GPU 1x128-tile quantisation of values the GPU computed with rounding
    error against the oracle's quantisation of the exact values.

    x_ref: oracle float32 values [M, N]; err: per-element bound on |x_gpu - x_ref|
    (float64 [M, N]).  Scales must agree within the amax's share of err
    (exactly for power-of-2 scales unless amax/448 lies that close to a power of
    two); codes must equal the oracle's unless x * m lies within the error of an
    E4M3 rounding midpoint, where either neighbour is correct; every code must
    decode to within one E4M3 step of x.  Returns the fraction of codes decided.
    """
    import oracle
    from oracle import e4m3

    global _E4M3_MAGS
    if _E4M3_MAGS is None:
        _E4M3_MAGS = np.unique(np.abs(e4m3.decode(np.arange(0x7F, dtype=np.uint8))))
    mags = _E4M3_MAGS
    q_o, s_o = oracle.act_quant(x_ref, pow2)
    M, N = q_o.shape
    xt = x_ref.astype(np.float64).reshape(M, N // 128, 128)
    Et = np.asarray(err, dtype=np.float64).reshape(M, N // 128, 128)
    so = s_o.astype(np.float64)
    sg = np.asarray(s_gpu, dtype=np.float64)
    amax = np.abs(xt).max(axis=2)
    e_amax = Et.max(axis=2)
    if not pow2:
        tol = amax / 448.0 * 2.0 ** -22 + e_amax / 448.0 * 1.01
        assert np.all(np.abs(sg - so) <= tol), "scale outside the error bound"
    else:
        lo2 = np.log2(np.maximum((amax - e_amax) / 448.0, 2.0 ** -80))
        hi2 = np.log2((amax + e_amax) / 448.0 * (1 + 2.0 ** -22))
        ambiguous = np.ceil(lo2) != np.ceil(hi2)
        assert np.all((sg == so) | ambiguous), "power-of-2 scale differs away from a power of 2"
    m = 1.0 / so[:, :, None]
    y = np.abs(xt) * m
    idx = np.clip(np.searchsorted(mags, y), 1, len(mags) - 1)
    mid_hi = (mags[idx - 1] + mags[idx]) / 2
    mid_lo = (mags[np.clip(idx - 2, 0, None)] + mags[idx - 1]) / 2
    near = np.minimum(np.abs(y - mid_hi), np.abs(y - mid_lo))
    slack = Et * m * 1.01 + y * 2.0 ** -21 + np.abs(sg[:, :, None] / so[:, :, None] - 1) * y
    sure = (near > slack).reshape(M, N)
    qg = np.asarray(q_gpu).reshape(M, N)
    assert np.array_equal(qg[sure], q_o[sure]), "code differs where the rounding is decided"
    dq = e4m3.decode(qg).astype(np.float64).reshape(M, N // 128, 128) * sg[:, :, None]
    step = (np.maximum(y, 2.0 ** -6) * 2.0 ** -3 + 2.0 ** -9) * so[:, :, None]
    assert np.all(np.abs(dq - xt) <= step + Et), "code off by more than one step"
    return float(sure.mean())


def gemm_error_bound(qa, sa, qb, sb, b_tile=False, extra_adds=0) -> np.ndarray:
    """Per-element bound on |C32 - C| for the promoted FP32 sum (float64 [M, N]).

    C = sum_kb P_kb * s_kb is the oracle's exact result (s_kb = sa[m,kb] * sb(n,kb)).
    The GPU forms each group's partial T_kb in the tensor core (FP32 accumulation
    of four K=32 products into TMEM), rounds s_kb to FP32, and adds T_kb * s_kb
    into an FP32 accumulator with one rounding per group (page 2,
    inprokorea.com free #735329, promotion passage and Figure 6).  With
    A1 = sum_kb |P_kb| s_kb and A2 = sum_kb s_kb sum_{k in kb} |a_k b_k|:
      * group partials: |T_kb - P_kb| <= 8 * 2^-24 * sum_{k in kb} |a_k b_k|
        (four K=32 accumulation steps; B300's FP8 accumulation measured like an
        aligned sum truncated to 25-26 significant bits, so each step loses at
        most 2^-23 of the magnitude it aligns to, itself at most the group's
        sum of |products|);
      * the scale product: 2^-24 |P_kb s_kb|;
      * the FP32 accumulation: at most nkb roundings of 2^-24 of a running sum
        bounded by A1.
    Hence |C32 - C| <= (nkb + 1) 2^-24 A1 + 8 * 2^-24 A2 (second-order terms are
    far below the first-order slack).  A single wrong element (a dropped group, a
    wrong scale) misses it by orders of magnitude.

    extra_adds: FP32 additions of partial sums beyond the per-group ones (a tile
    whose groups were split among CTAs is summed from its parts: one addition per
    extra part, each within 2^-24 of a magnitude bounded by A1).
    """
    qa = np.asarray(qa)
    qb = np.asarray(qb)
    M, K = qa.shape
    N = qb.shape[0]
    nkb = K // 128
    sa64 = np.asarray(sa, np.float64)
    sb64 = np.asarray(sb, np.float64)
    mag_a, mag_b = qa & 0x7F, qb & 0x7F          # |decode(c)| = decode(c & 0x7F) (no NaN codes)
    A1 = np.zeros((M, N))
    A2 = np.zeros((M, N))
    for kb in range(nkb):
        sl = slice(128 * kb, 128 * (kb + 1))
        P = oracle.slice_partials(qa[:, sl], qb[:, sl])[0]
        Q = oracle.slice_partials(mag_a[:, sl], mag_b[:, sl])[0]
        sbk = sb64[:, kb] if b_tile else np.repeat(sb64[:, kb], 128)[:N]
        s = sa64[:, kb][:, None] * sbk[None, :]
        A1 += np.abs(P) * s
        A2 += Q * s
    return (nkb + 1 + extra_adds) * 2.0 ** -24 * A1 + 8 * 2.0 ** -24 * A2


def grouped_error_bound(qa, sa, offsets, qb, sb) -> np.ndarray:
    """gemm_error_bound per expert over contiguous row groups (float64 [T, N])."""
    off = np.asarray(offsets, np.int64)
    out = np.zeros((np.asarray(qa).shape[0], np.asarray(qb).shape[1]))
    for e in range(len(off) - 1):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            out[r0:r1] = gemm_error_bound(qa[r0:r1], np.asarray(sa)[r0:r1], qb[e], sb[e])
    return out


def assert_elementwise(c_gpu, c_ref: np.ndarray, bound32: np.ndarray, what: str = "") -> float:
    """Every element of the GPU result within its bound (FP32 output), or within the
    bound plus one BF16 rounding of the FP32 value (2^-8 of it, RNE) for BF16 output.
    Returns the largest |error| / bound."""
    is_bf16 = isinstance(c_gpu, torch.Tensor) and c_gpu.dtype == torch.bfloat16
    g = c_gpu.detach().float().cpu().numpy().astype(np.float64) if isinstance(c_gpu, torch.Tensor) \
        else np.asarray(c_gpu, np.float64)
    bound = bound32 + (2.0 ** -8 * (np.abs(c_ref) + bound32) if is_bf16 else 0.0)
    err = np.abs(g - c_ref)
    bad = err > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside the per-element bound; "
                             f"first at {list(i)}: gpu {g[i]!r} ref {c_ref[i]!r} bound {bound[i]!r}")
    return float((err / np.maximum(bound, 1e-300)).max())

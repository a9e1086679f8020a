"""Fine-grained E4M3 quantisation, as the pages define it.  TEST INFRASTRUCTURE ONLY.

Sources (page, passage):
  * tile shapes -- page 1 (xn--9g3bo1gtkw0l8ubf92bgle.kr qna #85187), Figure 7 (a):
    activations are grouped per token per 128 channels (1x128 tiles), weights
    per 128 input x 128 output channels (128x128 blocks);
  * scales stored as float32 next to the data -- page 1, "Storage Format" passage;
  * online amax per 1x128 tile / 128x128 block -- page 2 (inprokorea.com free
    #735329), fine-grained quantisation passage;
  * scales folded in at dequantisation, per group along K -- page 2, same passage;
  * integral power-of-2 scales for some activations -- page 1 and page 2,
    passage on the inputs of the Linear after attention / MoE up-projection;
  * backward re-quantisation into 128x1 tiles -- page 5 (inprokorea.com free
    #890463), passage on the backward pass.

Readings where the pages are silent (the pages give the tile shapes, the
online amax and the FP32 scale storage, but no formula):
  * amax' = max(amax, 2^-64): an all-zero or tiny tile still gets a finite,
    nonzero scale (the floor never binds on the workloads' data);
  * the stored scale is the dequantisation scale, s = fl32(amax'/448), so the
    tile amax maps to exactly +-448 (E4M3's largest finite value) and
    x ~ decode(q) * s, the direction in which page 2 multiplies it in;
  * the codes are encode(fl32(x * fl32(448/amax'))): one rounded multiply per
    element, not a division x/s;
  * power-of-2 mode rounds up, s = 2^ceil(log2(fl32(amax'/448))), so no scaled
    value exceeds 448; its multiplier 1/s is exact;
  * E4M3 rounding is to nearest even, saturating to +-448, keeping the sign of
    zero (e4m3.encode).
"""

from __future__ import annotations

import numpy as np

from .e4m3 import E4M3_MAX, decode, encode

TILE = 128
AMAX_FLOOR = np.float32(2.0 ** -64)


def scale_from_amax(amax, pow2: bool = False):
    """amax (float32 array) -> (dequant scale s, quant multiplier m), both float32."""
    a = np.maximum(np.asarray(amax, dtype=np.float32), AMAX_FLOOR)
    q = np.float32(E4M3_MAX)
    t = (a / q).astype(np.float32)                    # IEEE float32 division
    if not pow2:
        m = (q / a).astype(np.float32)
        return t, m
    mt, et = np.frexp(t.astype(np.float64))          # t = mt * 2^et, mt in [0.5, 1)
    exp = np.where(mt == 0.5, et - 1, et)            # ceil(log2 t)
    s = np.ldexp(1.0, exp).astype(np.float32)
    m = np.ldexp(1.0, -exp).astype(np.float32)
    return s, m


def _quant_groups(g: np.ndarray, axis: int, pow2: bool):
    """Quantise float32 array g with one scale per slice along `axis`."""
    amax = np.max(np.abs(g), axis=axis, keepdims=True).astype(np.float32)
    s, m = scale_from_amax(amax, pow2)
    y = (g * m).astype(np.float32)                    # one IEEE float32 multiply
    return encode(y), s


def act_quant(x, pow2: bool = False):
    """1x128 tiles along K.  x: float32 [M, K] -> (q uint8 [M, K], s float32 [M, K/128])."""
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    if K % TILE:
        raise ValueError("K must be a multiple of 128")
    g = x.reshape(M, K // TILE, TILE)
    q, s = _quant_groups(g, axis=2, pow2=pow2)
    return q.reshape(M, K), s.reshape(M, K // TILE)


def act_quant_t(x, pow2: bool = False):
    """128x1 tiles along M, output transposed.

    x: float32 [M, K] (M % 128 == 0) -> (qt uint8 [K, M], st float32 [K, M/128]),
    where column k of x, rows 128i..128i+127, forms one tile with scale st[k, i].
    """
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    if M % TILE:
        raise ValueError("M must be a multiple of 128 in transposed mode")
    g = x.reshape(M // TILE, TILE, K)
    q, s = _quant_groups(g, axis=1, pow2=pow2)       # q [M/128,128,K], s [M/128,1,K]
    qt = np.ascontiguousarray(q.reshape(M, K).T)
    st = np.ascontiguousarray(s.reshape(M // TILE, K).T)
    return qt, st


def weight_quant(w, pow2: bool = False, transposed: bool = False):
    """128x128 blocks.  w: float32 [N, K] (N, K % 128 == 0).

    Returns (q uint8 [N, K], s float32 [N/128, K/128]) and, when `transposed`,
    also (qt [K, N], st [K/128, N/128]) -- the same codes and scales transposed.
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    if N % TILE or K % TILE:
        raise ValueError("N and K must be multiples of 128")
    g = w.reshape(N // TILE, TILE, K // TILE, TILE)
    q, s = _quant_groups(g, axis=(1, 3), pow2=pow2)
    q = q.reshape(N, K)
    s = s.reshape(N // TILE, K // TILE)
    if not transposed:
        return q, s
    return q, s, np.ascontiguousarray(q.T), np.ascontiguousarray(s.T)


def requant_t(q, s, pow2: bool = False):
    """Backward re-quantisation of stored 1x128 codes into transposed 128x1 tiles.

    Page 5 (inprokorea.com free #890463), backward-pass passage: the FP8
    activations kept from the forward pass are read, dequantised, transposed
    and quantised again in 128x1 tiles for the weight gradient.
    q: uint8 [M, K] E4M3 codes with 1x128 scales s: float32 [M, K/128] (the
    layout act_quant produces); M % 128 == 0.  Each element is dequantised in
    float32 with one IEEE multiply, x = fl32(decode(q[r, k]) * s[r, k // 128])
    (E4M3 values are exact in float32), and x is then quantised exactly as
    act_quant_t.  Returns (qt uint8 [K, M], st float32 [K, M/128]).
    """
    q = np.asarray(q)
    M, K = q.shape
    if K % TILE or M % TILE:
        raise ValueError("M and K must be multiples of 128")
    v = decode(q).astype(np.float32)
    sc = np.repeat(np.asarray(s, dtype=np.float32), TILE, axis=1)[:, :K]
    x = (v * sc).astype(np.float32)                  # one IEEE float32 multiply
    return act_quant_t(x, pow2=pow2)


def dequant_tiles(q, s) -> np.ndarray:
    """Inverse of act_quant (float64): x_hat[r, k] = decode(q[r, k]) * s[r, k // 128]."""
    v = decode(q)
    return v * np.repeat(np.asarray(s, dtype=np.float64), TILE, axis=1)[:, : v.shape[1]]


def dequant_blocks(q, s) -> np.ndarray:
    """Inverse of weight_quant (float64)."""
    v = decode(q)
    sb = np.repeat(np.repeat(np.asarray(s, dtype=np.float64), TILE, axis=0), TILE, axis=1)
    return v * sb[: v.shape[0], : v.shape[1]]

"""Seeded synthetic workloads for the fine-grained FP8 path.

Recipe (one for every workload):

* Each tensor has its own PCG64 stream, ``numpy.random.default_rng([seed, tag])``,
  so any single tensor (one expert's weight, say) can be regenerated alone.
* Values are float32 draws ``standard_normal * std``.  Outliers are an
  independent Bernoulli(p) mask drawn after the values; a masked entry is either
  multiplied by a factor or replaced by a Student-t draw.
* The float32 values are rounded to BF16 (round-to-nearest-even, torch CPU), and
  those BF16 bytes are what both the GPU path and the oracle receive.

The five workloads mirror the DeepSeek-V3 FP8 training passages: a tiny dense
case, the FFN Fprop at hidden 7168 / inter 18432, the matching Dgrad/Wgrad,
the routed-expert MoE layer (256 experts, top-8, expert hidden 2048) and a
K sweep for accumulation precision.

The MoE expert weights of the full-size layer (11 G values) are too many to
draw on the host in reasonable time; ``expert_weight(..., device="cuda")``
draws them with torch's device Philox generator from a per-expert seed.  A test
that checks some experts on the CPU copies exactly those BF16 bytes back.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = [
    "TAG_X", "TAG_W", "TAG_DY", "TAG_ROUTER", "TAG_BIAS", "TAG_TOKENS", "TAG_H",
    "TAG_EXPERT_UP", "TAG_EXPERT_DOWN",
    "rng", "normal_f32", "normal_bf16", "bf16_to_f32", "f32_to_bf16",
    "DenseCase", "dense_case", "DENSE_CASES", "MoECase", "MOE_FULL", "MOE_SMALL",
    "moe_route", "expert_weight", "swiglu_like_bf16", "ragged_offsets",
]

TAG_X, TAG_W, TAG_DY, TAG_ROUTER, TAG_BIAS, TAG_TOKENS, TAG_H = 1, 2, 3, 4, 5, 6, 7
TAG_EXPERT_UP, TAG_EXPERT_DOWN = 1000, 2000


def rng(seed: int, tag: int) -> np.random.Generator:
    """Independent PCG64 stream for one named tensor."""
    return np.random.default_rng([int(seed), int(tag)])


def normal_f32(shape, std: float, seed: int, tag: int, outlier_p: float = 0.0,
               outlier_mult: float | None = None, outlier_t_nu: float | None = None
               ) -> np.ndarray:
    """float32 N(0, std^2) draws with optional outliers (see module recipe)."""
    g = rng(seed, tag)
    z = g.standard_normal(shape, dtype=np.float32)
    z *= np.float32(std)
    if outlier_p > 0.0:
        mask = g.random(shape) < outlier_p
        if outlier_t_nu is not None:
            z[mask] = g.standard_t(outlier_t_nu, size=int(mask.sum())).astype(np.float32)
        elif outlier_mult is not None:
            z[mask] *= np.float32(outlier_mult)
    return z


def f32_to_bf16(z: np.ndarray) -> torch.Tensor:
    """Round float32 to BF16 (RNE) on the CPU; returns a contiguous CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(z)).to(torch.bfloat16)


def bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    """Exact widening of BF16 (or float32) values to a float32 numpy array."""
    return t.detach().to("cpu").float().numpy()


def normal_bf16(shape, std, seed, tag, **kw) -> torch.Tensor:
    return f32_to_bf16(normal_f32(shape, std, seed, tag, **kw))


# --------------------------------------------------------------------------- dense
@dataclass(frozen=True)
class DenseCase:
    """One dense GEMM workload: C[M,N] = X[M,K] . W[N,K]^T."""
    name: str
    M: int
    N: int
    K: int
    x_std: float = 1.0
    w_std: float = 1.0
    x_outlier: dict = field(default_factory=dict)
    w_outlier: dict = field(default_factory=dict)
    out: str = "f32"        # output dtype of the GEMM: "f32" or "bf16"
    seed: int = 0

    def x(self) -> torch.Tensor:
        return normal_bf16((self.M, self.K), self.x_std, self.seed, TAG_X, **self.x_outlier)

    def w(self) -> torch.Tensor:
        return normal_bf16((self.N, self.K), self.w_std, self.seed, TAG_W, **self.w_outlier)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


DENSE_CASES = {
    # tiny dense: both operands N(0,1) with 1% of entries scaled x50
    "tiny": DenseCase("tiny", 256, 256, 512, 1.0, 1.0,
                      dict(outlier_p=0.01, outlier_mult=50.0),
                      dict(outlier_p=0.01, outlier_mult=50.0), out="f32"),
    # Fprop at the DeepSeek-V3 FFN width: X 4096x7168 (0.1% x100), W 18432x7168 N(0,0.02)
    "fprop": DenseCase("fprop", 4096, 18432, 7168, 1.0, 0.02,
                       dict(outlier_p=0.001, outlier_mult=100.0), {}, out="bf16"),
    # K sweep: N(0,1) with 0.5% Student-t(2) replacements on both operands
    "ksweep4096": DenseCase("ksweep4096", 2048, 2048, 4096, 1.0, 1.0,
                            dict(outlier_p=0.005, outlier_t_nu=2.0),
                            dict(outlier_p=0.005, outlier_t_nu=2.0), out="f32"),
    "ksweep8192": DenseCase("ksweep8192", 2048, 2048, 8192, 1.0, 1.0,
                            dict(outlier_p=0.005, outlier_t_nu=2.0),
                            dict(outlier_p=0.005, outlier_t_nu=2.0), out="f32"),
    "ksweep16384": DenseCase("ksweep16384", 2048, 2048, 16384, 1.0, 1.0,
                             dict(outlier_p=0.005, outlier_t_nu=2.0),
                             dict(outlier_p=0.005, outlier_t_nu=2.0), out="f32"),
}


def dense_case(name: str) -> DenseCase:
    return DENSE_CASES[name]


def dy_bf16(M: int = 4096, N: int = 18432, seed: int = 0) -> torch.Tensor:
    """Output gradient of the FFN up-projection, N(0, 1e-3^2)."""
    return normal_bf16((M, N), 1e-3, seed, TAG_DY)


__all__.append("dy_bf16")


# ----------------------------------------------------------------------------- MoE
@dataclass(frozen=True)
class MoECase:
    """Routed-expert layer: T tokens of width H, E experts, top-k, expert inter I.

    Up-projection per expert: [2I, H] (gate rows then up rows); down: [H, I].
    """
    name: str
    T: int
    H: int
    E: int
    topk: int
    I: int
    seed: int = 0
    router_std: float = 0.02
    bias_range: float = 0.1
    w_std: float = 0.02

    @property
    def rows(self) -> int:
        return self.T * self.topk

    def tokens(self) -> torch.Tensor:
        return normal_bf16((self.T, self.H), 1.0, self.seed, TAG_TOKENS)

    def router(self) -> np.ndarray:
        return normal_f32((self.E, self.H), self.router_std, self.seed, TAG_ROUTER)

    def bias(self) -> np.ndarray:
        g = rng(self.seed, TAG_BIAS)
        return g.uniform(-self.bias_range, self.bias_range, self.E).astype(np.float32)

    def up_flops(self) -> int:
        return 2 * self.rows * (2 * self.I) * self.H

    def down_flops(self) -> int:
        return 2 * self.rows * self.H * self.I


MOE_FULL = MoECase("moe", T=8192, H=7168, E=256, topk=8, I=2048)
# small variant with the same structure that the oracle finishes in seconds
MOE_SMALL = MoECase("moe_small", T=96, H=512, E=8, topk=2, I=128)


def moe_route(tokens_f32: np.ndarray, router_f32: np.ndarray, bias_f32: np.ndarray,
              topk: int) -> dict:
    """Sigmoid-affinity top-k routing with a per-expert selection bias.

    affinity = sigmoid(x . R^T) in float32; the k experts with the largest
    affinity + bias are chosen (ties -> lower expert index).  The (token,
    expert) pairs are then ordered by expert, then token, which gives the row
    order of the grouped GEMM and the int32 offsets[E+1].
    """
    T = tokens_f32.shape[0]
    E = router_f32.shape[0]
    logits = (tokens_f32.astype(np.float32) @ router_f32.astype(np.float32).T).astype(np.float32)
    aff = (np.float32(1.0) / (np.float32(1.0) + np.exp(-logits))).astype(np.float32)
    sel = aff + bias_f32[None, :].astype(np.float32)
    order = np.argsort(-sel, axis=1, kind="stable")[:, :topk]
    tok = np.repeat(np.arange(T, dtype=np.int64), topk)
    exp = order.reshape(-1).astype(np.int64)
    perm = np.lexsort((tok, exp))
    counts = np.bincount(exp, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return dict(topk=order, token_of_row=tok[perm], expert_of_row=exp[perm],
                counts=counts, offsets=offsets)


def _expert_seed(seed: int, tag: int) -> int:
    return (int(seed) * 1_000_003 + int(tag)) & 0x7FFFFFFFFFFFFFFF


def expert_weight(case: MoECase, e: int, kind: str, device="cpu") -> torch.Tensor:
    """One expert's BF16 weight, [2I, H] for kind="up", [H, I] for kind="down".

    On the CPU this is the module's PCG64 recipe; on a CUDA device it is torch's
    Philox generator keyed by the same (seed, tag), which is what the full-size
    layer uses (the bytes are copied back for any expert the oracle checks).
    """
    if kind == "up":
        shape, tag = (2 * case.I, case.H), TAG_EXPERT_UP + e
    elif kind == "down":
        shape, tag = (case.H, case.I), TAG_EXPERT_DOWN + e
    else:
        raise ValueError(kind)
    dev = torch.device(device)
    if dev.type == "cpu":
        return normal_bf16(shape, case.w_std, case.seed, tag)
    g = torch.Generator(device=dev)
    g.manual_seed(_expert_seed(case.seed, tag))
    z = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    return (z * case.w_std).to(torch.bfloat16)


def swiglu_like_bf16(shape, seed: int, tag: int = TAG_H, std: float = 1.7) -> torch.Tensor:
    """Stand-in for the down-projection input h = silu(g) * u.

    g, u ~ N(0, std^2) with std close to that of the up-projection output
    (sqrt(7168) * 0.02 ~ 1.7).  Drawn directly so that the down-projection's
    check does not depend on the up-projection's rounding.
    """
    g = normal_f32(shape, std, seed, tag)
    u = normal_f32(shape, std, seed, tag + 100)
    h = (g / (np.float32(1.0) + np.exp(-g))) * u
    return f32_to_bf16(h.astype(np.float32))


def ragged_offsets(sizes) -> np.ndarray:
    """int32 offsets[E+1] from a list of per-expert row counts."""
    off = np.zeros(len(sizes) + 1, dtype=np.int32)
    off[1:] = np.cumsum(np.asarray(sizes, dtype=np.int64))
    return off

"""CPU oracle for fine-grained FP8 quantisation and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY.  Plain numpy, float64/int64 where precision matters,
written from the DeepSeek-V3 FP8 training passages on the five scraped pages,
cited per function as page + passage/figure: page 1 = xn--9g3bo1gtkw0l8ubf92bgle.kr
qna #85187, page 2 = inprokorea.com free #735329, page 5 = inprokorea.com free
#890463 (pages 3 and 4 hold nothing on this path).  It shares no code, header, table or constant generator
with the CUDA library, and the CUDA library never imports it.  Only the tests,
the smoke check and the benchmark's CPU-baseline leg may call it.

Pins (checked in tests/test_oracle_*.py without a GPU):
  e4m3   exhaustive over all 256 codes; round-trip; monotonicity; every
         midpoint ties to even; structured float32 sweeps against two library
         casts (ml_dtypes, torch); saturation.
  quant  amax maps to +-448 exactly; power-of-2 scale rule; error bound of
         one E4M3 half-ulp times the tile amax; a hand-worked tile fixture;
         transposed mode equals quantising the transpose; backward
         re-quantisation of stored codes against a hand-worked block and a
         two-step error bound.
  gemm   brute force in exact rationals on tiny shapes; int64 per-slice sums;
         special cases that reduce to a library matmul; scale linearity;
         Dgrad/Wgrad transposition identities.
  group  E=1 equals dense; empty experts; relabelling invariance.
  gemm_quant  (the GEMM result quantised into 1x128 E4M3 tiles) products that
         are exact E4M3 values with a 448 in every tile come back unchanged at
         scale 1; scale direction under power-of-2 operand scales; the tile
         amax takes code +-448 and every element lies within half an E4M3 step;
         an all-zero tile.
  swiglu silu against scipy's logistic and the odd identity
         silu(x) - silu(-x) = x; a worked case where silu(64) = 64 exactly makes
         h = 64 * up and the up codes come back under scale 64; swapping the
         gate and up halves changes the result; power-of-2 scales and the
         half-step bound on random tiles.
  accum  (accumulation.py, a model of limited-width aligned accumulation)
         full width is an exact sum; terms below the last kept bit vanish and
         terms at it are kept; group sums are exact before alignment; error of
         at most one truncation step per group; fewer bits, larger error.
Parity unpinned: the "about 2% error at K=4096 with ~14-bit accumulation"
figure (no mechanism detail to reproduce it); it is context only.
"""

from .e4m3 import E4M3_MAX, decode, encode  # noqa: F401
from .quant import (act_quant, act_quant_t, weight_quant, requant_t,  # noqa: F401
                    dequant_tiles, dequant_blocks, scale_from_amax)
from .scaled_gemm import (gemm, gemm_quant, grouped_gemm, grouped_swiglu_quant,  # noqa: F401
                          silu, slice_partials)

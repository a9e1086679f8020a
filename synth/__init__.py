"""Seeded synthetic inputs shared by the CUDA path and the CPU oracle.

This package holds no arithmetic of the FP8 method itself: no quantisation, no
scaling, no GEMM.  It only draws the BF16 tensors (and the MoE routing that
decides which rows meet which expert) that both sides then consume byte for
byte.
"""

from .inputs import *  # noqa: F401,F403

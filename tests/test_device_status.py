"""Failure detection without a GPU fault: bounded waits report FP8FG_ERR_TIMEOUT.

The self-test kernel waits on an mbarrier that nothing ever arrives on, with a
short cycle limit; the wait must give up, record the timeout in the library
status word and return, leaving the context usable.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import e4m3
from tests import helpers as H

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared(cuda_lib):
    assert cuda_lib.device_status() == cuda_lib.OK
    assert cuda_lib.selftest_wait_timeout(1 << 20) == cuda_lib.ERR_TIMEOUT
    assert cuda_lib.device_status() == cuda_lib.OK


def test_context_usable_after_timeout(cuda_lib):
    cuda_lib.selftest_wait_timeout(1 << 18)
    g = np.random.default_rng(0)
    qa = e4m3.encode(g.standard_normal((130, 256)).astype(np.float32) * 30)
    qb = e4m3.encode(g.standard_normal((256, 256)).astype(np.float32) * 30)
    sa = np.ones((130, 2), np.float32)
    sb = np.full((2, 2), 0.5, np.float32)
    out = cuda_lib.gemm(H.to_dev(qa), H.to_dev(sa), H.to_dev(qb), H.to_dev(sb),
                        out_dtype=torch.float32)
    assert cuda_lib.device_status() == cuda_lib.OK
    assert H.normwise_rel_err(out, oracle.gemm(qa, sa, qb, sb)) <= 1e-5


def test_long_wait_limit_does_not_fire_on_normal_work(cuda_lib):
    cuda_lib.set_wait_limit(1 << 30)
    try:
        g = np.random.default_rng(1)
        qa = e4m3.encode(g.standard_normal((512, 1024)).astype(np.float32))
        qb = e4m3.encode(g.standard_normal((512, 1024)).astype(np.float32))
        sa = np.ones((512, 8), np.float32)
        sb = np.ones((4, 8), np.float32)
        cuda_lib.gemm(H.to_dev(qa), H.to_dev(sa), H.to_dev(qb), H.to_dev(sb))
        assert cuda_lib.device_status() == cuda_lib.OK
    finally:
        cuda_lib.set_wait_limit(0)

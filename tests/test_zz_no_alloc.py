"""The allocation-free GEMM entry point, called through the C ABI.

Some callers cannot allocate device memory at the moment they run the GEMM: a
memory pool that is locked or being captured into a graph, an allocator that
must not be re-entered, a runtime whose memory budget was fixed up front.
fp8_blockscaled_gemm_noalloc gives them the stream-K GEMM with its scratch in
an array the library keeps on the device, so they pass only inputs and the
output.  Its results must match those of fp8_blockscaled_gemm_ws given a
workspace from torch, on two calls in a row (the second call finds the first
call's partial tiles in the shared array).

This file is collected last, so a run that stops at the first failure has run
every other test.  It also passes alone in a fresh process: the first call on
a device looks up the array's device address.
"""

import ctypes

import pytest
import torch

import fp8_fine_grained_19_b300 as fp8
from tests import helpers as H

TOL = {torch.float32: 1e-5, torch.bfloat16: 4e-3}
A16 = 1 << 20            # a fake, 16-byte aligned "device pointer" (never dereferenced)


def _device_operands(M, N, K, b_tile, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)

    def codes(r, c):      # E4M3 codes without NaN (0x7F / 0xFF), both signs
        mag = torch.randint(0, 0x7F, (r, c), generator=g, device="cuda", dtype=torch.int32)
        sgn = torch.randint(0, 2, (r, c), generator=g, device="cuda", dtype=torch.int32) * 0x80
        return (mag | sgn).to(torch.uint8)

    a, b = codes(M, K), codes(N, K)
    sa = torch.exp(torch.rand((M, K // 128), generator=g, device="cuda") * 6 - 3)
    sb_shape = (N, K // 128) if b_tile else (N // 128, K // 128)
    sb = torch.exp(torch.rand(sb_shape, generator=g, device="cuda") * 6 - 3)
    return a, sa, b, sb


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,b_tile,dtype,force", [
    (4096, 7168, 18432, False, torch.bfloat16, False),   # Dgrad shape: splits by itself
    (300, 768, 1280, False, torch.float32, True),         # forced split, many parts per tile
    (129, 400, 2048, True, torch.float32, True),          # 1x128 B scales
    (520, 1024, 384, False, torch.bfloat16, False),       # no split: the array is not used
])
def test_noalloc_matches_workspace_entry_point(cuda_lib, M, N, K, b_tile, dtype, force):
    lib = cuda_lib.load()
    a, sa, b, sb = _device_operands(M, N, K, b_tile, M + N + K)
    flags = (fp8.B_TILE1x128 if b_tile else 0) | (fp8.STREAM_K if force else 0)
    ct = fp8.F32 if dtype == torch.float32 else fp8.BF16
    sp = torch.cuda.current_stream().cuda_stream
    ptrs = (a.data_ptr(), sa.data_ptr(), b.data_ptr(), sb.data_ptr())

    need = lib.fp8_blockscaled_gemm_workspace_bytes(M, N, K, flags)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    ref = torch.empty((M, N), dtype=dtype, device="cuda")
    assert lib.fp8_blockscaled_gemm_ws(*ptrs, ref.data_ptr(), ct, M, N, K, flags,
                                       ws.data_ptr() if need else None, need, sp) == fp8.OK

    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=dtype, device="cuda")
        assert lib.fp8_blockscaled_gemm_noalloc(*ptrs, out.data_ptr(), ct, M, N, K, flags, sp) == fp8.OK
        torch.cuda.synchronize()
        assert fp8.device_status() == fp8.OK
        assert H.normwise_rel_err(out, ref.double().cpu().numpy()) <= TOL[dtype], call
        # same kernels, same split and the same order of additions: identical
        assert torch.equal(out, ref), call


def test_noalloc_host_validation():
    # every rule is checked on the host before any CUDA call (no device needed)
    lib = fp8.load()
    f = lib.fp8_blockscaled_gemm_noalloc
    ok = (A16, A16, A16, A16, A16)
    assert f(*ok, 0, 128, 256, 256, fp8.WHOLE_K, None) == fp8.ERR_INVALID_ARG      # no study mode
    assert f(*ok, 0, 128, 256, 256, 64, None) == fp8.ERR_INVALID_ARG               # unknown flag
    assert f(*ok, 0, 128, 256, 200, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE          # K % 128
    assert f(A16 + 4, A16, A16, A16, A16, 0, 128, 256, 256, 0, None) == fp8.ERR_MISALIGNED
    assert f(None, None, A16, A16, None, 0, 0, 256, 256, 0, None) == fp8.OK        # M == 0
    assert isinstance(ctypes.c_void_p(A16).value, int)

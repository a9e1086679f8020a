"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host (CPU only: no call here reaches a kernel launch)."""

import ctypes
import os
import re

import pytest

import fp8_fine_grained_19_b300 as fp8
from fp8_fine_grained_19_b300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8fg.h")


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fp8.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_four_ops():
    names = declared_functions()
    for op in ("fp8_act_quant", "fp8_weight_quant", "fp8_blockscaled_gemm", "fp8_grouped_gemm",
               "fp8_get_device_status", "fp8fg_status_string"):
        assert op in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.fp8fg_abi_version() == 6
    for code in range(7):
        assert fp8.status_string(code)
    assert "unknown" in fp8.status_string(99)


# Host validation: every case below must be rejected before any CUDA call.
A16 = 1 << 20            # a fake, 16-byte aligned "device pointer" (never dereferenced)
MIS = A16 + 4            # misaligned


def test_act_quant_rejections(lib):
    f = lib.fp8_act_quant
    assert f(None, 0, 4, 128, A16, A16, 0, None) == fp8.ERR_INVALID_ARG          # null x
    assert f(A16, 7, 4, 128, A16, A16, 0, None) == fp8.ERR_INVALID_ARG           # bad dtype
    assert f(A16, 0, 4, 128, A16, A16, 8, None) == fp8.ERR_INVALID_ARG           # bad flag
    assert f(A16, 0, -1, 128, A16, A16, 0, None) == fp8.ERR_INVALID_ARG          # negative M
    assert f(A16, 0, 4, 100, A16, A16, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE     # K % 128
    assert f(A16, 0, 4, 0, A16, A16, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE
    assert f(A16, 0, 100, 128, A16, A16, fp8.TRANSPOSE, None) == fp8.ERR_UNSUPPORTED_SHAPE
    assert f(MIS, 0, 4, 128, A16, A16, 0, None) == fp8.ERR_MISALIGNED
    assert f(A16, 0, 4, 128, A16, MIS, 0, None) == fp8.ERR_MISALIGNED
    assert f(A16, 0, 1 << 31, 128, A16, A16, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE
    assert f(None, 0, 0, 128, None, None, 0, None) == fp8.OK                     # M == 0: no-op


def test_weight_quant_rejections(lib):
    f = lib.fp8_weight_quant
    assert f(A16, 0, 128, 128, A16, A16, A16, None, 0, None) == fp8.ERR_INVALID_ARG   # q_t w/o s_t
    assert f(A16, 0, 128, 128, A16, A16, None, None, fp8.TRANSPOSE, None) == fp8.ERR_INVALID_ARG
    assert f(A16, 0, 100, 128, A16, A16, None, None, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE
    assert f(A16, 0, 128, 130, A16, A16, None, None, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE
    assert f(A16, 0, 128, 128, MIS, A16, None, None, 0, None) == fp8.ERR_MISALIGNED


def test_requant_transpose_rejections(lib):
    f = lib.fp8_requant_transpose
    assert f(A16, A16, 128, 128, A16, A16, fp8.TRANSPOSE, None) == fp8.ERR_INVALID_ARG  # flag
    assert f(None, A16, 128, 128, A16, A16, 0, None) == fp8.ERR_INVALID_ARG
    assert f(A16, A16, -128, 128, A16, A16, 0, None) == fp8.ERR_INVALID_ARG
    assert f(A16, A16, 100, 128, A16, A16, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE       # M % 128
    assert f(A16, A16, 128, 200, A16, A16, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE       # K % 128
    assert f(A16, MIS, 128, 128, A16, A16, 0, None) == fp8.ERR_MISALIGNED
    assert f(None, None, 0, 128, None, None, 0, None) == fp8.OK                     # M == 0


def test_gemm_rejections(lib):
    f = lib.fp8_blockscaled_gemm
    ok = (A16, A16, A16, A16, A16)
    assert f(*ok, 2, 128, 256, 256, 0, None) == fp8.ERR_INVALID_ARG                   # dtype
    assert f(*ok, 0, 128, 256, 256, 16, None) == fp8.ERR_INVALID_ARG                  # flag
    assert f(*ok, 0, 128, 256, 256, fp8.WHOLE_K | fp8.B_TILE1x128, None) == fp8.ERR_INVALID_ARG
    assert f(None, A16, A16, A16, A16, 0, 128, 256, 256, 0, None) == fp8.ERR_INVALID_ARG
    assert f(*ok, 0, 128, 256, 200, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE             # K % 128
    assert f(*ok, 0, 128, 200, 256, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE             # N % 128
    assert f(*ok, 0, 128, 200, 256, fp8.B_TILE1x128, None) == fp8.ERR_UNSUPPORTED_SHAPE  # N % 16
    assert f(A16, A16, MIS, A16, A16, 0, 128, 256, 256, 0, None) == fp8.ERR_MISALIGNED
    assert f(None, None, A16, A16, None, 0, 0, 256, 256, 0, None) == fp8.OK             # M == 0


def test_gemm_quant_rejections(lib):
    f = lib.fp8_blockscaled_gemm_quant
    ok = (A16, A16, A16, A16, A16, A16)
    assert f(*ok, 128, 256, 256, 2, None) == fp8.ERR_INVALID_ARG                      # TRANSPOSE
    assert f(*ok, 128, 256, 256, 8, None) == fp8.ERR_INVALID_ARG                      # unknown
    assert f(A16, A16, A16, A16, A16, None, 128, 256, 256, 0, None) == fp8.ERR_INVALID_ARG
    assert f(*ok, 128, 256, 200, 0, None) == fp8.ERR_UNSUPPORTED_SHAPE                # K % 128
    assert f(*ok, 128, 144, 256, fp8.B_TILE1x128, None) == fp8.ERR_UNSUPPORTED_SHAPE  # N % 128
    assert f(A16, A16, A16, A16, A16, MIS, 128, 256, 256, 0, None) == fp8.ERR_MISALIGNED
    assert f(None, None, A16, A16, None, None, 0, 256, 256, fp8.POW2, None) == fp8.OK  # M == 0


def test_grouped_rejections(lib):
    f = lib.fp8_grouped_gemm
    args = lambda E=4, T=512, N=256, K=256, flags=0, off=A16: (
        A16, A16, off, E, T, A16, A16, A16, 0, N, K, flags, None)
    assert f(*args(E=0)) == fp8.ERR_INVALID_ARG
    assert f(*args(off=None)) == fp8.ERR_INVALID_ARG
    assert f(*args(flags=1)) == fp8.ERR_INVALID_ARG
    assert f(*args(E=2000)) == fp8.ERR_UNSUPPORTED_SHAPE
    assert f(*args(N=200)) == fp8.ERR_UNSUPPORTED_SHAPE
    assert f(*args(off=A16 + 2)) == fp8.ERR_MISALIGNED
    assert f(None, None, A16, 4, 0, A16, A16, None, 0, 256, 256, 0, None) == fp8.OK  # no rows


def test_grouped_swiglu_rejections(lib):
    f = lib.fp8_grouped_gemm_swiglu_quant
    args = lambda E=4, T=512, N=512, K=256, flags=fp8.POW2, off=A16, s=A16: (
        A16, A16, off, E, T, A16, A16, A16, s, N, K, flags, None)
    assert f(*args(E=0)) == fp8.ERR_INVALID_ARG
    assert f(*args(off=None)) == fp8.ERR_INVALID_ARG
    assert f(*args(s=None)) == fp8.ERR_INVALID_ARG
    assert f(*args(flags=fp8.TRANSPOSE)) == fp8.ERR_INVALID_ARG
    assert f(*args(N=384)) == fp8.ERR_UNSUPPORTED_SHAPE                  # 2I % 256
    assert f(*args(K=200)) == fp8.ERR_UNSUPPORTED_SHAPE
    assert f(*args(E=2000)) == fp8.ERR_UNSUPPORTED_SHAPE
    assert f(*args(off=A16 + 2)) == fp8.ERR_MISALIGNED
    assert f(*args(s=MIS)) == fp8.ERR_MISALIGNED
    # no rows: nothing launched, null row buffers accepted (no device needed)
    assert f(None, None, A16, 4, 0, A16, A16, None, None, 512, 256, fp8.POW2, None) == fp8.OK


def test_selftest_rejects_bad_limit(lib):
    assert lib.fp8fg_selftest_wait_timeout(0, None) == fp8.ERR_INVALID_ARG
    assert lib.fp8fg_selftest_wait_timeout((1 << 31) + 1, None) == fp8.ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fp8, "_LIB", None)
    monkeypatch.setattr(fp8, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        fp8.load()


def test_binding_rejects_mixed_devices():
    # the library launches on the current device and reads raw pointers, so a
    # call whose tensors live on different devices must not reach it
    import torch
    a = torch.empty(4)
    b = torch.empty(4, device="meta")
    with pytest.raises(ValueError):
        fp8._same_device(a, b)
    assert fp8._same_device(a, None, a) == a.device


def test_gemm_ws_rejections(lib):
    f = lib.fp8_blockscaled_gemm_ws
    ok = (A16, A16, A16, A16, A16)
    st = fp8.STREAM_K
    assert f(*ok, 0, 128, 256, 256, fp8.WHOLE_K, A16, 1 << 30, None) == fp8.ERR_INVALID_ARG   # no study mode
    assert f(*ok, 0, 128, 256, 256, 32, A16, 1 << 30, None) == fp8.ERR_INVALID_ARG            # unknown flag
    assert f(*ok, 0, 128, 256, 256, st, None, 0, None) == fp8.ERR_INVALID_ARG                 # forced, no workspace
    assert f(*ok, 0, 128, 256, 200, 0, A16, 1 << 30, None) == fp8.ERR_UNSUPPORTED_SHAPE       # K % 128
    assert f(*ok, 0, 128, 256, 256, 0, MIS, 1 << 30, None) == fp8.ERR_MISALIGNED              # workspace
    assert f(None, None, A16, A16, None, 0, 0, 256, 256, st, A16, 1 << 30, None) == fp8.OK    # M == 0
    # the plain entry point has no workspace, so it rejects the forced split
    assert lib.fp8_blockscaled_gemm(*ok, 0, 128, 256, 256, st, None) == fp8.ERR_INVALID_ARG


def test_workspace_query_without_device(lib):
    # without a device (or for invalid sizes) nothing is split
    assert lib.fp8_blockscaled_gemm_workspace_bytes(4096, 7168, 18432, 0) in (0, 148 * 128 * 256 * 4)
    assert lib.fp8_blockscaled_gemm_workspace_bytes(0, 7168, 18432, 0) == 0
    assert lib.fp8_blockscaled_gemm_workspace_bytes(128, 256, 200, 0) == 0

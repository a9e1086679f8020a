"""Python binding of libfp8fg.so (fine-grained FP8 quantisation and block-scaled GEMMs).

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  The functions have the
C ABI's names without the ``fp8_`` prefix; each checks tensor dtypes, devices
and contiguity, allocates the outputs with torch, and raises ``Fp8Error`` on a
non-OK status.  There is no CPU fallback: without the built library or a CUDA
device the calls raise.
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "Fp8Error", "load", "lib_path", "act_quant", "weight_quant", "requant_transpose", "gemm",
    "gemm_quant", "grouped_gemm", "grouped_swiglu_quant",
    "device_status", "set_wait_limit", "selftest_wait_timeout", "status_string",
    "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED_SHAPE", "ERR_MISALIGNED", "ERR_CUDA",
    "ERR_TIMEOUT", "ERR_BAD_OFFSETS", "POW2", "TRANSPOSE", "B_TILE1x128", "WHOLE_K", "STREAM_K",
    "BF16", "F32", "gemm_workspace_bytes",
]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_CUDA, ERR_TIMEOUT, \
    ERR_BAD_OFFSETS = range(7)
BF16, F32 = 0, 1
POW2, TRANSPOSE, B_TILE1x128, WHOLE_K, STREAM_K = 1, 2, 4, 8, 16

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB: ctypes.CDLL | None = None

_vp, _i64, _u32, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint, ctypes.c_int32
_SIGS = {
    "fp8_act_quant": [_vp, ctypes.c_int, _i64, _i64, _vp, _vp, _u32, _vp],
    "fp8_weight_quant": [_vp, ctypes.c_int, _i64, _i64, _vp, _vp, _vp, _vp, _u32, _vp],
    "fp8_requant_transpose": [_vp, _vp, _i64, _i64, _vp, _vp, _u32, _vp],
    "fp8_blockscaled_gemm": [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, _i64, _i64, _i64, _u32, _vp],
    "fp8_blockscaled_gemm_ws": [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, _i64, _i64, _i64, _u32, _vp,
                                ctypes.c_size_t, _vp],
    "fp8_blockscaled_gemm_workspace_bytes": [_i64, _i64, _i64, _u32],
    "fp8_blockscaled_gemm_noalloc": [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, _i64, _i64, _i64, _u32,
                                     _vp],
    "fp8_blockscaled_gemm_quant": [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _u32, _vp],
    "fp8_grouped_gemm": [_vp, _vp, _vp, _i32, _i64, _vp, _vp, _vp, ctypes.c_int, _i64, _i64,
                         _u32, _vp],
    "fp8_grouped_gemm_swiglu_quant": [_vp, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _i64, _i64,
                                      _u32, _vp],
    "fp8_get_device_status": [_vp],
    "fp8fg_status_string": [ctypes.c_int],
    "fp8fg_abi_version": [],
    "fp8fg_set_wait_limit": [ctypes.c_uint64],
    "fp8fg_selftest_wait_timeout": [ctypes.c_uint32, _vp],
}


class Fp8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib_path() -> str:
    return os.path.join(_HERE, "libfp8fg.so")


def load() -> ctypes.CDLL:
    """Load libfp8fg.so from this package directory (raises if it is missing)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m fp8_fine_grained_19_b300.build`")
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_char_p if name == "fp8fg_status_string" else (
            None if name == "fp8fg_set_wait_limit" else (
                ctypes.c_size_t if name == "fp8_blockscaled_gemm_workspace_bytes" else ctypes.c_int))
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    return load().fp8fg_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise Fp8Error(status, where)


def _stream(stream, device: torch.device) -> int:
    """Raw handle of `stream` (default: the current stream of `device`)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return int(stream.cuda_stream)


def _same_device(*tensors) -> torch.device:
    """The one CUDA device every given tensor lives on (None entries are skipped).

    The library launches on the calling thread's current device and builds its
    TMA descriptors over the raw pointers, so operands on another GPU would be
    read as peer memory; mixed devices are rejected here instead."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one CUDA device, got {sorted(map(str, devs))}")
    return devs.pop()


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtypes, name: str) -> None:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _src_dtype(t: torch.Tensor) -> int:
    return BF16 if t.dtype == torch.bfloat16 else F32


_SRC = (torch.bfloat16, torch.float32)


def _run(fn: str, device: torch.device, *args) -> int:
    """Call library entry point `fn` with `device` current (the library launches on
    the calling thread's current device)."""
    with torch.cuda.device(device):
        return getattr(load(), fn)(*args)


def act_quant(x: torch.Tensor, pow2: bool = False, transpose: bool = False, stream=None):
    """1x128 tiles -> (q uint8 [M, K], s float32 [M, K/128]);
    transpose=True: 128x1 tiles -> (q [K, M], s [K, M/128])."""
    _need(x, _SRC, "x")
    M, K = x.shape
    if transpose:
        q = torch.empty((K, M), dtype=torch.uint8, device=x.device)
        s = torch.empty((K, M // 128 if M % 128 == 0 else 1), dtype=torch.float32, device=x.device)
    else:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
        s = torch.empty((M, K // 128 if K % 128 == 0 else 1), dtype=torch.float32, device=x.device)
    flags = (POW2 if pow2 else 0) | (TRANSPOSE if transpose else 0)
    dev = x.device
    _check(_run("fp8_act_quant", dev, _ptr(x), _src_dtype(x), M, K, _ptr(q), _ptr(s), flags,
                _stream(stream, dev)), "fp8_act_quant")
    return q, s


def weight_quant(w: torch.Tensor, pow2: bool = False, transposed: bool = False, stream=None):
    """128x128 blocks -> (q [N, K], s [N/128, K/128]) (+ (q_t [K, N], s_t) if transposed)."""
    _need(w, _SRC, "w")
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((max(N // 128, 1), max(K // 128, 1)), dtype=torch.float32, device=w.device)
    qt = st = None
    if transposed:
        qt = torch.empty((K, N), dtype=torch.uint8, device=w.device)
        st = torch.empty((max(K // 128, 1), max(N // 128, 1)), dtype=torch.float32, device=w.device)
    dev = w.device
    _check(_run("fp8_weight_quant", dev, _ptr(w), _src_dtype(w), N, K, _ptr(q), _ptr(s), _ptr(qt),
                _ptr(st), POW2 if pow2 else 0, _stream(stream, dev)), "fp8_weight_quant")
    return (q, s, qt, st) if transposed else (q, s)


def requant_transpose(q: torch.Tensor, s: torch.Tensor, pow2: bool = False, stream=None):
    """Stored 1x128 codes (q [M, K], s [M, K/128]) -> 128x1 tiles (q_t [K, M], s_t [K, M/128])."""
    _need(q, (torch.uint8,), "q")
    _need(s, (torch.float32,), "s")
    dev = _same_device(q, s)
    M, K = q.shape
    qt = torch.empty((K, M), dtype=torch.uint8, device=dev)
    st = torch.empty((K, M // 128 if M % 128 == 0 else 1), dtype=torch.float32, device=dev)
    _check(_run("fp8_requant_transpose", dev, _ptr(q), _ptr(s), M, K, _ptr(qt), _ptr(st),
                POW2 if pow2 else 0, _stream(stream, dev)), "fp8_requant_transpose")
    return qt, st


def _out_code(dtype) -> int:
    if dtype == torch.bfloat16:
        return BF16
    if dtype == torch.float32:
        return F32
    raise ValueError(f"unsupported output dtype {dtype}")


def gemm_workspace_bytes(M: int, N: int, K: int, b_tile: bool = False, stream_k: bool = False,
                         device=None) -> int:
    """Workspace bytes the stream-K split of this GEMM uses on `device` (0: no split)."""
    flags = (B_TILE1x128 if b_tile else 0) | (STREAM_K if stream_k else 0)
    dev = _device_arg(device)
    with torch.cuda.device(dev):
        return int(load().fp8_blockscaled_gemm_workspace_bytes(M, N, K, flags))


def gemm(a, sa, b, sb, out_dtype=torch.bfloat16, b_tile: bool = False, out=None, stream=None,
         whole_k: bool = False, stream_k="auto", workspace=None):
    """C[M, N] = sum_kb (A_kb . B_kb^T) * sa[:, kb] * sb(., kb), promoted to FP32 per 128 K.

    whole_k: study mode without promotion (all of K in the tensor core, scaled by
    sa[0, 0] * sb[0, 0]).
    stream_k: "auto" splits the K slices of the last tiles among all SMs when the
    tiles would leave most SMs idle (a workspace is then taken from torch, or
    `workspace` is used); True forces the split; False never splits."""
    for t, n in ((a, "a"), (b, "b")):
        _need(t, (torch.uint8,), n)
    for t, n in ((sa, "sa"), (sb, "sb")):
        _need(t, (torch.float32,), n)
    dev = _same_device(a, sa, b, sb, out)
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("a and b disagree on K")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    _need(out, (torch.bfloat16, torch.float32), "out")
    flags = (B_TILE1x128 if b_tile else 0) | (WHOLE_K if whole_k else 0)
    if whole_k or stream_k is False:
        _check(_run("fp8_blockscaled_gemm", dev, _ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(out),
                    _out_code(out.dtype), M, N, K, flags, _stream(stream, dev)),
               "fp8_blockscaled_gemm")
        return out
    if stream_k is True:
        flags |= STREAM_K
    need = gemm_workspace_bytes(M, N, K, b_tile, stream_k is True, dev) if M > 0 else 0
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, (torch.uint8,), "workspace")
        if workspace.device != dev:
            raise ValueError("workspace must be on the device of the operands")
    _check(_run("fp8_blockscaled_gemm_ws", dev, _ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(out),
                _out_code(out.dtype), M, N, K, flags, _ptr(workspace) if need else None,
                workspace.numel() if (need and workspace is not None) else 0, _stream(stream, dev)),
           "fp8_blockscaled_gemm_ws")
    return out


def gemm_quant(a, sa, b, sb, b_tile: bool = False, pow2: bool = False, out=None,
               out_scales=None, stream=None):
    """The gemm result quantised in the epilogue: (q uint8 [M, N], s float32 [M, N/128])."""
    for t, n in ((a, "a"), (b, "b")):
        _need(t, (torch.uint8,), n)
    for t, n in ((sa, "sa"), (sb, "sb")):
        _need(t, (torch.float32,), n)
    dev = _same_device(a, sa, b, sb, out, out_scales)
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("a and b disagree on K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.uint8, device=dev)
    if out_scales is None:
        out_scales = torch.empty((M, max(N // 128, 1)), dtype=torch.float32, device=dev)
    _need(out, (torch.uint8,), "out")
    _need(out_scales, (torch.float32,), "out_scales")
    flags = (B_TILE1x128 if b_tile else 0) | (POW2 if pow2 else 0)
    _check(_run("fp8_blockscaled_gemm_quant", dev, _ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(out),
                _ptr(out_scales), M, N, K, flags, _stream(stream, dev)),
           "fp8_blockscaled_gemm_quant")
    return out, out_scales


def grouped_gemm(a, sa, offsets, b, sb, out_dtype=torch.bfloat16, out=None, stream=None):
    """Per-expert gemm over row groups offsets[e]..offsets[e+1] (device int32 [E+1])."""
    _need(a, (torch.uint8,), "a")
    _need(b, (torch.uint8,), "b")
    _need(sa, (torch.float32,), "sa")
    _need(sb, (torch.float32,), "sb")
    _need(offsets, (torch.int32,), "offsets")
    dev = _same_device(a, sa, offsets, b, sb, out)
    T, K = a.shape
    E, N, Kb = b.shape
    if Kb != K or offsets.numel() != E + 1:
        raise ValueError("shape mismatch between a, b and offsets")
    if out is None:
        out = torch.empty((T, N), dtype=out_dtype, device=dev)
    _need(out, (torch.bfloat16, torch.float32), "out")
    _check(_run("fp8_grouped_gemm", dev, _ptr(a), _ptr(sa), _ptr(offsets), E, T, _ptr(b), _ptr(sb),
                _ptr(out), _out_code(out.dtype), N, K, 0, _stream(stream, dev)),
           "fp8_grouped_gemm")
    return out


def grouped_swiglu_quant(a, sa, offsets, b, sb, pow2: bool = True, out=None, out_scales=None,
                         stream=None):
    """Routed up-projection (b [E, 2I, K]: gate rows then up rows) followed by
    h = silu(g) * u, returned as the down-projection input (q uint8 [T, I],
    s float32 [T, I/128])."""
    _need(a, (torch.uint8,), "a")
    _need(b, (torch.uint8,), "b")
    _need(sa, (torch.float32,), "sa")
    _need(sb, (torch.float32,), "sb")
    _need(offsets, (torch.int32,), "offsets")
    dev = _same_device(a, sa, offsets, b, sb, out, out_scales)
    T, K = a.shape
    E, N, Kb = b.shape
    if Kb != K or offsets.numel() != E + 1:
        raise ValueError("shape mismatch between a, b and offsets")
    I = N // 2
    if out is None:
        out = torch.empty((T, I), dtype=torch.uint8, device=dev)
    if out_scales is None:
        out_scales = torch.empty((T, max(I // 128, 1)), dtype=torch.float32, device=dev)
    _need(out, (torch.uint8,), "out")
    _need(out_scales, (torch.float32,), "out_scales")
    _check(_run("fp8_grouped_gemm_swiglu_quant", dev, _ptr(a), _ptr(sa), _ptr(offsets), E, T,
                _ptr(b), _ptr(sb), _ptr(out), _ptr(out_scales), N, K, POW2 if pow2 else 0,
                _stream(stream, dev)),
           "fp8_grouped_gemm_swiglu_quant")
    return out, out_scales


def _device_arg(device) -> torch.device:
    return torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)


def device_status(stream=None, device=None) -> int:
    """Synchronise the stream; return and clear the library's device status word
    of that stream's device (default: the current device)."""
    dev = stream.device if stream is not None else _device_arg(device)
    return int(_run("fp8_get_device_status", dev, _stream(stream, dev)))


def set_wait_limit(cycles: int) -> None:
    load().fp8fg_set_wait_limit(int(cycles))


def selftest_wait_timeout(limit_cycles: int = 1 << 20, stream=None, device=None) -> int:
    """Run the bounded-wait self-test; returns the device status it produced."""
    dev = stream.device if stream is not None else _device_arg(device)
    _check(_run("fp8fg_selftest_wait_timeout", dev, int(limit_cycles), _stream(stream, dev)),
           "fp8fg_selftest_wait_timeout")
    return device_status(stream, dev)

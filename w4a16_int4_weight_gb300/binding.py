"""Thin binding of libw4a16 (C ABI in include/w4a16.h): ctypes, plus a CPython
marshalling module for the per-call GEMM entry points.

Argument marshalling only: every entry point forwards raw device pointers,
sizes and the current CUDA stream to the library, which validates and runs all
of the work in its own kernels.  Importing this module fails loudly if the
library has not been built (``python -m w4a16_int4_weight_gb300.build``);
there is no fallback.
"""

from __future__ import annotations

import ctypes
import operator
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libw4a16.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_TIMEOUT = range(5)
UINT4B8, UINT4 = 0, 1
FP16, BF16 = 0, 1
PATH_AUTO, PATH_DECODE, PATH_FUSED, PATH_DENSE, PATH_FUSED_TMEM, PATH_FUSED_SMEM = range(6)
QTYPES = {"uint4b8": UINT4B8, "uint4": UINT4}
DTYPES = {"fp16": FP16, "bf16": BF16}
PATHS = {"auto": PATH_AUTO, "decode": PATH_DECODE, "fused": PATH_FUSED, "dense": PATH_DENSE,
         "fused_tmem": PATH_FUSED_TMEM, "fused_smem": PATH_FUSED_SMEM}
OPT_STATIC_WEIGHTS = 0x100


class W4A16Error(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"w4a16 error {code}: {message}")
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError(f"libw4a16.so is not built ({LIB_PATH}); run "
                      "`python -m w4a16_int4_weight_gb300.build`")

lib = ctypes.CDLL(LIB_PATH)



class _RangeCheckedInt:
    """ctypes argument type for a C integer parameter.  ctypes itself keeps only the
    low bits of a Python int that does not fit (2**32 + 128 would pass as 128);
    this refuses such a value with OverflowError instead."""
    ctype = ctypes.c_int
    bits = 32

    @classmethod
    def from_param(cls, v):
        if isinstance(v, ctypes._SimpleCData):   # a ctypes integer object, as ctypes accepts
            v = v.value
        v = operator.index(v)
        if not -(1 << (cls.bits - 1)) <= v < (1 << (cls.bits - 1)):
            raise OverflowError(f"{v} does not fit a {cls.bits}-bit C integer")
        return cls.ctype(v)


class _CheckedInt64(_RangeCheckedInt):
    ctype = ctypes.c_int64
    bits = 64


class LaunchInfo(ctypes.Structure):
    """w4a16_launch_info."""
    _fields_ = [("path", ctypes.c_int), ("token_tile", ctypes.c_int), ("k_split", ctypes.c_int),
                ("stages", ctypes.c_int), ("grid", ctypes.c_int64), ("smem_bytes", ctypes.c_int64)]


_P = ctypes.c_void_p
_I64 = _CheckedInt64
_I = _RangeCheckedInt
_SZ = ctypes.POINTER(ctypes.c_size_t)

_SIGS = {
    "w4a16_version": (ctypes.c_int, []),
    "w4a16_last_error_string": (ctypes.c_char_p, []),
    "w4a16_packed_layout": (ctypes.c_int, [_I64, _I64, _I, _I, _I, _SZ, _SZ, _SZ, ctypes.POINTER(ctypes.c_int64)]),
    "w4a16_pack": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I, _I, _I, _P]),
    "w4a16_pack_ex": (ctypes.c_int, [_P, _I, _P, _P, _I, _P, _I64, _I64, _I, _I, _I, _P]),
    "w4a16_gemm": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P]),
    "w4a16_gemm_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _I, _P]),
    "w4a16_linear": (ctypes.c_int, [_P, _I64, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I, _I, _I, _I, _P]),
    "w4a16_route": (ctypes.c_int, [_I64, _I64, _I64, _I, _I, _I, _I]),
    "w4a16_launch_plan": (ctypes.c_int, [_I64, _I64, _I64, _I, _I, _I, _I, _I, _I, ctypes.POINTER(LaunchInfo)]),
    "w4a16_dequant": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I, _I, _I, _P]),
    "w4a16_gemm_dense": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _I, _P]),
    "w4a16_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int)]),
    "w4a16_selftest_wait_timeout": (ctypes.c_int, [_P]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)

# Per-call entry points: the CPython marshalling module built beside the library
# (csrc/py_fastcall.c) when the Python headers were available, else ctypes.  Both
# take the same integer arguments and call the same libw4a16 functions.
try:
    from . import _w4a16_fastcall as _fastcall
    _fastcall.bind(ctypes.cast(lib.w4a16_gemm_ex, ctypes.c_void_p).value,
                   ctypes.cast(lib.w4a16_linear, ctypes.c_void_p).value)
    _gemm_ex_call, _linear_call = _fastcall.gemm_ex, _fastcall.linear
except ImportError:
    _fastcall = None
    _gemm_ex_call, _linear_call = lib.w4a16_gemm_ex, lib.w4a16_linear


def last_error() -> str:
    return lib.w4a16_last_error_string().decode()


def _check(code: int) -> None:
    if code != OK:
        raise W4A16Error(code, last_error())


def _ptr(x):
    """Device/host address of a torch tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


_RAW_STREAM = None


def _current_stream_handle():
    """torch's current CUDA stream on the current device, as a raw handle.  The
    raw query costs well under a microsecond; torch.cuda.current_stream() builds
    a Python object per call (several microseconds), which is used only when the
    raw query is not available."""
    global _RAW_STREAM
    import torch
    if _RAW_STREAM is None:
        get_dev = getattr(torch._C, "_cuda_getDevice", None)
        get_raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _RAW_STREAM = (lambda: get_raw(get_dev())) if get_dev and get_raw else False
    if _RAW_STREAM:
        return _RAW_STREAM()
    return torch.cuda.current_stream().cuda_stream


def _stream(stream):
    if stream is None:
        return _current_stream_handle()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _qt(qtype):
    return QTYPES[qtype] if isinstance(qtype, str) else int(qtype)


def _dt(dtype):
    if isinstance(dtype, str):
        return DTYPES[dtype]
    try:
        import torch
        if dtype is torch.float16:
            return FP16
        if dtype is torch.bfloat16:
            return BF16
    except ImportError:
        pass
    return int(dtype)


def version() -> int:
    return lib.w4a16_version()


def packed_layout(N, K, G, qtype, dtype):
    """(total_bytes, scales_off, zeros_off, ldq_words) of the packed buffer."""
    tot, so, zo = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    ldq = ctypes.c_int64()
    _check(lib.w4a16_packed_layout(N, K, G, _qt(qtype), _dt(dtype), ctypes.byref(tot),
                                   ctypes.byref(so), ctypes.byref(zo), ctypes.byref(ldq)))
    return tot.value, so.value, zo.value, ldq.value


def pack(q, scales, zeros, Wpacked, N, K, G, qtype, dtype, stream=None):
    _check(lib.w4a16_pack(_ptr(q), _ptr(scales), _ptr(zeros), _ptr(Wpacked), N, K, G,
                          _qt(qtype), _dt(dtype), _stream(stream)))


def gemm(A, Wq, scales, zeros, C, M, N, K, G, qtype, dtype, stream=None):
    _check(lib.w4a16_gemm(_ptr(A), _ptr(Wq), _ptr(scales), _ptr(zeros), _ptr(C), M, N, K, G,
                          _qt(qtype), _dt(dtype), _stream(stream)))


def gemm_ex(A, Wq, scales, zeros, Wdense, C, M, N, K, G, qtype, dtype, path="auto",
            stream=None, static_weights=False):
    p = PATHS[path] if isinstance(path, str) else int(path)
    if static_weights:
        p |= OPT_STATIC_WEIGHTS
    if _fastcall is not None:   # takes tensors, int addresses or None as they are
        code = _fastcall.gemm_ex(A, Wq, scales, zeros, Wdense, C, M, N, K, G, _qt(qtype), _dt(dtype),
                                 p, _stream(stream))
    else:
        code = lib.w4a16_gemm_ex(_ptr(A), _ptr(Wq), _ptr(scales), _ptr(zeros), _ptr(Wdense), _ptr(C),
                                 M, N, K, G, _qt(qtype), _dt(dtype), p, _stream(stream))
    if code:
        raise W4A16Error(code, last_error())


def linear(A, Wq, scales, zeros, bias, Wdense, C, M, N, K, G, qtype, dtype, path="auto",
           stream=None, static_weights=False, lda=0, ldc=0):
    """gemm_ex plus bias[N] (dtype) added before the output rounding; bias may be None;
    lda / ldc: row pitches of A and C in elements (0 = contiguous)."""
    p = PATHS[path] if isinstance(path, str) else int(path)
    if static_weights:
        p |= OPT_STATIC_WEIGHTS
    call = _fastcall.linear if _fastcall is not None else lib.w4a16_linear
    _check(call(_ptr(A), lda, _ptr(Wq), _ptr(scales), _ptr(zeros), _ptr(bias),
                _ptr(Wdense), _ptr(C), ldc, M, N, K, G, _qt(qtype), _dt(dtype), p,
                _stream(stream)))


QFORMATS = {"unpacked": 0, "gptq": 1, "exllama": 2, "kn": 3}
LAYOUTS = {"ng": 0, "gn": 1}


def pack_ex(qsrc, qformat, scales, zeros, param_layout, Wpacked, N, K, G, qtype, dtype, stream=None):
    """Pack from a checkpoint word format ("unpacked", "gptq", "exllama", "kn"), scales and
    zeros laid out "ng" ([N][ng], [N/8][ng]) or "gn" ([ng][N], [ng][N/8])."""
    f = QFORMATS[qformat] if isinstance(qformat, str) else int(qformat)
    lay = LAYOUTS[param_layout] if isinstance(param_layout, str) else int(param_layout)
    _check(lib.w4a16_pack_ex(_ptr(qsrc), f, _ptr(scales), _ptr(zeros), lay, _ptr(Wpacked), N, K, G,
                             _qt(qtype), _dt(dtype), _stream(stream)))


def route(M, N, K, G, qtype, dtype, has_dense=False) -> int:
    return lib.w4a16_route(M, N, K, G, _qt(qtype), _dt(dtype), int(bool(has_dense)))


def dequant(Wq, scales, zeros, W, N, K, G, qtype, dtype, stream=None):
    _check(lib.w4a16_dequant(_ptr(Wq), _ptr(scales), _ptr(zeros), _ptr(W), N, K, G,
                             _qt(qtype), _dt(dtype), _stream(stream)))


def gemm_dense(A, W, C, M, N, K, dtype, stream=None):
    _check(lib.w4a16_gemm_dense(_ptr(A), _ptr(W), _ptr(C), M, N, K, _dt(dtype),
                                _stream(stream)))


def device_status():
    """(status code, wait site) after synchronising the device; clears the status."""
    site = ctypes.c_int(0)
    code = lib.w4a16_device_status(ctypes.byref(site))
    return code, site.value


SELFTEST_SITE = 90   # W4A16_SELFTEST_SITE


def selftest_wait_timeout(stream=None):
    """Enqueue the failure-detection self-test: one warp's bounded wait on a barrier
    that nothing completes gives up after about a second; device_status() then
    reports (ERR_DEVICE_TIMEOUT, SELFTEST_SITE)."""
    _check(lib.w4a16_selftest_wait_timeout(_stream(stream)))


PATH_NAMES = {v: k for k, v in PATHS.items()}


def launch_plan(M, N, K, G, qtype, dtype, path="auto", has_dense=False, num_sms=152):
    """How gemm_ex would launch on a GPU with num_sms SMs (host-only): a dict with the
    kernel ("decode", "fused_tmem", "fused_smem" or "dense"), token_tile, k_split,
    stages, grid and smem_bytes."""
    p = PATHS[path] if isinstance(path, str) else int(path)
    info = LaunchInfo()
    _check(lib.w4a16_launch_plan(M, N, K, G, _qt(qtype), _dt(dtype), p, 1 if has_dense else 0,
                                 num_sms, ctypes.byref(info)))
    return {"path": PATH_NAMES[info.path], "token_tile": info.token_tile, "k_split": info.k_split,
            "stages": info.stages, "grid": info.grid, "smem_bytes": info.smem_bytes}

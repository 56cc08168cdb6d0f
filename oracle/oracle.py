"""ctypes front end of the plain-C oracle in ``w4a16_oracle.c``.

TEST INFRASTRUCTURE ONLY: used by the tests, the package smoke check and the
benchmark's CPU baseline; never by the product path.  Every function here only
marshals numpy arrays into the C routines, which hold all of the arithmetic.

Citations for each routine are in the C file's header.  No routine is "parity
unpinned": tests/test_oracle_pins.py pins each one against values and
identities fixed by the pages or by mathematics.
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liborc_w4a16.so")

FP16, BF16 = 0, 1
DTYPE_CODE = {"fp16": FP16, "bf16": BF16}

_lock = threading.Lock()
_lib = None


def _compile(src: str, out: str) -> None:
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    _compile(_SRC, tmp)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def source() -> str:
    """Text of the oracle's C source."""
    with open(_SRC) as f:
        return f.read()


def build_variant(text: str, out_dir: str) -> str:
    """Compile a modified copy of the C source (for tests that plant a mistake in
    the oracle and check that a pin catches it); returns the library path."""
    src = os.path.join(out_dir, "w4a16_oracle_variant.c")
    with open(src, "w") as f:
        f.write(text)
    out = os.path.join(out_dir, "liborc_variant.so")
    _compile(src, out)
    return out


def _configure(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    sig = {
        "orc_num_threads": (I, []),
        "orc_f16_value": (ctypes.c_double, [ctypes.c_uint16]),
        "orc_bf16_value": (ctypes.c_double, [ctypes.c_uint16]),
        "orc_round_f16": (ctypes.c_uint16, [ctypes.c_double]),
        "orc_round_bf16": (ctypes.c_uint16, [ctypes.c_double]),
        "orc_values": (None, [P, I64, I, P]),
        "orc_round": (None, [P, I64, I, P]),
        "orc_shift_table": (I, [I]),
        "orc_pack_q": (None, [P, I64, I64, I64, P]),
        "orc_unpack_q": (None, [P, I64, I64, I64, P]),
        "orc_zero_point": (I, [P, I64, I64, I64]),
        "orc_dequant": (None, [P, P, P, I64, I64, I64, I, P]),
        "orc_gemm": (I, [P, P, I64, I64, I64, I, P]),
        "orc_gemm_rows": (I, [P, P, P, I64, I64, I64, I, P]),
        "orc_gemm_pairs": (None, [P, P, P, P, I64, I64, I, P]),
        "orc_linear_rows": (I, [P, P, I64, P, P, P, I64, I64, I64, I64, I, P]),
        "orc_add_bias": (None, [P, I64, I64, P, I]),
        "orc_encode_gptq": (None, [P, I64, I64, P]),
        "orc_decode_gptq": (None, [P, I64, I64, P]),
        "orc_encode_kn": (None, [P, I64, I64, P]),
        "orc_decode_kn": (None, [P, I64, I64, P]),
        "orc_encode_exllama": (None, [P, I64, I64, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


def load_variant(path: str):
    """A library built by build_variant, with the oracle's signatures."""
    return _configure(ctypes.CDLL(path))


@contextlib.contextmanager
def using_library(lib):
    """Route every oracle call to `lib` (a load_variant result) inside the block."""
    global _lib
    prev = _load()
    with _lock:
        _lib = lib
    try:
        yield
    finally:
        with _lock:
            _lib = prev


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return _load().orc_num_threads()


def values(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of fp16/bf16 bit patterns."""
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().orc_values(_ptr(b), b.size, DTYPE_CODE[dtype], _ptr(out))
    return out


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """IEEE round-to-nearest-even of float64 values to fp16/bf16 bit patterns."""
    a = _c(x, np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().orc_round(_ptr(a), a.size, DTYPE_CODE[dtype], _ptr(out))
    return out


def shift_table() -> list[int]:
    """Bit offset of K-value i (0..7) inside a packed word."""
    lib = _load()
    return [lib.orc_shift_table(i) for i in range(8)]


def ldq_words(K: int) -> int:
    """Row pitch of the packed q section in 32-bit words: K/8 rounded up to 4."""
    return ((K // 8 + 3) // 4) * 4


def pack_q(q: np.ndarray, ldq: int | None = None) -> np.ndarray:
    """uint8 [N, K] (0..15) -> uint32 [N, ldq] packed words."""
    qq = _c(q, np.uint8)
    N, K = qq.shape
    ldq = ldq_words(K) if ldq is None else ldq
    out = np.empty((N, ldq), dtype=np.uint32)
    _load().orc_pack_q(_ptr(qq), N, K, ldq, _ptr(out))
    return out


def unpack_q(words: np.ndarray, K: int) -> np.ndarray:
    """uint32 [N, ldq] packed words -> uint8 [N, K]."""
    w = _c(words, np.uint32)
    N, ldq = w.shape
    out = np.empty((N, K), dtype=np.uint8)
    _load().orc_unpack_q(_ptr(w), N, K, ldq, _ptr(out))
    return out


def encode_q(q, fmt: str) -> np.ndarray:
    """Unpacked q [N, K] -> checkpoint words: "gptq" [N, K/8] (sequential along K),
    "exllama" [N, K/8] (shuffled), "kn" [K, N/8] (sequential along N)."""
    qq = _c(q, np.uint8)
    N, K = qq.shape
    lib = _load()
    if fmt == "kn":
        out = np.empty((K, N // 8), dtype=np.uint32)
        lib.orc_encode_kn(_ptr(qq), N, K, _ptr(out))
    else:
        out = np.empty((N, K // 8), dtype=np.uint32)
        {"gptq": lib.orc_encode_gptq, "exllama": lib.orc_encode_exllama}[fmt](_ptr(qq), N, K, _ptr(out))
    return out


def decode_q(words, fmt: str, N: int, K: int) -> np.ndarray:
    """Checkpoint words ("gptq" or "kn") -> unpacked q [N, K]."""
    w = _c(words, np.uint32)
    out = np.empty((N, K), dtype=np.uint8)
    lib = _load()
    {"gptq": lib.orc_decode_gptq, "kn": lib.orc_decode_kn}[fmt](_ptr(w), N, K, _ptr(out))
    return out


def zero_point(zeros, ng: int, n: int, g: int) -> int:
    z = _c(zeros, np.int32)
    return _load().orc_zero_point(_ptr(z), ng, n, g)


def dequant(q, scales, zeros, group_size: int, dtype: str) -> np.ndarray:
    """w[n,k] = rne_dtype((q[n,k] - zero[n,g]) * scale[n,g]) as uint16 bits [N, K]."""
    qq = _c(q, np.uint8)
    N, K = qq.shape
    g_eff = K if group_size == -1 else group_size
    s = _c(scales, np.uint16)
    z = _c(zeros, np.int32)
    assert s.shape == (N, K // g_eff)
    out = np.empty((N, K), dtype=np.uint16)
    _load().orc_dequant(_ptr(qq), _ptr(s), _ptr(z), N, K, g_eff, DTYPE_CODE[dtype], _ptr(out))
    return out


def gemm(A, W, dtype: str) -> np.ndarray:
    """C[m,n] = sum_k A[m,k] W[n,k] in float64 (A, W given as dtype bits)."""
    a = _c(A, np.uint16)
    w = _c(W, np.uint16)
    M, K = a.shape
    N = w.shape[0]
    out = np.empty((M, N), dtype=np.float64)
    if _load().orc_gemm(_ptr(a), _ptr(w), M, N, K, DTYPE_CODE[dtype], _ptr(out)):
        raise MemoryError("oracle: out of host memory")
    return out


def gemm_rows(A, W, rows, dtype: str) -> np.ndarray:
    a = _c(A, np.uint16)
    w = _c(W, np.uint16)
    r = _c(rows, np.int64)
    K = a.shape[1]
    N = w.shape[0]
    out = np.empty((r.size, N), dtype=np.float64)
    if _load().orc_gemm_rows(_ptr(a), _ptr(w), _ptr(r), r.size, N, K, DTYPE_CODE[dtype], _ptr(out)):
        raise MemoryError("oracle: out of host memory")
    return out


def gemm_pairs(A, W, ms, ns, dtype: str) -> np.ndarray:
    a = _c(A, np.uint16)
    w = _c(W, np.uint16)
    mm = _c(ms, np.int64)
    nn = _c(ns, np.int64)
    out = np.empty(mm.size, dtype=np.float64)
    _load().orc_gemm_pairs(_ptr(a), _ptr(w), _ptr(mm), _ptr(nn), mm.size, a.shape[1],
                           DTYPE_CODE[dtype], _ptr(out))
    return out


def add_bias(C: np.ndarray, bias, dtype: str) -> np.ndarray:
    """C[m,n] + bias[n] in float64 (bias given as dtype bits [N]); returns a new array."""
    out = np.array(C, dtype=np.float64, order="C", copy=True)
    b = _c(bias, np.uint16)
    M, N = out.shape
    assert b.shape == (N,)
    _load().orc_add_bias(_ptr(out), M, N, _ptr(b), DTYPE_CODE[dtype])
    return out


def linear(A, q, scales, zeros, group_size: int, dtype: str, bias=None) -> np.ndarray:
    """The whole layer from unpacked q: dequant, float64 GEMM, then + bias[n] if given."""
    C = gemm(A, dequant(q, scales, zeros, group_size, dtype), dtype)
    return C if bias is None else add_bias(C, bias, dtype)


def linear_rows_packed(A, words, K: int, scales, zeros, rows, group_size: int,
                       dtype: str) -> np.ndarray:
    """unpack -> dequant -> GEMM on selected rows of A, from packed words."""
    a = _c(A, np.uint16)
    w = _c(words, np.uint32)
    s = _c(scales, np.uint16)
    z = _c(zeros, np.int32)
    r = _c(rows, np.int64)
    N, ldq = w.shape
    g_eff = K if group_size == -1 else group_size
    out = np.empty((r.size, N), dtype=np.float64)
    rc = _load().orc_linear_rows(_ptr(a), _ptr(w), ldq, _ptr(s), _ptr(z), _ptr(r), r.size,
                                 N, K, g_eff, DTYPE_CODE[dtype], _ptr(out))
    if rc:
        raise MemoryError("oracle: out of host memory")
    return out


def rel_error(C_bits_or_values, C_ref: np.ndarray, dtype: str | None = None) -> float:
    """max|C - C_ref| / (max|C_ref| + 1e-6), C given as dtype bits (with dtype) or values."""
    C = values(C_bits_or_values, dtype) if dtype is not None else np.asarray(C_bits_or_values)
    return float(np.max(np.abs(C - C_ref)) / (np.max(np.abs(C_ref)) + 1e-6))

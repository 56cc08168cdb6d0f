"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and validates arguments before touching the GPU."""

import os
import re

import pytest

from w4a16_int4_weight_gb300 import build as wbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    wbuild.build()
    from w4a16_int4_weight_gb300 import binding
    return binding


def header_symbols():
    with open(os.path.join(ROOT, "include", "w4a16.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(w4a16_\w+)\s*\(", text, re.M)))


def test_library_exports_every_declared_symbol(B):
    syms = header_symbols()
    assert len(syms) >= 10
    for s in syms:
        assert hasattr(B.lib, s), s
    assert set(syms) == set(B.EXPORTED)
    assert B.version() == 100


def test_packed_layout_sizes(B):
    # K=4096: K/8 = 512 words (already a multiple of 4); scales N x 32 bf16
    tot, so, zo, ldq = B.packed_layout(4096, 4096, 128, "uint4b8", "bf16")
    assert ldq == 512 and so == 4096 * 512 * 4 and zo == 0
    assert tot == so + 4096 * 32 * 2
    # K=48: K/8 = 6 words -> pitch 8; sections on 256-byte boundaries
    tot, so, zo, ldq = B.packed_layout(8, 48, -1, "uint4", "fp16")
    assert ldq == 8 and so == 256 and zo == 512 and tot == 768
    # N=200: scale rows pad to 200 (already a multiple of 8), zero rows to 28 words
    tot, so, zo, ldq = B.packed_layout(200, 1024, 64, "uint4", "fp16")
    assert so == 200 * 128 * 4 and zo == so + 16 * 200 * 2 and tot == zo + 16 * 28 * 4
    tot, so, zo, ldq = B.packed_layout(11008, 4096, 32, "uint4", "bf16")
    assert so == 11008 * 512 * 4
    assert zo == so + 11008 * 128 * 2
    assert tot == zo + (11008 // 8) * 128 * 4


FAKE = 1 << 20   # any 256-aligned address: validation rejects before it is used


@pytest.mark.parametrize("args,needle", [
    (dict(K=24), "divisible by 16"),
    (dict(K=0), "out of range"),
    (dict(N=0), "out of range"),
    (dict(G=96), "group size"),
    (dict(K=4096 + 16, G=128), "divisible by group_size"),
    (dict(qtype=7), "quant type"),
    (dict(dtype=5), "dtype"),
    (dict(qtype=1, N=12), "divisible by 8"),
    (dict(qtype=1, zeros=0), "zeros"),
    (dict(qtype=0, zeros=FAKE), "NULL for uint4b8"),
    (dict(A=FAKE + 2), "A must be"),
    (dict(Wq=FAKE + 4), "Wq must be"),
    (dict(scales=0), "scales must be"),
    (dict(C=0), "C must be"),
    (dict(M=-1), "M=-1"),
    (dict(path=9), "unknown path"),
    (dict(path=6), "unknown path"),
    (dict(path=3), "dense copy"),
    (dict(path=1, M=65), "M <= 64"),
])
def test_gemm_rejects_invalid_arguments(B, args, needle):
    a = dict(A=FAKE, Wq=FAKE, scales=FAKE, zeros=None, Wdense=None, C=FAKE, M=4, N=256, K=4096,
             G=128, qtype=0, dtype=1, path=0)
    a.update(args)
    if a["qtype"] == 1 and "zeros" not in args:
        a["zeros"] = FAKE
    code = B.lib.w4a16_gemm_ex(a["A"], a["Wq"], a["scales"], a["zeros"], a["Wdense"], a["C"],
                               a["M"], a["N"], a["K"], a["G"], a["qtype"], a["dtype"], a["path"], None)
    assert code == B.ERR_INVALID_ARG
    assert needle in B.last_error()


def test_m_zero_is_a_noop(B):
    assert B.lib.w4a16_gemm(FAKE, FAKE, FAKE, None, FAKE, 0, 256, 4096, 128, 0, 1, None) == B.OK


def test_pack_and_dequant_validation(B):
    assert B.lib.w4a16_pack(FAKE + 1, FAKE, None, FAKE, 64, 64, 32, 0, 0, None) == B.ERR_INVALID_ARG
    assert "q must be" in B.last_error()
    assert B.lib.w4a16_pack(FAKE, FAKE, None, FAKE + 16, 64, 64, 32, 0, 0, None) == B.ERR_INVALID_ARG
    assert "Wpacked" in B.last_error()
    assert B.lib.w4a16_dequant(FAKE, FAKE, None, FAKE + 8, 64, 64, 32, 0, 0, None) == B.ERR_INVALID_ARG
    assert "W must be" in B.last_error()
    assert B.lib.w4a16_gemm_dense(FAKE, FAKE, FAKE, 4, 64, 40, 1, None) == B.ERR_INVALID_ARG
    assert "multiple of 16" in B.last_error()


def test_router(B):
    # small M -> decode; larger M -> fused with the tile in tensor memory; dense
    # copy used only for large M
    assert B.route(1, 4096, 4096, 128, "uint4b8", "bf16") == B.PATH_DECODE
    assert B.route(16, 11008, 4096, 64, "uint4", "bf16") == B.PATH_DECODE
    assert B.route(8, 11008, 4096, 32, "uint4", "bf16") == B.PATH_DECODE
    assert B.route(9, 11008, 4096, 32, "uint4", "bf16") == B.PATH_FUSED_TMEM   # G = 32 from 9 tokens, zero points
    assert B.route(9, 11008, 4096, 32, "uint4b8", "bf16") == B.PATH_DECODE     # ... but not without them
    assert B.route(16, 28672, 8192, 32, "uint4", "bf16") == B.PATH_DECODE      # ... nor on large layers
    assert B.route(16, 4096, 4096, -1, "uint4b8", "bf16") == B.PATH_DECODE     # one group
    assert B.route(17, 28672, 8192, 64, "uint4b8", "fp16") == B.PATH_FUSED_TMEM
    assert B.route(128, 28672, 8192, 64, "uint4", "bf16") == B.PATH_FUSED_TMEM
    assert B.route(129, 28672, 8192, 64, "uint4", "bf16") == B.PATH_FUSED_TMEM
    assert B.route(2048, 14336, 4096, 128, "uint4b8", "bf16") == B.PATH_FUSED_TMEM
    assert B.route(2048, 14336, 4096, 128, "uint4b8", "bf16", has_dense=True) == B.PATH_DENSE
    assert B.route(2047, 14336, 4096, 128, "uint4b8", "bf16", has_dense=True) == B.PATH_FUSED_TMEM
    assert B.route(4, 14336, 4096, 128, "uint4b8", "bf16", has_dense=True) == B.PATH_DECODE
    assert B.route(4, 14336, 4100, 128, "uint4b8", "bf16") == -1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib.util
    src = os.path.join(ROOT, "w4a16_int4_weight_gb300", "binding.py")
    # load a copy of the binding from a directory with no library next to it
    dst = tmp_path / "binding.py"
    dst.write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("binding_copy", dst)
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError, match="not built"):
        spec.loader.exec_module(mod)


@pytest.mark.parametrize("args,needle", [
    (dict(bias=FAKE + 1), "bias"),
    (dict(lda=4000), "lda=4000"),      # < K
    (dict(lda=4100), "lda=4100"),      # not a multiple of 8
    (dict(ldc=255), "ldc=255"),        # < N
])
def test_linear_rejects_bad_bias_and_strides(B, args, needle):
    a = dict(A=FAKE, lda=0, Wq=FAKE, scales=FAKE, zeros=None, bias=None, Wdense=None, C=FAKE, ldc=0,
             M=4, N=256, K=4096, G=128, qtype=0, dtype=1, path=0)
    a.update(args)
    code = B.lib.w4a16_linear(a["A"], a["lda"], a["Wq"], a["scales"], a["zeros"], a["bias"], a["Wdense"],
                              a["C"], a["ldc"], a["M"], a["N"], a["K"], a["G"], a["qtype"], a["dtype"],
                              a["path"], None)
    assert code == B.ERR_INVALID_ARG
    assert needle in B.last_error()


def test_pack_ex_rejects_bad_formats(B):
    assert B.lib.w4a16_pack_ex(FAKE, 7, FAKE, None, 0, FAKE + 256, 64, 64, 32, 0, 0, None) == B.ERR_INVALID_ARG
    assert "format" in B.last_error()
    assert B.lib.w4a16_pack_ex(FAKE, 1, FAKE, None, 5, FAKE + 256, 64, 64, 32, 0, 0, None) == B.ERR_INVALID_ARG
    assert "layout" in B.last_error()
    assert B.lib.w4a16_pack_ex(FAKE, 3, FAKE, None, 0, FAKE + 256, 60, 64, 32, 0, 0, None) == B.ERR_INVALID_ARG
    assert "N divisible by 8" in B.last_error()
    assert B.lib.w4a16_pack_ex(FAKE + 2, 1, FAKE, None, 0, FAKE + 256, 64, 64, 32, 0, 0, None) == B.ERR_INVALID_ARG
    assert "4-byte aligned" in B.last_error()


def test_cpython_marshalling_matches_ctypes(B):
    # the binding's per-call module forwards the same arguments to the same C
    # functions: identical status and message on every validation outcome
    if B._fastcall is None:
        pytest.skip("Python headers unavailable: the binding calls through ctypes only")
    base = [FAKE, FAKE, FAKE, None, None, FAKE, 4, 256, 4096, 128, 0, 1, 0, None]
    variants = [
        {9: 7},                      # group size
        {8: 4100},                   # K % 16
        {6: 0},                      # M = 0: no-op, OK without touching the GPU
        {10: 1},                     # uint4 without zero points
        {11: 5},                     # dtype
        {12: 9},                     # path
        {0: FAKE + 2},               # A alignment
        {6: -1},                     # negative M
    ]
    for v in variants:
        args = list(base)
        for i, x in v.items():
            args[i] = x
        got = B._gemm_ex_call(*args)
        msg = B.last_error()
        want = B.lib.w4a16_gemm_ex(*args)
        assert got == want, v
        if want != B.OK:
            assert B.last_error() == msg, v
    largs = [FAKE, 0, FAKE, FAKE, None, None, None, FAKE, 0, 4, 256, 4096, 7, 0, 1, 0, None]
    assert B._linear_call(*largs) == B.lib.w4a16_linear(*largs) == B.ERR_INVALID_ARG
    with pytest.raises(TypeError):
        B._gemm_ex_call(*base[:13])
    # buffers may also be passed as tensors (their data_ptr()); a bad object raises
    import torch
    buf = torch.zeros(16, dtype=torch.uint8)
    targs = [buf, buf, buf, None, None, buf] + base[6:]
    targs[9] = 7
    assert B._gemm_ex_call(*targs) == B.ERR_INVALID_ARG and "group size" in B.last_error()
    targs[1] = object()
    with pytest.raises(AttributeError):
        B._gemm_ex_call(*targs)


def test_out_of_range_integers_are_refused(B):
    # a size or enum that does not fit its C parameter raises instead of being
    # truncated to its low bits (2**32 + 128 must not pass as group size 128)
    import ctypes
    assert B.lib.w4a16_route(1, 4096, 4096, 128, 0, 1, 0) >= 0
    # ctypes integer objects and numpy integers are taken at their value
    import numpy as np
    assert B.lib.w4a16_route(ctypes.c_int64(1), np.int64(4096), 4096, ctypes.c_int(128), 0, 1, 0) == \
        B.lib.w4a16_route(1, 4096, 4096, 128, 0, 1, 0)
    with pytest.raises(ctypes.ArgumentError, match="TypeError"):
        B.lib.w4a16_route(ctypes.c_double(1.0), 4096, 4096, 128, 0, 1, 0)
    with pytest.raises(ctypes.ArgumentError, match="OverflowError"):
        B.lib.w4a16_route(1, 4096, 4096, 2**32 + 128, 0, 1, 0)
    with pytest.raises(ctypes.ArgumentError, match="OverflowError"):
        B.lib.w4a16_route(2**64 + 1, 4096, 4096, 128, 0, 1, 0)
    base = [FAKE, FAKE, FAKE, None, None, FAKE, 4, 256, 4096, 2**32 + 128, 0, 1, 0, None]
    with pytest.raises(ctypes.ArgumentError, match="OverflowError"):
        B.lib.w4a16_gemm_ex(*base)
    if B._fastcall is not None:
        with pytest.raises(OverflowError):
            B._gemm_ex_call(*base)
        base[9], base[6] = 128, 2**64
        with pytest.raises(OverflowError):
            B._gemm_ex_call(*base)

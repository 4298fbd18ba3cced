"""The C ABI boundary without a GPU: libfp4q.so builds for sm_103a, loads,
exports every entry point that include/fp4q.h declares, and rejects invalid
arguments on the host before touching the device."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp4q.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4q_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from fp4_block_scaled_bf16_gb300 import build
    path = build.build()
    L = ctypes.CDLL(path)
    L.fp4q_status_string.restype = ctypes.c_char_p
    return L


def test_header_declares_the_boundary():
    names = declared_functions()
    assert names == sorted(["fp4q_amax", "fp4q_tensor_scale", "fp4q_quantize", "fp4q_dequantize",
                            "fp4q_gemm", "fp4q_get_device_status", "fp4q_status_string"] +
                           [n for n in names if n not in (
                               "fp4q_amax", "fp4q_tensor_scale", "fp4q_quantize", "fp4q_dequantize",
                               "fp4q_gemm", "fp4q_get_device_status", "fp4q_status_string")])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_lists_every_export():
    names = declared_functions()
    src = open(os.path.join(ROOT, "fp4_block_scaled_bf16_gb300", "fp4q.py")).read()
    for n in names:
        assert f'"{n}"' in src, n


def test_status_strings(lib):
    for code in range(7):
        s = lib.fp4q_status_string(code)
        assert s and s != b"unknown status"
    assert lib.fp4q_status_string(99) == b"unknown status"


def _q(lib, **kw):
    a = dict(inp=16, rows=32, cols=32, axis=0, fmt=0, ts=16, rnd=0, pr=16, sr=16, pc=16, sc=16)
    a.update(kw)
    P = ctypes.c_void_p
    f = lib.fp4q_quantize
    f.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, ctypes.c_int,
                  ctypes.c_uint64, P, P, P, P, P, P, P]
    return f(P(a["inp"]), a["rows"], a["cols"], a["axis"], a["fmt"], P(a["ts"]), a["rnd"], 0,
             P(a["pr"]), P(a["sr"]), P(a["pc"]), P(a["sc"]), None, None, None)


def test_host_validation_rejects_before_launch(lib):
    ERR_ARG, ERR_SHAPE, ERR_ALIGN = 1, 2, 3
    assert _q(lib, rows=17) == ERR_SHAPE
    assert _q(lib, cols=8) == ERR_SHAPE
    assert _q(lib, rows=-16) == ERR_SHAPE
    assert _q(lib, axis=4) == ERR_ARG
    assert _q(lib, axis=1, rows=2 ** 32, cols=2 ** 32) == ERR_SHAPE   # > 2^31 - 1 tiles
    assert _q(lib, axis=2, rows=2 ** 26, cols=2 ** 26) == ERR_SHAPE
    assert _q(lib, axis=3, pc=0) == ERR_ARG          # 16 x 16 scaling writes both layouts
    assert _q(lib, axis=3, pr=0) == ERR_ARG
    assert _q(lib, fmt=2) == ERR_ARG
    assert _q(lib, rnd=2) == ERR_ARG
    assert _q(lib, ts=0) == ERR_ARG
    assert _q(lib, inp=0) == ERR_ARG
    assert _q(lib, pr=0) == ERR_ARG
    assert _q(lib, axis=1, pc=0) == ERR_ARG
    assert _q(lib, inp=24) == ERR_ALIGN
    assert _q(lib, axis=2, sc=40) == ERR_ALIGN

    P = ctypes.c_void_p
    g = lib.fp4q_gemm
    g.argtypes = [P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P,
                  ctypes.c_int, P]
    ok = P(16)
    assert g(ok, ok, ok, ok, ok, ok, 128, 128, 96, 0, ok, 0, None) == ERR_SHAPE    # K % 64
    assert g(ok, ok, ok, ok, ok, ok, 65535 * 256 + 1, 128, 128, 0, ok, 0, None) == ERR_SHAPE
    assert g(ok, ok, ok, ok, ok, ok, 128, 2 ** 31, 128, 0, ok, 0, None) == ERR_SHAPE
    assert g(ok, ok, ok, ok, ok, ok, 128, 128, 128, 5, ok, 0, None) == ERR_ARG
    assert g(ok, ok, ok, ok, ok, ok, 128, 128, 128, 0, None, 0, None) == ERR_ARG
    assert g(None, ok, ok, ok, ok, ok, 128, 128, 128, 0, ok, 0, None) == ERR_ARG
    assert g(P(8), ok, ok, ok, ok, ok, 128, 128, 128, 0, ok, 0, None) == ERR_ALIGN
    assert g(ok, ok, ok, ok, ok, ok, 0, 128, 128, 0, ok, 0, None) == 0             # empty: no-op

    t = lib.fp4q_tensor_scale
    t.argtypes = [P, ctypes.c_int, ctypes.c_float, P, P]
    assert t(ok, 0, 3.0, ok, None) == ERR_ARG      # headroom not a power of two
    assert t(ok, 0, 0.5, ok, None) == ERR_ARG
    assert t(ok, 2, 1.0, ok, None) == ERR_ARG
    a = lib.fp4q_amax
    a.argtypes = [P, ctypes.c_int64, P, P]
    assert a(ok, 16, None, None) == ERR_ARG
    assert a(P(2), 16, ok, None) == ERR_ALIGN
    assert a(ok, 16, P(18), None) == ERR_ALIGN          # scalars: 4-byte alignment
    s = lib.fp4q_get_device_status
    s.argtypes = [P, P]
    assert s(None, None) == ERR_ARG

    i64 = ctypes.c_int64
    r = lib.fp4q_rebias_scales
    r.argtypes = [P, i64, i64, ctypes.c_int, P, P, P, P]
    buf = ctypes.create_string_buffer(64 * 16 + 16)
    base = (ctypes.addressof(buf) + 15) & ~15
    src, dst = P(base), P(base + 16 * 32)   # 16 rows of 16 codes, apart
    assert r(src, 16, 24, 1, dst, ok, ok, None) == ERR_SHAPE      # nblocks % 16
    assert r(src, -1, 16, 1, dst, ok, ok, None) == ERR_SHAPE
    assert r(src, 16, 16, 1, dst, None, ok, None) == ERR_ARG      # factor
    assert r(src, 16, 16, 1, dst, ok, None, None) == ERR_ARG      # flag
    assert r(None, 16, 16, 1, dst, ok, ok, None) == ERR_ARG
    assert r(src, 16, 16, 1, P(base + 8), ok, ok, None) == ERR_ALIGN
    assert r(src, 16, 16, 1, ok, ok, P(18), None) == ERR_ALIGN
    assert r(src, 16, 16, 1, P(base + 16 * 8), ok, ok, None) == ERR_ARG   # overlapping in/out
    assert r(src, 0, 16, 1, dst, ok, ok, None) == 0                     # no rows: no-op

    r2 = lib.fp4q_rebias_scales_two_windows
    r2.argtypes = [P, i64, i64, P, P, P, P, P, P]
    buf2 = ctypes.create_string_buffer(16 * 16 + 16)   # a third 16 x 16 array, apart from src and dst
    lo = P((ctypes.addressof(buf2) + 15) & ~15)
    assert r2(src, 16, 24, dst, lo, ok, ok, ok, None) == ERR_SHAPE     # nblocks % 16
    assert r2(src, 16, 16, dst, lo, None, ok, ok, None) == ERR_ARG     # high factors
    assert r2(src, 16, 16, dst, lo, ok, None, ok, None) == ERR_ARG     # low factors
    assert r2(src, 16, 16, dst, lo, ok, ok, None, None) == ERR_ARG     # flag
    assert r2(src, 16, 16, dst, None, ok, ok, ok, None) == ERR_ARG
    assert r2(src, 16, 16, dst, P(base + 8), ok, ok, ok, None) == ERR_ALIGN
    assert r2(src, 16, 16, dst, lo, ok, P(18), ok, None) == ERR_ALIGN
    assert r2(src, 16, 16, dst, P(base + 16 * 8), ok, ok, ok, None) == ERR_ARG   # low codes over the input
    assert r2(src, 16, 16, dst, P(base + 16 * 40), ok, ok, ok, None) == ERR_ARG  # the two outputs overlap
    assert r2(src, 0, 16, dst, lo, ok, ok, ok, None) == 0                       # no rows: no-op

    w = lib.fp4q_gemm_nvfp4_two_windows
    w.argtypes = [P, P, P, P, P, P, P, P, P, i64, i64, i64, P, P, ctypes.c_int, P]
    assert w(ok, ok, ok, ok, ok, ok, ok, ok, ok, 128, 128, 128, None, ok, 0, None) == ERR_SHAPE   # K % 256
    assert w(ok, ok, None, ok, ok, ok, ok, ok, ok, 128, 128, 256, None, ok, 0, None) == ERR_ARG   # low codes
    assert w(ok, ok, ok, None, ok, ok, ok, ok, ok, 128, 128, 256, None, ok, 0, None) == ERR_ARG   # A factors
    assert w(ok, ok, ok, ok, ok, ok, ok, None, ok, 128, 128, 256, None, ok, 0, None) == ERR_ARG   # B factor
    assert w(ok, ok, P(8), ok, ok, ok, ok, ok, ok, 128, 128, 256, None, ok, 0, None) == ERR_ALIGN
    assert w(ok, ok, ok, P(18), ok, ok, ok, ok, ok, 128, 128, 256, None, ok, 0, None) == ERR_ALIGN
    assert w(ok, ok, ok, ok, ok, ok, ok, ok, ok, 0, 128, 256, None, ok, 0, None) == 0   # empty: no-op

    n = lib.fp4q_gemm_nvfp4_rebiased
    n.argtypes = [P, P, P, P, P, P, P, P, i64, i64, i64, P, P, ctypes.c_int, P]
    assert n(ok, ok, ok, ok, ok, ok, ok, ok, 128, 128, 128, None, ok, 0, None) == ERR_SHAPE   # K % 256
    assert n(ok, ok, None, ok, ok, ok, ok, ok, 128, 128, 256, None, ok, 0, None) == ERR_ARG  # A factor
    assert n(ok, ok, ok, ok, ok, ok, None, ok, 128, 128, 256, None, ok, 0, None) == ERR_ARG  # B factor
    assert n(ok, ok, P(18), ok, ok, ok, ok, ok, 128, 128, 256, None, ok, 0, None) == ERR_ALIGN
    assert n(ok, ok, ok, ok, ok, ok, ok, ok, 128, 128, 256, P(18), ok, 0, None) == ERR_ALIGN
    assert n(ok, ok, ok, ok, ok, ok, ok, ok, 0, 128, 256, None, ok, 0, None) == 0   # empty: no-op

    nq = lib.fp4q_gemm_nvfp4_rebiased_quantize
    nq.argtypes = [P, P, P, P, P, P, P, P, i64, i64, i64, P, ctypes.c_int, P, P, P, P, P, P]
    assert nq(ok, ok, ok, ok, ok, ok, ok, ok, 128, 48, 256, None, 0, ok, ok, ok, ok, None, None) == ERR_SHAPE  # N % 32
    assert nq(ok, ok, ok, ok, ok, ok, ok, ok, 128, 64, 256, None, 0, ok, ok, None, ok, None, None) == ERR_ARG
    assert nq(ok, ok, ok, ok, ok, ok, ok, ok, 128, 64, 256, None, 0, None, ok, ok, ok, None, None) == ERR_ARG
    assert nq(ok, ok, ok, ok, ok, ok, ok, ok, 128, 64, 256, None, 3, ok, ok, ok, ok, None, None) == ERR_ARG
    assert nq(ok, ok, ok, ok, ok, ok, ok, ok, 128, 64, 256, None, 0, ok, ok, ok, ok, P(18), None) == ERR_ALIGN
    assert nq(ok, ok, ok, ok, ok, ok, ok, ok, 0, 64, 256, None, 0, ok, ok, ok, ok, None, None) == 0
    qi = lib.fp4q_gemm_quantize_if
    qi.argtypes = [P, P, P, P, P, P, i64, i64, i64, ctypes.c_int, P, P, P, P, P, P, P]
    assert qi(ok, ok, ok, ok, ok, ok, 128, 64, 128, 0, None, ok, ok, ok, ok, None, None) == ERR_ARG   # flag
    assert qi(ok, ok, ok, ok, ok, ok, 128, 64, 128, 0, ok, ok, ok, None, ok, None, None) == ERR_ARG   # payload
    assert qi(ok, ok, ok, ok, ok, ok, 128, 48, 128, 0, ok, ok, ok, ok, ok, None, None) == ERR_SHAPE
    assert qi(ok, ok, ok, ok, ok, ok, 0, 64, 128, 0, ok, ok, ok, ok, ok, None, None) == 0

    c = lib.fp4q_gemm_if
    c.argtypes = [P, P, P, P, P, P, i64, i64, i64, ctypes.c_int, P, P, ctypes.c_int, P]
    assert c(ok, ok, ok, ok, ok, ok, 128, 128, 128, 0, None, ok, 0, None) == ERR_ARG     # flag required
    assert c(ok, ok, ok, ok, ok, ok, 128, 128, 128, 0, P(18), ok, 0, None) == ERR_ALIGN
    assert c(ok, ok, ok, ok, ok, ok, 128, 128, 96, 0, ok, ok, 0, None) == ERR_SHAPE
    assert c(ok, ok, ok, ok, ok, ok, 0, 128, 128, 0, ok, ok, 0, None) == 0


def test_product_path_has_no_fallback():
    # the binding raises at import time when the library is missing; it never
    # routes through the oracle or the CPU
    src = open(os.path.join(ROOT, "fp4_block_scaled_bf16_gb300", "fp4q.py")).read()
    assert "oracle" not in src.replace("# ", "")
    for f in os.listdir(os.path.join(ROOT, "fp4_block_scaled_bf16_gb300")):
        if f.endswith(".py"):
            body = open(os.path.join(ROOT, "fp4_block_scaled_bf16_gb300", f)).read()
            assert "import oracle" not in body and "from oracle" not in body, f

"""CPU oracle for UE5M3-scaled FP4 quantisation and the block-scaled GEMM.

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by bench.py's CPU-baseline / reference leg, never by the product package.
The arithmetic lives in ``fp4q_oracle.c`` (plain scalar C, binary32 without
FMA contraction, binary64 GEMM); this module compiles it with gcc on first use
and marshals numpy arrays to it.  It shares nothing with the CUDA library.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (E2M1 payloads, UE5M3 block-16 scales, periodic tensor scaling,
selective stochastic rounding on backward gradients).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

UE5M3 = 0
UE4M3 = 1
ROW = 0
COL = 1
BOTH = 2
RNE = 0
SR = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4q_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fno-finite-math-only"]
# FP4Q_ORACLE_SANITIZE=1 builds a separate AddressSanitizer + UBSan copy (the
# sanitizer runtimes must then be preloaded, e.g.
#   LD_PRELOAD="$(gcc -print-file-name=libasan.so):$(gcc -print-file-name=libubsan.so)"
#   ASAN_OPTIONS=detect_leaks=0 FP4Q_ORACLE_SANITIZE=1 python -m pytest tests -m "not gpu" -k oracle)
if os.environ.get("FP4Q_ORACLE_SANITIZE") == "1":
    _SO = os.path.join(_BUILD, "liboracle_sanitize.so")
    _CFLAGS = [f for f in _CFLAGS if f != "-O2"] + ["-O1", "-g", "-fsanitize=address,undefined",
                                                     "-fno-sanitize-recover=all"]
else:
    _SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (contraction off) if missing or stale."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _SO + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, u64, u32, f32, i32 = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                   ctypes.c_float, ctypes.c_int)
        sig = {
            "orc_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_scale_decode": (ctypes.c_double, [ctypes.c_uint8, i32]),
            "orc_scale_max": (ctypes.c_double, [i32]),
            "orc_scale_encode": (ctypes.c_uint8, [f32, i32, P]),
            "orc_e2m1_rne": (ctypes.c_uint8, [f32]),
            "orc_e2m1_sr": (ctypes.c_uint8, [f32, u32]),
            "orc_philox4x32_10": (None, [P, P, P]),
            "orc_philox4x64_10": (None, [P, P, P]),
            "orc_sr_uniform": (u32, [u64, u64, u32]),
            "orc_amax_bf16": (f32, [P, i64, P]),
            "orc_tensor_scale": (f32, [f32, i32, f32]),
            "orc_quantize": (None, [P, i64, i64, i32, i32, f32, i32, u64, P, P, P]),
            "orc_quantize_band": (None, [P, i64, i64, i64, i32, i32, f32, i32, u64, P, P, P]),
            "orc_quantize_2d": (None, [P, i64, i64, i32, f32, i32, u64, P, P, P, P, P]),
            "orc_dequantize": (None, [P, P, i64, i64, i32, f32, P, P]),
            "orc_gemm": (None, [P, P, f32, P, P, f32, i64, i64, i64, i32, P, P, i64, P]),
            "orc_deq_es_matrix": (None, [P, P, i64, i64, i32, P]),
            "orc_e2m1_rne_array": (None, [P, i64, P]),
            "orc_e2m1_sr_array": (None, [P, P, i64, P]),
            "orc_scale_encode_array": (None, [P, i64, i32, P, P]),
            "orc_sr_uniform_array": (None, [u64, P, i64, u32, P]),
            "orc_rebias_scales": (None, [P, i64, i64, i32, P, P, P]),
            "orc_rebias_scales2": (None, [P, i64, i64, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats
def e2m1_decode(nib: int) -> float:
    return _load().orc_e2m1_decode(int(nib))


def scale_decode(code: int, fmt: int = UE5M3) -> float:
    return _load().orc_scale_decode(int(code), int(fmt))


def scale_max(fmt: int = UE5M3) -> float:
    return _load().orc_scale_max(int(fmt))


def scale_encode(s, fmt: int = UE5M3):
    """Vectorised scale encode: returns (codes uint8, saturated uint8)."""
    s = _c(np.atleast_1d(s), np.float32)
    out = np.empty(s.shape, np.uint8)
    sat = np.empty(s.shape, np.uint8)
    _load().orc_scale_encode_array(_ptr(s), s.size, int(fmt), _ptr(out), _ptr(sat))
    return out, sat


def e2m1_rne(q) -> np.ndarray:
    q = _c(np.atleast_1d(q), np.float32)
    out = np.empty(q.shape, np.uint8)
    _load().orc_e2m1_rne_array(_ptr(q), q.size, _ptr(out))
    return out


def e2m1_sr(q, u16) -> np.ndarray:
    """Stochastic rounding of q with 16-bit uniform integers u16 (low 16 bits used)."""
    q = _c(np.atleast_1d(q), np.float32)
    rb = _c(np.broadcast_to(np.asarray(u16, np.uint32), q.shape), np.uint32)
    out = np.empty(q.shape, np.uint8)
    _load().orc_e2m1_sr_array(_ptr(q), _ptr(rb), q.size, _ptr(out))
    return out


# ---------------------------------------------------------------- philox
def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.empty(4, np.uint32)
    _load().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def philox4x64_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint64)
    k = _c(key, np.uint64)
    out = np.empty(4, np.uint64)
    _load().orc_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_uniforms(seed: int, idx, axis: int) -> np.ndarray:
    """The 16-bit uniforms elements with logical indices idx draw on an axis."""
    idx = _c(np.atleast_1d(idx), np.uint64)
    out = np.empty(idx.shape, np.uint32)
    _load().orc_sr_uniform_array(ctypes.c_uint64(seed), _ptr(idx), idx.size, int(axis), _ptr(out))
    return out


# ---------------------------------------------------------------- tensor level
def _as_bf16_bits(x) -> np.ndarray:
    """Accept a uint16 array of BF16 patterns or a torch bfloat16 tensor."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        x = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    x = np.asarray(x)
    if x.dtype != np.uint16:
        raise TypeError("expected BF16 bit patterns (uint16) or a torch.bfloat16 tensor")
    return np.ascontiguousarray(x)


def amax(x) -> tuple[float, bool]:
    x = _as_bf16_bits(x)
    bad = ctypes.c_int(0)
    m = _load().orc_amax_bf16(_ptr(x), x.size, ctypes.byref(bad))
    return float(np.float32(m)), bool(bad.value)


def tensor_scale(amax_value: float, fmt: int = UE5M3, headroom: float = 1.0) -> float:
    return float(np.float32(_load().orc_tensor_scale(float(amax_value), int(fmt), float(headroom))))


def quantize(x, axis: int, T: float, fmt: int = UE5M3, rnd: int = RNE, seed: int = 0,
             row_base: int = 0):
    """Quantise a [rows, cols] BF16 tensor along one axis.

    Returns (payload uint8 [o, i/2], scales uint8 [o, i/16], stats uint64[4])
    with (o, i) = (rows, cols) for ROW and (cols, rows) for COL.

    row_base > 0 treats x as rows row_base .. row_base + rows - 1 of a larger
    tensor with the same columns: the result is that tensor's output for
    those rows (ROW), or for that span of every column (COL); only the
    stochastic-rounding counters (logical indices) depend on it.
    """
    x = _as_bf16_bits(x)
    rows, cols = x.shape
    if rows % 16 or cols % 16 or row_base % 16 or row_base < 0:
        raise ValueError("rows, cols and row_base must be non-negative multiples of 16")
    outer, inner = (rows, cols) if axis == ROW else (cols, rows)
    payload = np.zeros((outer, inner // 2), np.uint8)
    scales = np.zeros((outer, inner // 16), np.uint8)
    stats = np.zeros(4, np.uint64)
    _load().orc_quantize_band(_ptr(x), int(row_base), rows, cols, int(axis), int(fmt), float(T),
                              int(rnd), ctypes.c_uint64(seed), _ptr(payload), _ptr(scales),
                              _ptr(stats))
    return payload, scales, stats


def quantize_2d(x, T: float, fmt: int = UE5M3, rnd: int = RNE, seed: int = 0):
    """One scale per 16 x 16 tile, both layouts from one quantisation.

    Returns (payload_row [rows, cols/2], scales_row [rows, cols/16],
    payload_col [cols, rows/2], scales_col [cols, rows/16], stats uint64[4]).
    """
    x = _as_bf16_bits(x)
    rows, cols = x.shape
    if rows % 16 or cols % 16:
        raise ValueError("rows and cols must be multiples of 16")
    pr = np.zeros((rows, cols // 2), np.uint8)
    sr = np.zeros((rows, cols // 16), np.uint8)
    pc = np.zeros((cols, rows // 2), np.uint8)
    sc = np.zeros((cols, rows // 16), np.uint8)
    stats = np.zeros(4, np.uint64)
    _load().orc_quantize_2d(_ptr(x), rows, cols, int(fmt), float(T), int(rnd), ctypes.c_uint64(seed),
                            _ptr(pr), _ptr(sr), _ptr(pc), _ptr(sc), _ptr(stats))
    return pr, sr, pc, sc, stats


def dequantize(payload, scales, T: float, fmt: int = UE5M3):
    """Returns (binary32 values, their BF16 rounding as uint16 patterns)."""
    payload = _c(payload, np.uint8)
    scales = _c(scales, np.uint8)
    outer, inner = payload.shape[0], payload.shape[1] * 2
    f = np.empty((outer, inner), np.float32)
    b = np.empty((outer, inner), np.uint16)
    _load().orc_dequantize(_ptr(payload), _ptr(scales), outer, inner, int(fmt), float(T),
                           _ptr(f), _ptr(b))
    return f, b


def deq_es(payload, scales, fmt: int = UE5M3) -> np.ndarray:
    """e * s of every element as binary64 (exact), [outer, inner]."""
    payload = _c(payload, np.uint8)
    scales = _c(scales, np.uint8)
    outer, inner = payload.shape[0], payload.shape[1] * 2
    out = np.empty((outer, inner), np.float64)
    _load().orc_deq_es_matrix(_ptr(payload), _ptr(scales), outer, inner, int(fmt), _ptr(out))
    return out


def rebias_scales(scales, per_row: bool = True):
    """UE5M3 scale codes [rows, nb] -> (UE4M3 codes [rows, nb], factors
    [rows] or [1], fits): v = f * v4 exactly for every group whose non-zero
    scales lie in 14 binades -- per row, the row's top 14; per tensor, the
    fixed binades 3..16 (f = 2^9)."""
    scales = _c(scales, np.uint8)
    rows, nb = scales.shape
    out = np.empty_like(scales)
    f = np.empty(rows if per_row else 1, np.float32)
    nofit = np.zeros(1, np.int32)
    _load().orc_rebias_scales(_ptr(scales), rows, nb, int(bool(per_row)), _ptr(out), _ptr(f), _ptr(nofit))
    return out, f, not bool(nofit[0])


def rebias_scales2(scales):
    """UE5M3 scale codes [rows, nb] -> (hi codes, lo codes, hi factors, lo
    factors, fits): each row's top 14 binades as UE4M3 codes times
    2^(e_top - 7), the 14 below them times 2^(e_top - 21); every value is
    hi * f_hi + lo * f_lo with one of the two codes zero; fits unless a
    value lies below both windows."""
    scales = _c(scales, np.uint8)
    rows, nb = scales.shape
    hi, lo = np.empty_like(scales), np.empty_like(scales)
    fh, fl = np.empty(rows, np.float32), np.empty(rows, np.float32)
    nofit = np.zeros(1, np.int32)
    _load().orc_rebias_scales2(_ptr(scales), rows, nb, _ptr(hi), _ptr(lo), _ptr(fh), _ptr(fl), _ptr(nofit))
    return hi, lo, fh, fl, not bool(nofit[0])


def gemm(A, As, TA, B, Bs, TB, fmt: int = UE5M3, ms=None, ns=None) -> np.ndarray:
    """(T_A T_B) * sum_k deq(A)[m,k] deq(B)[n,k] in binary64.

    Full [M, N] when ms is None, else the listed (ms[t], ns[t]) entries.
    """
    A, As, B, Bs = (_c(a, np.uint8) for a in (A, As, B, Bs))
    M, K = A.shape[0], A.shape[1] * 2
    N = B.shape[0]
    if ms is None:
        out = np.empty((M, N), np.float64)
        _load().orc_gemm(_ptr(A), _ptr(As), float(TA), _ptr(B), _ptr(Bs), float(TB),
                         M, N, K, int(fmt), None, None, 0, _ptr(out))
        return out
    ms = _c(ms, np.int64)
    ns = _c(ns, np.int64)
    out = np.empty(ms.shape, np.float64)
    _load().orc_gemm(_ptr(A), _ptr(As), float(TA), _ptr(B), _ptr(Bs), float(TB),
                     M, N, K, int(fmt), _ptr(ms), _ptr(ns), ms.size, _ptr(out))
    return out


class PeriodicScaler:
    """Periodic tensor scaling ("UE5M3 FP4 Block Scaling ...", Abstract: the
    wider UE5M3 range permits periodic rather than current tensor scaling).

    Reading: the tensor scale is refreshed every ``period`` quantisations from
    the last observed amax (step 0 uses an explicit amax of the first tensor);
    every quantisation records its own tensor's amax for the next refresh.
    """

    def __init__(self, period: int = 16, fmt: int = UE5M3, headroom: float = 1.0):
        self.period, self.fmt, self.headroom = period, fmt, headroom
        self.step = 0
        self.T = 1.0
        self.last_amax = None

    def quantize(self, x, axis=ROW, rnd=RNE, seed=0):
        if self.step % self.period == 0:
            if self.last_amax is None:
                self.last_amax = amax(x)[0]
            self.T = tensor_scale(self.last_amax, self.fmt, self.headroom)
        out = quantize(x, axis, self.T, self.fmt, rnd, seed)
        self.last_amax = amax(x)[0]
        self.step += 1
        return out

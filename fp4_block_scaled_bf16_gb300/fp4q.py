"""Python binding of libfp4q.so (include/fp4q.h): argument marshalling only.

Every function named ``fp4q_*`` here calls the C entry point of the same name
with the device pointers of the torch tensors it is given, on the current
torch CUDA stream; all arithmetic happens in the library's CUDA kernels.  The
lower-case helpers (``quantize``, ``gemm`` ...) only allocate the output
tensors with torch before calling them.

Importing this module loads the library and raises if it is missing: there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfp4q.so")

OK, ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_CUDA, ERR_NONFINITE, ERR_TIMEOUT = range(7)
AXIS_ROW, AXIS_COL, AXIS_BOTH, AXIS_BOTH_2D = 0, 1, 2, 3
RNE, SR = 0, 1
UE5M3, UE4M3 = 0, 1

# every symbol include/fp4q.h declares
EXPORTS = ("fp4q_amax", "fp4q_tensor_scale", "fp4q_quantize", "fp4q_dequantize", "fp4q_gemm",
           "fp4q_gemm_quantize", "fp4q_gemm_nvfp4", "fp4q_rebias_scales", "fp4q_gemm_nvfp4_rebiased",
           "fp4q_gemm_if", "fp4q_gemm_nvfp4_rebiased_quantize", "fp4q_gemm_quantize_if",
           "fp4q_rebias_scales_two_windows", "fp4q_gemm_nvfp4_two_windows",
           "fp4q_get_device_status", "fp4q_status_string")


class Fp4qError(RuntimeError):
    def __init__(self, fn, code, lib):
        msg = lib.fp4q_status_string(code).decode()
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libfp4q.so not built at {path}; run "
                          "`python -m fp4_block_scaled_bf16_gb300.build`")
    lib = ctypes.CDLL(path)
    P, i64, i32, u64, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                             ctypes.c_float)
    lib.fp4q_amax.argtypes = [P, i64, P, P]
    lib.fp4q_tensor_scale.argtypes = [P, i32, f32, P, P]
    lib.fp4q_quantize.argtypes = [P, i64, i64, i32, i32, P, i32, u64, P, P, P, P, P, P, P]
    lib.fp4q_dequantize.argtypes = [P, P, i64, i64, i32, P, P, i32, P]
    lib.fp4q_gemm.argtypes = [P, P, P, P, P, P, i64, i64, i64, i32, P, i32, P]
    lib.fp4q_gemm_quantize.argtypes = [P, P, P, P, P, P, i64, i64, i64, i32, P, P, P, P, P, P]
    lib.fp4q_gemm_nvfp4.argtypes = [P, P, P, P, P, P, i64, i64, i64, P, i32, P]
    lib.fp4q_rebias_scales.argtypes = [P, i64, i64, i32, P, P, P, P]
    lib.fp4q_rebias_scales_two_windows.argtypes = [P, i64, i64, P, P, P, P, P, P]
    lib.fp4q_gemm_nvfp4_two_windows.argtypes = [P, P, P, P, P, P, P, P, P, i64, i64, i64, P, P, i32, P]
    lib.fp4q_gemm_nvfp4_rebiased.argtypes = [P, P, P, P, P, P, P, P, i64, i64, i64, P, P, i32, P]
    lib.fp4q_gemm_if.argtypes = [P, P, P, P, P, P, i64, i64, i64, i32, P, P, i32, P]
    lib.fp4q_gemm_nvfp4_rebiased_quantize.argtypes = [P, P, P, P, P, P, P, P, i64, i64, i64, P, i32, P, P, P, P,
                                                      P, P]
    lib.fp4q_gemm_quantize_if.argtypes = [P, P, P, P, P, P, i64, i64, i64, i32, P, P, P, P, P, P, P]
    lib.fp4q_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), P]
    lib.fp4q_status_string.argtypes = [i32]
    lib.fp4q_status_string.restype = ctypes.c_char_p
    for name in EXPORTS[:-1]:
        getattr(lib, name).restype = i32
    return lib


_lib = load_library()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn, code):
    if code != OK:
        raise Fp4qError(fn, code, _lib)


# ------------------------------------------------------------ validation
# The library trusts the sizes it is given: a buffer smaller than they imply
# would be read or written out of bounds on the device.  So every entry point
# checks here, before the call, that each tensor has exactly the shape the
# sizes imply, the expected dtype, is contiguous, and lives on the current
# CUDA device (the library launches on the current device's current stream).
# Shapes are checked before devices, so that these checks run without a GPU.
def _mat(t, name, shape, dtype):
    if t is None:
        raise ValueError(f"{name} is required")
    shape = tuple(int(d) for d in shape)
    if tuple(t.shape) != shape:
        raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _scalar(t, name, n=1, dtype=torch.float32):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.numel() < n:
        raise ValueError(f"{name} must hold at least {n} element(s), got {t.numel()}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _sizes(**kw):
    for k, v in kw.items():
        if int(v) < 0:
            raise ValueError(f"{k} must be >= 0, got {v}")
        if int(v) % 16:
            raise ValueError(f"{k} must be a multiple of 16, got {v}")


def _on_device(*named):
    """Every given tensor is a contiguous CUDA tensor on the current device."""
    cur = torch.cuda.current_device() if torch.cuda.is_available() else None
    for name, t in named:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device.index != cur:
            raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{cur}; "
                             "call inside torch.cuda.device(...) of the tensors' device")


def _out_dtype(out):
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"out must be bfloat16 or float32, got {out.dtype}")


# ------------------------------------------------------------ C entry points
def fp4q_amax(x: torch.Tensor, out_amax: torch.Tensor) -> None:
    if x.dtype != torch.bfloat16:
        raise ValueError(f"x must be torch.bfloat16, got {x.dtype}")
    _scalar(out_amax, "out_amax")
    _on_device(("x", x), ("out_amax", out_amax))
    _check("fp4q_amax", _lib.fp4q_amax(_ptr(x), x.numel(), _ptr(out_amax), _stream()))


def fp4q_tensor_scale(amax: torch.Tensor, fmt: int, headroom: float, out_scale: torch.Tensor) -> None:
    _scalar(amax, "amax")
    _scalar(out_scale, "out_scale")
    _on_device(("amax", amax), ("out_scale", out_scale))
    _check("fp4q_tensor_scale",
           _lib.fp4q_tensor_scale(_ptr(amax), fmt, headroom, _ptr(out_scale), _stream()))


def fp4q_quantize(x, axis, fmt, tensor_scale, rnd, seed, payload_row, scales_row, payload_col,
                  scales_col, stats=None, amax=None) -> None:
    if x.dim() != 2:
        raise ValueError(f"x must be 2-D [rows, cols], got shape {tuple(x.shape)}")
    rows, cols = x.shape
    _sizes(rows=rows, cols=cols)
    u8 = torch.uint8
    _mat(x, "x", (rows, cols), torch.bfloat16)
    row = axis in (AXIS_ROW, AXIS_BOTH, AXIS_BOTH_2D)
    col = axis in (AXIS_COL, AXIS_BOTH, AXIS_BOTH_2D)
    if not (row or col):
        raise ValueError(f"unknown axis {axis}")
    if row:
        _mat(payload_row, "payload_row", (rows, cols // 2), u8)
        _mat(scales_row, "scales_row", (rows, cols // 16), u8)
    else:
        payload_row = scales_row = None
    if col:
        _mat(payload_col, "payload_col", (cols, rows // 2), u8)
        _mat(scales_col, "scales_col", (cols, rows // 16), u8)
    else:
        payload_col = scales_col = None
    _scalar(tensor_scale, "tensor_scale")
    if stats is not None:
        _scalar(stats, "stats", 4 * (2 if axis == AXIS_BOTH else 1), torch.int64)
    if amax is not None:
        _scalar(amax, "amax")
    _on_device(("x", x), ("payload_row", payload_row), ("scales_row", scales_row),
               ("payload_col", payload_col), ("scales_col", scales_col),
               ("tensor_scale", tensor_scale), ("stats", stats), ("amax", amax))
    _check("fp4q_quantize", _lib.fp4q_quantize(
        _ptr(x), rows, cols, axis, fmt, _ptr(tensor_scale), rnd, ctypes.c_uint64(seed),
        _ptr(payload_row), _ptr(scales_row), _ptr(payload_col), _ptr(scales_col),
        _ptr(stats), _ptr(amax), _stream()))


def fp4q_dequantize(payload, scales, rows, cols, fmt, tensor_scale, out) -> None:
    _sizes(rows=rows, cols=cols)
    _mat(payload, "payload", (rows, cols // 2), torch.uint8)
    _mat(scales, "scales", (rows, cols // 16), torch.uint8)
    _out_dtype(out)
    _mat(out, "out", (rows, cols), out.dtype)
    _scalar(tensor_scale, "tensor_scale")
    _on_device(("payload", payload), ("scales", scales), ("tensor_scale", tensor_scale), ("out", out))
    f32 = out.dtype == torch.float32
    _check("fp4q_dequantize", _lib.fp4q_dequantize(
        _ptr(payload), _ptr(scales), rows, cols, fmt, _ptr(tensor_scale), _ptr(out), int(f32),
        _stream()))


def _gemm_operands(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K):
    if M < 0 or N < 0:
        raise ValueError(f"M and N must be >= 0, got {M}, {N}")
    _sizes(K=K)
    _mat(A, "A", (M, K // 2), torch.uint8)
    _mat(A_scales, "A_scales", (M, K // 16), torch.uint8)
    _mat(B, "B", (N, K // 2), torch.uint8)
    _mat(B_scales, "B_scales", (N, K // 16), torch.uint8)
    _scalar(A_tscale, "A_tscale")
    _scalar(B_tscale, "B_tscale")
    return [("A", A), ("A_scales", A_scales), ("A_tscale", A_tscale), ("B", B),
            ("B_scales", B_scales), ("B_tscale", B_tscale)]


def fp4q_gemm(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, out) -> None:
    ops = _gemm_operands(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K)
    _out_dtype(out)
    _mat(out, "out", (M, N), out.dtype)
    _on_device(*ops, ("out", out))
    f32 = out.dtype == torch.float32
    _check("fp4q_gemm", _lib.fp4q_gemm(
        _ptr(A), _ptr(A_scales), _ptr(A_tscale), _ptr(B), _ptr(B_scales), _ptr(B_tscale),
        M, N, K, fmt, _ptr(out), int(f32), _stream()))


def fp4q_gemm_nvfp4(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, out) -> None:
    """Native NVFP4 GEMM: UE4M3-scaled operands on the block-scaled MMA."""
    ops = _gemm_operands(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K)
    _out_dtype(out)
    _mat(out, "out", (M, N), out.dtype)
    _on_device(*ops, ("out", out))
    f32 = out.dtype == torch.float32
    _check("fp4q_gemm_nvfp4", _lib.fp4q_gemm_nvfp4(
        _ptr(A), _ptr(A_scales), _ptr(A_tscale), _ptr(B), _ptr(B_scales), _ptr(B_tscale),
        M, N, K, _ptr(out), int(f32), _stream()))


def fp4q_rebias_scales(scales, rows, nblocks, per_row, out_scales, out_factor, inout_nofit) -> None:
    """UE5M3 codes -> UE4M3 codes times a power of two per row (per_row) or for
    the tensor; ORs 1 into inout_nofit when a group does not fit."""
    if rows < 0 or nblocks < 0 or nblocks % 16:
        raise ValueError(f"rows >= 0 and nblocks a multiple of 16 required, got {rows}, {nblocks}")
    _mat(scales, "scales", (rows, nblocks), torch.uint8)
    _mat(out_scales, "out_scales", (rows, nblocks), torch.uint8)
    _scalar(out_factor, "out_factor", rows if per_row else 1)
    _scalar(inout_nofit, "inout_nofit", 1, torch.int32)
    _on_device(("scales", scales), ("out_scales", out_scales), ("out_factor", out_factor),
               ("inout_nofit", inout_nofit))
    _check("fp4q_rebias_scales", _lib.fp4q_rebias_scales(
        _ptr(scales), rows, nblocks, int(bool(per_row)), _ptr(out_scales), _ptr(out_factor),
        _ptr(inout_nofit), _stream()))


def fp4q_gemm_nvfp4_rebiased(A, A_scales4, A_factor, A_tscale, B, B_scales4, B_factor, B_tscale,
                             M, N, K, skip_if_set, out) -> None:
    """Native block-scaled GEMM on rebiased operands (per-row A factor,
    per-tensor B factor); a no-op when the device int skip_if_set is set."""
    ops = _gemm_operands(A, A_scales4, A_tscale, B, B_scales4, B_tscale, M, N, K)
    _scalar(A_factor, "A_factor", M)
    _scalar(B_factor, "B_factor")
    if skip_if_set is not None:
        _scalar(skip_if_set, "skip_if_set", 1, torch.int32)
    _out_dtype(out)
    _mat(out, "out", (M, N), out.dtype)
    _on_device(*ops, ("A_factor", A_factor), ("B_factor", B_factor), ("skip_if_set", skip_if_set),
               ("out", out))
    f32 = out.dtype == torch.float32
    _check("fp4q_gemm_nvfp4_rebiased", _lib.fp4q_gemm_nvfp4_rebiased(
        _ptr(A), _ptr(A_scales4), _ptr(A_factor), _ptr(A_tscale), _ptr(B), _ptr(B_scales4),
        _ptr(B_factor), _ptr(B_tscale), M, N, K, _ptr(skip_if_set), _ptr(out), int(f32), _stream()))


def fp4q_rebias_scales_two_windows(scales, rows, nblocks, out_hi, out_lo, out_factor_hi, out_factor_lo,
                                   inout_nofit) -> None:
    """UE5M3 codes -> UE4M3 codes in two 14-binade windows per row (high and
    low) with their power-of-two factors; ORs 1 into inout_nofit when a code
    lies below both."""
    if rows < 0 or nblocks < 0 or nblocks % 16:
        raise ValueError(f"rows >= 0 and nblocks a multiple of 16 required, got {rows}, {nblocks}")
    for t, name in ((scales, "scales"), (out_hi, "out_hi"), (out_lo, "out_lo")):
        _mat(t, name, (rows, nblocks), torch.uint8)
    _scalar(out_factor_hi, "out_factor_hi", rows)
    _scalar(out_factor_lo, "out_factor_lo", rows)
    _scalar(inout_nofit, "inout_nofit", 1, torch.int32)
    _on_device(("scales", scales), ("out_hi", out_hi), ("out_lo", out_lo), ("out_factor_hi", out_factor_hi),
               ("out_factor_lo", out_factor_lo), ("inout_nofit", inout_nofit))
    _check("fp4q_rebias_scales_two_windows", _lib.fp4q_rebias_scales_two_windows(
        _ptr(scales), rows, nblocks, _ptr(out_hi), _ptr(out_lo), _ptr(out_factor_hi), _ptr(out_factor_lo),
        _ptr(inout_nofit), _stream()))


def fp4q_gemm_nvfp4_two_windows(A, A_scales_hi, A_scales_lo, A_factor_hi, A_tscale, B, B_scales4, B_factor,
                                B_tscale, M, N, K, skip_if_set, out) -> None:
    """Native block-scaled GEMM with A's codes in two windows (two
    accumulators, the low one scaled by 2^-14) and B's per-tensor rebiased;
    a no-op when the device int skip_if_set is set."""
    ops = _gemm_operands(A, A_scales_hi, A_tscale, B, B_scales4, B_tscale, M, N, K)
    _mat(A_scales_lo, "A_scales_lo", (M, K // 16), torch.uint8)
    _scalar(A_factor_hi, "A_factor_hi", M)
    _scalar(B_factor, "B_factor")
    if skip_if_set is not None:
        _scalar(skip_if_set, "skip_if_set", 1, torch.int32)
    _out_dtype(out)
    _mat(out, "out", (M, N), out.dtype)
    _on_device(*ops, ("A_scales_lo", A_scales_lo), ("A_factor_hi", A_factor_hi), ("B_factor", B_factor),
               ("skip_if_set", skip_if_set), ("out", out))
    f32 = out.dtype == torch.float32
    _check("fp4q_gemm_nvfp4_two_windows", _lib.fp4q_gemm_nvfp4_two_windows(
        _ptr(A), _ptr(A_scales_hi), _ptr(A_scales_lo), _ptr(A_factor_hi), _ptr(A_tscale), _ptr(B),
        _ptr(B_scales4), _ptr(B_factor), _ptr(B_tscale), M, N, K, _ptr(skip_if_set), _ptr(out), int(f32),
        _stream()))


def fp4q_gemm_if(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, run_if_set, out) -> None:
    """fp4q_gemm, run only when the device int run_if_set is non-zero."""
    ops = _gemm_operands(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K)
    _scalar(run_if_set, "run_if_set", 1, torch.int32)
    _out_dtype(out)
    _mat(out, "out", (M, N), out.dtype)
    _on_device(*ops, ("run_if_set", run_if_set), ("out", out))
    f32 = out.dtype == torch.float32
    _check("fp4q_gemm_if", _lib.fp4q_gemm_if(
        _ptr(A), _ptr(A_scales), _ptr(A_tscale), _ptr(B), _ptr(B_scales), _ptr(B_tscale),
        M, N, K, fmt, _ptr(run_if_set), _ptr(out), int(f32), _stream()))


def _quantize_outputs(M, N, c_tscale, out_bf16, out_payload, out_scales, out_amax):
    if N % 32:
        raise ValueError(f"N must be a multiple of 32 for the epilogue quantisation, got {N}")
    _mat(out_payload, "out_payload", (M, N // 2), torch.uint8)
    _mat(out_scales, "out_scales", (M, N // 16), torch.uint8)
    if out_bf16 is not None:
        _mat(out_bf16, "out_bf16", (M, N), torch.bfloat16)
    _scalar(c_tscale, "c_tscale")
    if out_amax is not None:
        _scalar(out_amax, "out_amax")
    return [("c_tscale", c_tscale), ("out_bf16", out_bf16), ("out_payload", out_payload),
            ("out_scales", out_scales), ("out_amax", out_amax)]


def fp4q_gemm_nvfp4_rebiased_quantize(A, A_scales4, A_factor, A_tscale, B, B_scales4, B_factor, B_tscale,
                                      M, N, K, skip_if_set, fmt, c_tscale, out_bf16, out_payload, out_scales,
                                      out_amax=None) -> None:
    """fp4q_gemm_nvfp4_rebiased with the BF16 result quantised row-wise in its
    epilogue; out_amax is max-ed into (the caller zeroes it)."""
    ops = _gemm_operands(A, A_scales4, A_tscale, B, B_scales4, B_tscale, M, N, K)
    _scalar(A_factor, "A_factor", M)
    _scalar(B_factor, "B_factor")
    if skip_if_set is not None:
        _scalar(skip_if_set, "skip_if_set", 1, torch.int32)
    qo = _quantize_outputs(M, N, c_tscale, out_bf16, out_payload, out_scales, out_amax)
    _on_device(*ops, ("A_factor", A_factor), ("B_factor", B_factor), ("skip_if_set", skip_if_set), *qo)
    _check("fp4q_gemm_nvfp4_rebiased_quantize", _lib.fp4q_gemm_nvfp4_rebiased_quantize(
        _ptr(A), _ptr(A_scales4), _ptr(A_factor), _ptr(A_tscale), _ptr(B), _ptr(B_scales4), _ptr(B_factor),
        _ptr(B_tscale), M, N, K, _ptr(skip_if_set), fmt, _ptr(c_tscale), _ptr(out_bf16), _ptr(out_payload),
        _ptr(out_scales), _ptr(out_amax), _stream()))


def fp4q_gemm_quantize_if(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, run_if_set, c_tscale,
                          out_bf16, out_payload, out_scales, out_amax=None) -> None:
    """fp4q_gemm_quantize run only when the device int run_if_set is
    non-zero; out_amax max-ed into, not zeroed."""
    ops = _gemm_operands(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K)
    _scalar(run_if_set, "run_if_set", 1, torch.int32)
    qo = _quantize_outputs(M, N, c_tscale, out_bf16, out_payload, out_scales, out_amax)
    _on_device(*ops, ("run_if_set", run_if_set), *qo)
    _check("fp4q_gemm_quantize_if", _lib.fp4q_gemm_quantize_if(
        _ptr(A), _ptr(A_scales), _ptr(A_tscale), _ptr(B), _ptr(B_scales), _ptr(B_tscale), M, N, K, fmt,
        _ptr(run_if_set), _ptr(c_tscale), _ptr(out_bf16), _ptr(out_payload), _ptr(out_scales),
        _ptr(out_amax), _stream()))


def fp4q_gemm_quantize(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, c_tscale,
                       out_bf16, out_payload, out_scales, out_amax=None) -> None:
    ops = _gemm_operands(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K)
    if N % 32:
        raise ValueError(f"N must be a multiple of 32 for the epilogue quantisation, got {N}")
    _mat(out_payload, "out_payload", (M, N // 2), torch.uint8)
    _mat(out_scales, "out_scales", (M, N // 16), torch.uint8)
    if out_bf16 is not None:
        _mat(out_bf16, "out_bf16", (M, N), torch.bfloat16)
    _scalar(c_tscale, "c_tscale")
    if out_amax is not None:
        _scalar(out_amax, "out_amax")
    _on_device(*ops, ("c_tscale", c_tscale), ("out_bf16", out_bf16), ("out_payload", out_payload),
               ("out_scales", out_scales), ("out_amax", out_amax))
    _check("fp4q_gemm_quantize", _lib.fp4q_gemm_quantize(
        _ptr(A), _ptr(A_scales), _ptr(A_tscale), _ptr(B), _ptr(B_scales), _ptr(B_tscale),
        M, N, K, fmt, _ptr(c_tscale), _ptr(out_bf16), _ptr(out_payload), _ptr(out_scales),
        _ptr(out_amax), _stream()))


def fp4q_get_device_status(stream: torch.cuda.Stream | None = None) -> int:
    """The latched device status, read in the order of `stream` (default: the
    current stream); waits for that stream only."""
    v = ctypes.c_int(0)
    s = ctypes.c_void_p((stream or torch.cuda.current_stream()).cuda_stream)
    _check("fp4q_get_device_status", _lib.fp4q_get_device_status(ctypes.byref(v), s))
    return v.value


def fp4q_status_string(code: int) -> str:
    return _lib.fp4q_status_string(code).decode()


# ------------------------------------------------------------ allocating helpers
def amax(x: torch.Tensor) -> torch.Tensor:
    out = torch.empty(1, dtype=torch.float32, device=x.device)
    fp4q_amax(x, out)
    return out


def tensor_scale(amax_t: torch.Tensor, fmt: int = UE5M3, headroom: float = 1.0) -> torch.Tensor:
    out = torch.empty(1, dtype=torch.float32, device=amax_t.device)
    fp4q_tensor_scale(amax_t, fmt, headroom, out)
    return out


class Quantized:
    """Outputs of one quantisation (device tensors)."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def quantize(x: torch.Tensor, axis: int = AXIS_ROW, T: torch.Tensor | None = None,
             fmt: int = UE5M3, rnd: int = RNE, seed: int = 0, stats: bool = False,
             want_amax: bool = False) -> Quantized:
    """Allocates outputs and calls fp4q_quantize.  T defaults to the current
    tensor scale (fp4q_amax + fp4q_tensor_scale)."""
    R, C = x.shape
    dev = x.device
    if T is None:
        T = tensor_scale(amax(x), fmt)
    pr = sr = pc = sc = None
    if axis in (AXIS_ROW, AXIS_BOTH, AXIS_BOTH_2D):
        pr = torch.empty((R, C // 2), dtype=torch.uint8, device=dev)
        sr = torch.empty((R, C // 16), dtype=torch.uint8, device=dev)
    if axis in (AXIS_COL, AXIS_BOTH, AXIS_BOTH_2D):
        pc = torch.empty((C, R // 2), dtype=torch.uint8, device=dev)
        sc = torch.empty((C, R // 16), dtype=torch.uint8, device=dev)
    st = torch.empty((2 if axis == AXIS_BOTH else 1, 4), dtype=torch.int64, device=dev) if stats else None
    am = torch.empty(1, dtype=torch.float32, device=dev) if want_amax else None
    fp4q_quantize(x, axis, fmt, T, rnd, seed, pr, sr, pc, sc, st, am)
    return Quantized(payload_row=pr, scales_row=sr, payload_col=pc, scales_col=sc, stats=st,
                     amax=am, T=T, fmt=fmt)


def gemm_quantize(A, A_scales, A_tscale, B, B_scales, B_tscale, c_tscale, fmt: int = UE5M3,
                  want_bf16: bool = True, want_amax: bool = True) -> Quantized:
    """fp4q_gemm_quantize with allocated outputs: the row-wise quantised C
    (payload_row, scales_row), optionally bf16(C) (`C`) and max |bf16(C)|."""
    M, K = A.shape[0], A.shape[1] * 2
    N = B.shape[0]
    dev = A.device
    pr = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
    sr = torch.empty((M, N // 16), dtype=torch.uint8, device=dev)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if want_bf16 else None
    am = torch.empty(1, dtype=torch.float32, device=dev) if want_amax else None
    fp4q_gemm_quantize(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, c_tscale, C, pr, sr, am)
    return Quantized(payload_row=pr, scales_row=sr, C=C, amax=am, T=c_tscale, fmt=fmt)


def dequantize(payload, scales, T, fmt: int = UE5M3, dtype=torch.bfloat16) -> torch.Tensor:
    R, C = payload.shape[0], payload.shape[1] * 2
    out = torch.empty((R, C), dtype=dtype, device=payload.device)
    fp4q_dequantize(payload, scales, R, C, fmt, T, out)
    return out


def gemm_nvfp4(A, A_scales, A_tscale, B, B_scales, B_tscale, dtype=torch.bfloat16, out=None) -> torch.Tensor:
    """C = (T_A T_B) deq(A) deq(B)^T on the native block-scaled MMA (UE4M3 scales)."""
    M, K = A.shape[0], A.shape[1] * 2
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=dtype, device=A.device)
    fp4q_gemm_nvfp4(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, out)
    return out


def gemm(A, A_scales, A_tscale, B, B_scales, B_tscale, fmt: int = UE5M3,
         dtype=torch.bfloat16, out=None) -> torch.Tensor:
    """C = (T_A T_B) deq(A) deq(B)^T for K-major quantised A [M, K/2], B [N, K/2]."""
    M, K = A.shape[0], A.shape[1] * 2
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=dtype, device=A.device)
    fp4q_gemm(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, out)
    return out


def rebias_scales(scales, per_row: bool = True, nofit: torch.Tensor | None = None):
    """fp4q_rebias_scales with allocated outputs: (UE4M3 codes, factors,
    nofit).  A given `nofit` (int32 [1]) is OR-ed into, not cleared."""
    R, nb = scales.shape
    codes = torch.empty_like(scales)
    factor = torch.empty(R if per_row else 1, dtype=torch.float32, device=scales.device)
    if nofit is None:
        nofit = torch.zeros(1, dtype=torch.int32, device=scales.device)
    fp4q_rebias_scales(scales, R, nb, per_row, codes, factor, nofit)
    return codes, factor, nofit


def gemm_ue5m3_rebiased(A, A_scales, A_tscale, B, B_scales, B_tscale, dtype=torch.bfloat16, out=None,
                        nofit: torch.Tensor | None = None) -> torch.Tensor:
    """The UE5M3 contraction of `gemm` on the native block-scaled MMA: A's
    scales rebiased per row, B's for the tensor, then the native GEMM, and the
    emulated GEMM in its place (decided on the device) when a group does not
    fit.  `nofit` (int32 [1], zeroed here) receives the decision."""
    M, K = A.shape[0], A.shape[1] * 2
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=dtype, device=A.device)
    if nofit is None:
        nofit = torch.empty(1, dtype=torch.int32, device=A.device)
    nofit.zero_()
    a4, fa, _ = rebias_scales(A_scales, True, nofit)
    b4, fb, _ = rebias_scales(B_scales, False, nofit)
    fp4q_gemm_nvfp4_rebiased(A, a4, fa, A_tscale, B, b4, fb, B_tscale, M, N, K, nofit, out)
    fp4q_gemm_if(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, UE5M3, nofit, out)
    return out


def rebias_scales_two_windows(scales, nofit: torch.Tensor | None = None):
    """fp4q_rebias_scales_two_windows with allocated outputs: (high codes, low
    codes, high factors, low factors, nofit).  A given `nofit` (int32 [1]) is
    OR-ed into, not cleared."""
    R, nb = scales.shape
    hi, lo = torch.empty_like(scales), torch.empty_like(scales)
    fh = torch.empty(R, dtype=torch.float32, device=scales.device)
    fl = torch.empty(R, dtype=torch.float32, device=scales.device)
    if nofit is None:
        nofit = torch.zeros(1, dtype=torch.int32, device=scales.device)
    fp4q_rebias_scales_two_windows(scales, R, nb, hi, lo, fh, fl, nofit)
    return hi, lo, fh, fl, nofit


def gemm_ue5m3_two_windows(A, A_scales, A_tscale, B, B_scales, B_tscale, dtype=torch.bfloat16, out=None,
                           nofit: torch.Tensor | None = None) -> torch.Tensor:
    """gemm_ue5m3_rebiased with A's scales in two windows per row: the native
    GEMM with two accumulators, and the emulated GEMM in its place (decided on
    the device) when a code of A lies below both windows or one of B outside
    B's window.  `nofit` (int32 [1], zeroed here) receives the decision."""
    M, K = A.shape[0], A.shape[1] * 2
    N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=dtype, device=A.device)
    if nofit is None:
        nofit = torch.empty(1, dtype=torch.int32, device=A.device)
    nofit.zero_()
    ah, al, fh, _, _ = rebias_scales_two_windows(A_scales, nofit)
    b4, fb, _ = rebias_scales(B_scales, False, nofit)
    fp4q_gemm_nvfp4_two_windows(A, ah, al, fh, A_tscale, B, b4, fb, B_tscale, M, N, K, nofit, out)
    fp4q_gemm_if(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, UE5M3, nofit, out)
    return out


def gemm_quantize_ue5m3_rebiased(A, A_scales, A_tscale, B, B_scales, B_tscale, c_tscale,
                                 want_bf16: bool = True, want_amax: bool = True,
                                 nofit: torch.Tensor | None = None) -> Quantized:
    """gemm_quantize's outputs (UE5M3 operands and result scales) from
    gemm_ue5m3_rebiased's path: the native MMA through rebiased codes with
    the quantisation in its epilogue, the emulated fused GEMM in its place
    (decided on the device) when a group does not fit."""
    fmt = UE5M3
    M, K = A.shape[0], A.shape[1] * 2
    N = B.shape[0]
    dev = A.device
    pr = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
    sr = torch.empty((M, N // 16), dtype=torch.uint8, device=dev)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if want_bf16 else None
    am = torch.zeros(1, dtype=torch.float32, device=dev) if want_amax else None
    if nofit is None:
        nofit = torch.empty(1, dtype=torch.int32, device=dev)
    nofit.zero_()
    a4, fa, _ = rebias_scales(A_scales, True, nofit)
    b4, fb, _ = rebias_scales(B_scales, False, nofit)
    fp4q_gemm_nvfp4_rebiased_quantize(A, a4, fa, A_tscale, B, b4, fb, B_tscale, M, N, K, nofit, fmt, c_tscale, C,
                                      pr, sr, am)
    fp4q_gemm_quantize_if(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, UE5M3, nofit, c_tscale, C, pr,
                          sr, am)
    return Quantized(payload_row=pr, scales_row=sr, C=C, amax=am, T=c_tscale, fmt=fmt)


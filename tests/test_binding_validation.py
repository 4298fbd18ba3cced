"""The Python binding refuses, before calling the library, any tensor whose
shape does not match the sizes passed (the library trusts them: a smaller
buffer would be read or written out of bounds on the device), a wrong dtype,
a missing output, and tensors that are not on the current CUDA device.
Shapes are checked first, so these checks run here without a GPU: a call
whose shapes are all right fails only at the device check."""
import types

import pytest
import torch


@pytest.fixture(scope="module")
def fp4q():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    return fp4q


def u8(*s):
    return torch.zeros(*s, dtype=torch.uint8)


def bf(*s):
    return torch.zeros(*s, dtype=torch.bfloat16)


T = torch.ones(1)


def raises(fn, *args, match):
    with pytest.raises(ValueError, match=match):
        fn(*args)


def test_quantize_shapes(fp4q):
    q = fp4q.fp4q_quantize
    x = bf(32, 64)
    row = (u8(32, 32), u8(32, 4))
    col = (u8(64, 16), u8(64, 2))
    # right shapes: only the device check remains
    raises(q, x, fp4q.AXIS_ROW, 0, T, 0, 0, *row, None, None, match="CUDA")
    raises(q, x, fp4q.AXIS_COL, 0, T, 0, 0, None, None, *col, match="CUDA")
    raises(q, x, fp4q.AXIS_BOTH, 0, T, 0, 0, *row, *col, torch.zeros(2, 4, dtype=torch.int64),
           match="CUDA")
    # wrong or missing outputs, per axis
    raises(q, x, fp4q.AXIS_ROW, 0, T, 0, 0, u8(32, 31), row[1], None, None, match="payload_row")
    raises(q, x, fp4q.AXIS_ROW, 0, T, 0, 0, row[0], u8(32, 2), None, None, match="scales_row")
    raises(q, x, fp4q.AXIS_COL, 0, T, 0, 0, None, None, u8(32, 32), col[1], match="payload_col")
    raises(q, x, fp4q.AXIS_COL, 0, T, 0, 0, None, None, col[0], u8(16, 4), match="scales_col")
    raises(q, x, fp4q.AXIS_BOTH, 0, T, 0, 0, *row, None, None, match="payload_col is required")
    raises(q, x, fp4q.AXIS_BOTH_2D, 0, T, 0, 0, None, None, *col, match="payload_row is required")
    # stats: two structs for BOTH
    raises(q, x, fp4q.AXIS_BOTH, 0, T, 0, 0, *row, *col, torch.zeros(1, 4, dtype=torch.int64),
           match="stats")
    raises(q, x, fp4q.AXIS_ROW, 0, T, 0, 0, *row, None, None, torch.zeros(1, 4, dtype=torch.int32),
           match="stats")
    # input and sizes
    raises(q, bf(32, 40), fp4q.AXIS_ROW, 0, T, 0, 0, u8(32, 20), u8(32, 2), None, None,
           match="multiple of 16")
    raises(q, torch.zeros(32, 64), fp4q.AXIS_ROW, 0, T, 0, 0, *row, None, None, match="bfloat16")
    raises(q, bf(2, 32, 64), fp4q.AXIS_ROW, 0, T, 0, 0, *row, None, None, match="2-D")
    raises(q, x, 7, 0, T, 0, 0, *row, *col, match="axis")
    raises(q, x, fp4q.AXIS_ROW, 0, torch.ones(0), 0, 0, *row, None, None, match="tensor_scale")
    raises(q, x, fp4q.AXIS_ROW, 0, T, 0, 0, row[0], row[1].to(torch.int8), None, None, match="uint8")


def test_dequantize_shapes(fp4q):
    d = fp4q.fp4q_dequantize
    raises(d, u8(32, 32), u8(32, 4), 32, 64, 0, T, bf(32, 64), match="CUDA")
    raises(d, u8(32, 32), u8(32, 4), 32, 64, 0, T, torch.zeros(32, 64), match="CUDA")
    raises(d, u8(32, 16), u8(32, 4), 32, 64, 0, T, bf(32, 64), match="payload")
    raises(d, u8(32, 32), u8(32, 2), 32, 64, 0, T, bf(32, 64), match="scales")
    raises(d, u8(32, 32), u8(32, 4), 32, 64, 0, T, bf(64, 32), match="out")
    raises(d, u8(32, 32), u8(32, 4), 32, 64, 0, T, torch.zeros(32, 64, dtype=torch.float16), match="out")


def _gemm_ops(M, N, K):
    return (u8(M, K // 2), u8(M, K // 16), T, u8(N, K // 2), u8(N, K // 16), T)


def test_gemm_shapes(fp4q):
    g = fp4q.fp4q_gemm
    M, N, K = 48, 80, 128
    A, As, TA, B, Bs, TB = _gemm_ops(M, N, K)
    raises(g, A, As, TA, B, Bs, TB, M, N, K, 0, bf(M, N), match="CUDA")
    raises(g, A, As, TA, B, Bs, TB, M, N, K, 0, torch.zeros(M, N), match="CUDA")
    # B's K and the operand scales checked against the K passed, not A's alone
    raises(g, A, As, TA, u8(N, K // 2 - 16), Bs, TB, M, N, K, 0, bf(M, N), match="B must")
    raises(g, A, u8(M, K // 16 - 1), TA, B, Bs, TB, M, N, K, 0, bf(M, N), match="A_scales")
    raises(g, A, As, TA, B, u8(N + 1, K // 16), TB, M, N, K, 0, bf(M, N), match="B_scales")
    raises(g, A, As, TA, B, Bs, TB, M + 16, N, K, 0, bf(M + 16, N), match="A must")
    raises(g, A, As, TA, B, Bs, TB, M, N, K, 0, bf(M, N - 1), match="out")
    raises(g, A, As, torch.ones(0), B, Bs, TB, M, N, K, 0, bf(M, N), match="A_tscale")
    raises(g, A, As, TA, B, Bs, TB, -1, N, K, 0, bf(M, N), match=">= 0")


def test_gemm_quantize_shapes(fp4q):
    g = fp4q.fp4q_gemm_quantize
    M, N, K = 32, 64, 64
    ops = _gemm_ops(M, N, K)
    raises(g, *ops, M, N, K, 0, T, bf(M, N), u8(M, N // 2), u8(M, N // 16), T, match="CUDA")
    raises(g, *ops, M, N, K, 0, T, None, u8(M, N // 2), u8(M, N // 16), None, match="CUDA")
    raises(g, *ops, M, N, K, 0, T, None, u8(M, N // 4), u8(M, N // 16), None, match="out_payload")
    raises(g, *ops, M, N, K, 0, T, None, u8(M, N // 2), u8(M, N // 8), None, match="out_scales")
    raises(g, *ops, M, N, K, 0, T, bf(M, N // 2), u8(M, N // 2), u8(M, N // 16), None, match="out_bf16")
    raises(g, *ops, M, N, K, 0, None, None, u8(M, N // 2), u8(M, N // 16), None, match="c_tscale")
    ops48 = _gemm_ops(M, 48, K)
    raises(g, *ops48, M, 48, K, 0, T, None, u8(M, 24), u8(M, 3), None, match="multiple of 32")


def test_rebias_shapes(fp4q):
    r = fp4q.fp4q_rebias_scales
    f1 = torch.ones(1)
    flag = torch.zeros(1, dtype=torch.int32)
    raises(r, u8(8, 32), 8, 32, True, u8(8, 32), torch.ones(8), flag, match="CUDA")
    raises(r, u8(8, 32), 8, 32, False, u8(8, 32), f1, flag, match="CUDA")
    raises(r, u8(8, 32), 8, 32, True, u8(8, 32), f1, flag, match="out_factor")   # one per row
    raises(r, u8(8, 24), 8, 24, True, u8(8, 24), torch.ones(8), flag, match="multiple of 16")
    raises(r, u8(8, 32), 8, 32, True, u8(8, 16), torch.ones(8), flag, match="out_scales")
    raises(r, u8(8, 32), 8, 32, True, u8(8, 32), torch.ones(8), torch.zeros(1), match="inout_nofit")


def test_rebiased_gemm_shapes(fp4q):
    M, N, K = 32, 64, 256
    A, As, TA, B, Bs, TB = _gemm_ops(M, N, K)
    flag = torch.zeros(1, dtype=torch.int32)
    g = fp4q.fp4q_gemm_nvfp4_rebiased
    raises(g, A, As, torch.ones(M), TA, B, Bs, torch.ones(1), TB, M, N, K, flag, bf(M, N), match="CUDA")
    raises(g, A, As, torch.ones(M), TA, B, Bs, torch.ones(1), TB, M, N, K, None, bf(M, N), match="CUDA")
    raises(g, A, As, torch.ones(M - 1), TA, B, Bs, torch.ones(1), TB, M, N, K, flag, bf(M, N),
           match="A_factor")
    raises(g, A, As, torch.ones(M), TA, B, Bs, None, TB, M, N, K, flag, bf(M, N), match="B_factor")
    raises(g, A, As, torch.ones(M), TA, B, Bs, torch.ones(1), TB, M, N, K, torch.zeros(1), bf(M, N),
           match="skip_if_set")
    c = fp4q.fp4q_gemm_if
    raises(c, A, As, TA, B, Bs, TB, M, N, K, 0, flag, bf(M, N), match="CUDA")
    raises(c, A, As, TA, B, Bs, TB, M, N, K, 0, None, bf(M, N), match="run_if_set")
    raises(c, A, As, TA, B, Bs, TB, M, N, K, 0, flag, bf(M, N + 16), match="out")


def test_two_window_shapes(fp4q):
    r = fp4q.fp4q_rebias_scales_two_windows
    f8 = torch.ones(8)
    flag = torch.zeros(1, dtype=torch.int32)
    raises(r, u8(8, 32), 8, 32, u8(8, 32), u8(8, 32), f8, f8, flag, match="CUDA")
    raises(r, u8(8, 24), 8, 24, u8(8, 24), u8(8, 24), f8, f8, flag, match="multiple of 16")
    raises(r, u8(8, 32), 8, 32, u8(8, 32), u8(8, 16), f8, f8, flag, match="out_lo")
    raises(r, u8(8, 32), 8, 32, u8(8, 32), u8(8, 32), torch.ones(1), f8, flag, match="out_factor_hi")
    raises(r, u8(8, 32), 8, 32, u8(8, 32), u8(8, 32), f8, f8, torch.zeros(1), match="inout_nofit")
    M, N, K = 32, 64, 256
    A, As, TA, B, Bs, TB = _gemm_ops(M, N, K)
    g = fp4q.fp4q_gemm_nvfp4_two_windows
    fa, fb = torch.ones(M), torch.ones(1)
    raises(g, A, As, u8(M, K // 16), fa, TA, B, Bs, fb, TB, M, N, K, flag, bf(M, N), match="CUDA")
    raises(g, A, As, u8(M, K // 32), fa, TA, B, Bs, fb, TB, M, N, K, flag, bf(M, N), match="A_scales_lo")
    raises(g, A, As, u8(M, K // 16), torch.ones(1), TA, B, Bs, fb, TB, M, N, K, flag, bf(M, N),
           match="A_factor_hi")
    raises(g, A, As, u8(M, K // 16), fa, TA, B, Bs, None, TB, M, N, K, flag, bf(M, N), match="B_factor")


def test_rebiased_fused_gemm_shapes(fp4q):
    M, N, K = 32, 64, 256
    A, As, TA, B, Bs, TB = _gemm_ops(M, N, K)
    flag = torch.zeros(1, dtype=torch.int32)
    fa, fb = torch.ones(M), torch.ones(1)
    g = fp4q.fp4q_gemm_nvfp4_rebiased_quantize
    raises(g, A, As, fa, TA, B, Bs, fb, TB, M, N, K, flag, 0, T, bf(M, N), u8(M, N // 2), u8(M, N // 16), T,
           match="CUDA")
    raises(g, A, As, fa, TA, B, Bs, fb, TB, M, N, K, flag, 0, T, None, u8(M, N // 4), u8(M, N // 16), None,
           match="out_payload")
    raises(g, A, As, torch.ones(1), TA, B, Bs, fb, TB, M, N, K, flag, 0, T, None, u8(M, N // 2),
           u8(M, N // 16), None, match="A_factor")
    ops48 = _gemm_ops(M, 48, K)
    raises(g, ops48[0], ops48[1], fa, TA, ops48[3], ops48[4], fb, TB, M, 48, K, flag, 0, T, None, u8(M, 24),
           u8(M, 3), None, match="multiple of 32")
    c = fp4q.fp4q_gemm_quantize_if
    raises(c, A, As, TA, B, Bs, TB, M, N, K, 0, flag, T, None, u8(M, N // 2), u8(M, N // 16), None, match="CUDA")
    raises(c, A, As, TA, B, Bs, TB, M, N, K, 0, None, T, None, u8(M, N // 2), u8(M, N // 16), None,
           match="run_if_set")
    raises(c, A, As, TA, B, Bs, TB, M, N, K, 0, flag, T, None, u8(M, N // 2), u8(M, N // 8), None,
           match="out_scales")


def test_scalar_entry_points(fp4q):
    raises(fp4q.fp4q_amax, bf(16), torch.ones(0), match="out_amax")
    raises(fp4q.fp4q_amax, torch.zeros(16), torch.ones(1), match="bfloat16")
    raises(fp4q.fp4q_amax, bf(16), torch.ones(1), match="CUDA")
    raises(fp4q.fp4q_tensor_scale, torch.ones(1, dtype=torch.float64), 0, 1.0, T, match="amax")
    raises(fp4q.fp4q_tensor_scale, T, 0, 1.0, torch.ones(1), match="CUDA")


def test_tensors_must_be_on_the_current_device(fp4q, monkeypatch):
    # stand-ins for CUDA tensors on device 1 while device 0 is current
    monkeypatch.setattr(torch.cuda, "is_available", lambda: True)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)

    def fake(index, contiguous=True):
        return types.SimpleNamespace(is_cuda=True, device=torch.device("cuda", index),
                                     is_contiguous=lambda: contiguous)
    fp4q._on_device(("a", fake(0)), ("b", None))
    with pytest.raises(ValueError, match="current device"):
        fp4q._on_device(("a", fake(0)), ("b", fake(1)))
    with pytest.raises(ValueError, match="contiguous"):
        fp4q._on_device(("a", fake(0, contiguous=False)))

"""GPU parity of the emulated UE5M3 block-scaled GEMM (tcgen05) against the
oracle's binary64 contraction of identical dequantised operands.

Tolerance (stated in parity_util): normwise max |C - R| / max |R| <= 1e-3 on
the FP32-output mode; the BF16 output must lie within one BF16 ulp of R plus
1e-3 max |R|.  The operands are the GPU's own quantised bytes, which the
quantiser tests prove equal to the oracle's.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (FP4 matrix multiplications of fprop, dgrad and wgrad on E2M1 +
UE5M3 block-16 operands, UE5M3 emulated in software)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import (GEMM_TOL, check_gemm_bf16, check_gemm_elementwise, gemm_abs_reference,
                         extreme_rows, gemm_error, sampled_check, stripes, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    yield fp4q
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def quantised(bits, lib, axis=0, rnd=0, seed=0, fmt=0):
    x = to_dev(bits)
    q = lib.quantize(x, axis, None, fmt, rnd, seed)
    if axis == 1:
        return q.payload_col, q.scales_col, q.T
    return q.payload_row, q.scales_row, q.T


def run_both(lib, A, B, fmt=0):
    C32 = lib.gemm(*A, *B, fmt=fmt, dtype=torch.float32)
    C16 = lib.gemm(*A, *B, fmt=fmt, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    return C32.cpu().numpy(), C16.float().cpu().numpy()


def _np_ops(A, B):
    pa, sa, ta = (t.cpu().numpy() if hasattr(t, "cpu") else t for t in A)
    pb, sb, tb = (t.cpu().numpy() if hasattr(t, "cpu") else t for t in B)
    return pa, sa, float(ta[0]), pb, sb, float(tb[0])


def full_reference(A, B, fmt=0):
    """R (binary64 contraction) and S (the same over magnitudes)."""
    pa, sa, ta, pb, sb, tb = _np_ops(A, B)
    R = oracle.gemm(pa, sa, ta, pb, sb, tb, fmt)
    return R, gemm_abs_reference(pa, sa, pb, sb, ta * tb, fmt)


def assert_close(C32, C16, ref, K):
    R, S = ref
    err = gemm_error(C32, R)
    assert err <= GEMM_TOL, err
    check_gemm_elementwise(C32, R, S, K)
    check_gemm_bf16(C16, R)
    return err


def rand_bits(shape, seed, spread=0.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    if spread:
        x *= (10.0 ** rng.uniform(-spread, spread, (1, shape[1]))).astype(np.float32)
    return workloads.f32_to_bf16_bits(x)


def test_tiny_config(lib):
    a, b = workloads.tiny_operands(seed=0)
    A, B = quantised(a, lib), quantised(b, lib)
    C32, C16 = run_both(lib, A, B)
    assert_close(C32, C16, full_reference(A, B), 256)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (128, 256, 128), (256, 512, 256), (100, 200, 64),
                                   (16, 16, 64), (300, 700, 320), (129, 257, 192), (640, 384, 1024)])
def test_shapes_and_ragged_tiles(M, N, K, lib):
    a = rand_bits((M + (-M) % 16, K), M * 7 + K, spread=2.0)[:M]
    b = rand_bits((N + (-N) % 16, K), N * 13 + K, spread=2.0)[:N]
    a = np.ascontiguousarray(np.pad(a, ((0, (-M) % 16), (0, 0))))
    b = np.ascontiguousarray(np.pad(b, ((0, (-N) % 16), (0, 0))))
    A, B = quantised(a, lib), quantised(b, lib)
    A = (A[0][:M].contiguous(), A[1][:M].contiguous(), A[2])
    B = (B[0][:N].contiguous(), B[1][:N].contiguous(), B[2])
    C32, C16 = run_both(lib, A, B)
    assert C32.shape == (M, N)
    assert_close(C32, C16, full_reference(A, B), K)


def test_two_waves_with_ragged_edges(lib):
    """More 256 x 512 tiles (9 x 10 = 90) than clusters of two CTAs fit on
    the GPU at once, so a second wave of clusters starts on SMs the first
    leaves, with ragged last tiles in M and N (the last tile's second N half
    partly past N) and K a multiple of 256 (scale codes by TMA).  Every element
    against the oracle's exact e*s operands contracted in binary64."""
    M, N, K = 2200, 5000, 512
    a = rand_bits((M + (-M) % 16, K), 11, spread=2.0)[:M]
    b = rand_bits((N + (-N) % 16, K), 12, spread=2.0)[:N]
    a = np.ascontiguousarray(np.pad(a, ((0, (-M) % 16), (0, 0))))
    b = np.ascontiguousarray(np.pad(b, ((0, (-N) % 16), (0, 0))))
    A, B = quantised(a, lib), quantised(b, lib)
    A = (A[0][:M].contiguous(), A[1][:M].contiguous(), A[2])
    B = (B[0][:N].contiguous(), B[1][:N].contiguous(), B[2])
    C32, C16 = run_both(lib, A, B)
    pa, sa, ta, pb, sb, tb = _np_ops(A, B)
    ea, eb = oracle.deq_es(pa, sa), oracle.deq_es(pb, sb)
    R = ta * tb * (ea @ eb.T)
    S = ta * tb * (np.abs(ea) @ np.abs(eb).T)
    assert_close(C32, C16, (R, S), K)


@pytest.mark.parametrize("fmt", [0, 1])
def test_wide_dynamic_range_and_formats(lib, fmt):
    # per-row magnitudes over 1e-8 .. 1e2 (the gradient distribution), SR on A
    a = workloads.gradients(256, 512, 5)
    b = rand_bits((384, 512), 6, spread=3.0)
    A, B = quantised(a, lib, rnd=1, seed=7, fmt=fmt), quantised(b, lib, fmt=fmt)
    C32, C16 = run_both(lib, A, B, fmt)
    assert_close(C32, C16, full_reference(A, B, fmt), 512)


def test_zero_and_k0(lib):
    z = np.zeros((128, 128), np.uint16)
    A = quantised(z, lib)
    C32, C16 = run_both(lib, A, A)
    assert (C32 == 0).all() and (C16 == 0).all()
    out = torch.full((16, 16), 7.0, device="cuda")
    e = torch.empty((16, 0), dtype=torch.uint8, device="cuda")
    one = torch.ones(1, device="cuda")
    lib.fp4q_gemm(e, e, one, e, e, one, 16, 16, 0, 0, out)
    torch.cuda.synchronize()
    assert (out == 0).all()


def test_full_fprop(lib):
    """Y = X W^T at 8192 x 16384 x 4096 (8B-class fprop), sampled stripes."""
    X, W = workloads.fprop_operands()
    A, B = quantised(X, lib), quantised(W, lib)
    C = lib.gemm(*A, *B, dtype=torch.float32)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    err = sampled_check(A, B, C, stripes(8192, rng, 128), stripes(16384, rng, 256))
    assert err <= GEMM_TOL, err


def test_full_dgrad_wgrad(lib):
    """dX = dY W (8192 x 4096 x 16384) and dW = dY^T X (16384 x 4096 x 8192)
    with SR gradients (seed 7), sampled stripes."""
    X, W = workloads.fprop_operands()
    dY = workloads.backward_gradient()
    d = to_dev(dY)
    qd = lib.quantize(d, 2, None, 0, 1, 7)
    Wc = quantised(W, lib, axis=1)
    Xc = quantised(X, lib, axis=1)
    rng = np.random.default_rng(1)
    dX = lib.gemm(qd.payload_row, qd.scales_row, qd.T, *Wc, dtype=torch.float32)
    torch.cuda.synchronize()
    rows = np.unique(np.r_[stripes(8192, rng, 128), extreme_rows(dY)])   # and the extreme-magnitude tokens
    err = sampled_check((qd.payload_row, qd.scales_row, qd.T), Wc, dX, rows, stripes(4096, rng, 256))
    assert err <= GEMM_TOL, err
    del dX
    dW = lib.gemm(qd.payload_col, qd.scales_col, qd.T, *Xc, dtype=torch.float32)
    torch.cuda.synchronize()
    err = sampled_check((qd.payload_col, qd.scales_col, qd.T), Xc, dW,
                         stripes(16384, rng, 128), stripes(4096, rng, 256))
    assert err <= GEMM_TOL, err


@pytest.mark.parametrize("name", ["qkv", "out", "down"])
def test_linear_block_shapes(lib, name):
    """8B-class block linears (qkv 4096->6144, out 4096->4096, down 16384->4096; up is
    the full-size case above), 8192 tokens:
    fprop, dgrad and wgrad through quantise + block-scaled GEMM with SR on
    dY, sampled stripes against the oracle."""
    X, W, dY = workloads.linear_block(name)
    fin, fout = workloads.LINEARS[name]
    Xr, Wr = quantised(X, lib), quantised(W, lib)
    Xc, Wc = quantised(X, lib, axis=1), quantised(W, lib, axis=1)
    qd = lib.quantize(to_dev(dY), 2, None, 0, 1, 7)
    Dr = (qd.payload_row, qd.scales_row, qd.T)
    Dc = (qd.payload_col, qd.scales_col, qd.T)
    rng = np.random.default_rng(len(name))
    for A, B, M, N in ((Xr, Wr, 8192, fout), (Dr, Wc, 8192, fin), (Dc, Xc, fout, fin)):
        C = lib.gemm(*A, *B, dtype=torch.float32)
        torch.cuda.synchronize()
        assert C.shape == (M, N)
        err = sampled_check(A, B, C, stripes(M, rng, 128), stripes(N, rng, 256))
        assert err <= GEMM_TOL, (name, M, N, err)
        del C

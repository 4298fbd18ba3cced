"""GPU parity of the GEMM with its result quantised in the epilogue (the
fusion the UE5M3 page lists among related work: quantisation in the
producing GEMM, "format-aware fusion"): the payload and scales must equal,
byte for byte, the oracle's row-wise RNE quantisation of the BF16 result the
GPU wrote; the fused amax must equal max |bf16(C)|; the result itself meets
the GEMM tolerance against the oracle's binary64 contraction.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (E2M1 + UE5M3 block-16 inputs of every FP4 linear) and Related
papers (quantisation fused into the producing GEMM)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import check_gemm_bf16, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    yield fp4q
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def rand_bits(shape, seed, spread=2.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    if spread:
        x *= (10.0 ** rng.uniform(-spread, spread, (1, shape[1]))).astype(np.float32)
    return workloads.f32_to_bf16_bits(x)


def operands(lib, M, N, K, seed, fmt=0):
    a = rand_bits((M + (-M) % 16, K), seed)
    b = rand_bits((N + (-N) % 16, K), seed + 1)
    qa, qb = lib.quantize(to_dev(a), fmt=fmt), lib.quantize(to_dev(b), fmt=fmt)
    A = (qa.payload_row[:M].contiguous(), qa.scales_row[:M].contiguous(), qa.T)
    B = (qb.payload_row[:N].contiguous(), qb.scales_row[:N].contiguous(), qb.T)
    return A, B


def check(lib, A, B, T=None, fmt=0, sample=None):
    M, N = A[0].shape[0], B[0].shape[0]
    if T is None:   # the current tensor scale of C, from a plain GEMM of the same operands
        C0 = lib.gemm(*A, *B, fmt=fmt)
        T = lib.tensor_scale(lib.amax(C0), fmt)
    q = lib.gemm_quantize(*A, *B, T, fmt)
    q2 = lib.gemm_quantize(*A, *B, T, fmt, want_bf16=False, want_amax=False)
    torch.cuda.synchronize()
    cb = q.C.view(torch.int16).cpu().numpy().view(np.uint16)
    # row-wise blocks are independent: pad the rows to a multiple of 16 for the oracle
    cpad = np.pad(cb, ((0, (-M) % 16), (0, 0)))
    p, s, _ = oracle.quantize(cpad, oracle.ROW, float(T.item()), fmt)
    p, s = p[:M], s[:M]
    gp, gs = q.payload_row.cpu().numpy(), q.scales_row.cpu().numpy()
    if not np.array_equal(gp, p):
        bad = np.argwhere(gp != p)
        raise AssertionError(f"payload: {len(bad)} bytes differ, first {bad[:4].tolist()}")
    assert np.array_equal(gs, s)
    assert torch.equal(q2.payload_row, q.payload_row) and torch.equal(q2.scales_row, q.scales_row)
    assert float(q.amax.item()) == oracle.amax(cb)[0]
    if sample is None:
        pa, sa = A[0].cpu().numpy(), A[1].cpu().numpy()
        pb, sb = B[0].cpu().numpy(), B[1].cpu().numpy()
        R = oracle.gemm(pa, sa, float(A[2].item()), pb, sb, float(B[2].item()), fmt)
        C = workloads.bf16_bits_to_f32(cb).astype(np.float64)
        check_gemm_bf16(C, R)
    return q


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 704, 320), (129, 288, 192), (640, 384, 1024),
                                   (16, 32, 256)])
def test_shapes(lib, M, N, K):
    A, B = operands(lib, M, N, K, M + N + K)
    check(lib, A, B)


@pytest.mark.parametrize("fmt", [0, 1])
def test_stale_scales_and_formats(lib, fmt):
    A, B = operands(lib, 256, 512, 256, 3, fmt)
    for T in (1e-4, 1.0, 1e3):
        check(lib, A, B, T=torch.tensor([T], dtype=torch.float32, device="cuda"), fmt=fmt)


def test_k0_and_empty(lib):
    M, N = 64, 96
    e = torch.empty((M, 0), dtype=torch.uint8, device="cuda")
    f = torch.empty((N, 0), dtype=torch.uint8, device="cuda")
    one = torch.ones(1, device="cuda")
    q = lib.gemm_quantize(e, e, one, f, f, one, one)
    torch.cuda.synchronize()
    assert (q.payload_row == 0).all() and (q.scales_row == 0).all() and float(q.amax.item()) == 0.0
    assert (q.C.float() == 0).all()


def test_full_fprop(lib):
    """Y = X W^T at 8192 x 16384 x 4096, its row-wise quantisation for the
    next layer in the epilogue (BF16 result checked by the other GEMM tests)."""
    X, W = workloads.fprop_operands()
    qx, qw = lib.quantize(to_dev(X)), lib.quantize(to_dev(W))
    A = (qx.payload_row, qx.scales_row, qx.T)
    B = (qw.payload_row, qw.scales_row, qw.T)
    check(lib, A, B, sample=True)

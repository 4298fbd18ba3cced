"""GPU parity of the native NVFP4 GEMM (fp4q_gemm_nvfp4: E2M1 operands with
UE4M3 block-16 scales on the tensor cores' block-scaled MMA) against the
oracle's binary64 contraction of the same dequantised operands, with the
tolerance of every GEMM check (normwise 1e-3 on FP32 output, the elementwise
bound, the BF16 bound).

The cases are ordered so that a failure says where to look: uniform scales
(the scales' placement cannot matter), scales that vary only by row (the
row -> scale mapping of A and of B), only by K block (the order of the four
block scales of an MMA), then operands from the UE4M3 quantiser at ragged
and 8B-class shapes.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (the native NVFP4 execution ablation; UE4M3 block scales are what
the tensor cores take natively)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import (GEMM_TOL, check_gemm_bf16, check_gemm_elementwise, gemm_abs_reference,
                         gemm_error, to_dev)

pytestmark = pytest.mark.gpu
UE4M3 = oracle.UE4M3


@pytest.fixture(scope="module", autouse=True)
def lib():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    yield fp4q
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(lib, pa, sa, ta, pb, sb, tb):
    A = (_dev(pa), _dev(sa), torch.tensor([ta], dtype=torch.float32, device="cuda"))
    B = (_dev(pb), _dev(sb), torch.tensor([tb], dtype=torch.float32, device="cuda"))
    C32 = lib.gemm_nvfp4(*A, *B, dtype=torch.float32)
    C16 = lib.gemm_nvfp4(*A, *B, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    return C32.cpu().numpy().astype(np.float64), C16.float().cpu().numpy().astype(np.float64)


def _check(lib, pa, sa, ta, pb, sb, tb):
    C32, C16 = _run(lib, pa, sa, ta, pb, sb, tb)
    R = oracle.gemm(pa, sa, ta, pb, sb, tb, UE4M3)
    S = gemm_abs_reference(pa, sa, pb, sb, ta * tb, UE4M3)
    err = gemm_error(C32, R)
    if err > GEMM_TOL:
        bad_rows = np.nonzero(np.abs(C32 - R).max(1) > GEMM_TOL * np.abs(R).max())[0]
        bad_cols = np.nonzero(np.abs(C32 - R).max(0) > GEMM_TOL * np.abs(R).max())[0]
        raise AssertionError(f"normwise error {err:.3e}; rows off {bad_rows[:16].tolist()} "
                             f"({bad_rows.size}), cols off {bad_cols[:16].tolist()} ({bad_cols.size})")
    check_gemm_elementwise(C32, R, S, pa.shape[1] * 2)
    check_gemm_bf16(C16, R)
    return err


def _payload(rng, rows, K):
    return rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)


def test_uniform_scales(lib):
    rng = np.random.default_rng(1)
    M, N, K = 128, 256, 256
    pa, pb = _payload(rng, M, K), _payload(rng, N, K)
    one = 0x38   # UE4M3 1.0
    _check(lib, pa, np.full((M, K // 16), one, np.uint8), 1.0, pb, np.full((N, K // 16), one, np.uint8), 1.0)


def test_scales_by_row(lib):
    rng = np.random.default_rng(2)
    M, N, K = 128, 256, 256
    pa, pb = _payload(rng, M, K), _payload(rng, N, K)
    sa = np.repeat(rng.integers(0x20, 0x50, (M, 1), dtype=np.uint8), K // 16, 1)
    sb = np.repeat(rng.integers(0x20, 0x50, (N, 1), dtype=np.uint8), K // 16, 1)
    _check(lib, pa, sa, 0.5, pb, sb, 2.0)


def test_scales_by_k_block(lib):
    rng = np.random.default_rng(3)
    M, N, K = 128, 256, 512
    pa, pb = _payload(rng, M, K), _payload(rng, N, K)
    sa = np.repeat(rng.integers(0x20, 0x50, (1, K // 16), dtype=np.uint8), M, 0)
    sb = np.repeat(rng.integers(0x20, 0x50, (1, K // 16), dtype=np.uint8), N, 0)
    _check(lib, pa, sa, 1.0, pb, sb, 1.0)


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 1024), (200, 300, 512), (16, 48, 256),
                                   (384, 776, 768)])
def test_random_scales_and_ragged_tiles(lib, M, N, K):
    rng = np.random.default_rng(M + N + K)
    pa, pb = _payload(rng, M, K), _payload(rng, N, K)
    sa = rng.integers(0, 0x7F, (M, K // 16), dtype=np.uint8)     # every finite UE4M3 code
    sb = rng.integers(0, 0x7F, (N, K // 16), dtype=np.uint8)
    _check(lib, pa, sa, 3e-3, pb, sb, 7.0)


def test_quantised_operands_match_the_emulated_gemm(lib):
    """Operands from the UE4M3 quantiser: the native GEMM and the emulated
    one (fp4q_gemm with UE4M3 scales) both meet the bound against the
    oracle."""
    rng = np.random.default_rng(4)
    M, N, K = 512, 768, 1024
    a = workloads.f32_to_bf16_bits((rng.standard_normal((M, K)) * np.exp(rng.standard_normal(K))).astype(np.float32))
    b = workloads.f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    qa = lib.quantize(to_dev(a), fmt=lib.UE4M3)
    qb = lib.quantize(to_dev(b), fmt=lib.UE4M3)
    A = (qa.payload_row, qa.scales_row, qa.T)
    B = (qb.payload_row, qb.scales_row, qb.T)
    Cn = lib.gemm_nvfp4(*A, *B, dtype=torch.float32)
    Ce = lib.gemm(*A, *B, fmt=lib.UE4M3, dtype=torch.float32)
    torch.cuda.synchronize()
    pa, sa, pb, sb = (t.cpu().numpy() for t in (A[0], A[1], B[0], B[1]))
    ta, tb = float(A[2].item()), float(B[2].item())
    R = oracle.gemm(pa, sa, ta, pb, sb, tb, UE4M3)
    S = gemm_abs_reference(pa, sa, pb, sb, ta * tb, UE4M3)
    for C in (Cn, Ce):
        C = C.cpu().numpy().astype(np.float64)
        assert gemm_error(C, R) <= GEMM_TOL
        check_gemm_elementwise(C, R, S, K)


def test_k0_and_empty(lib):
    out = torch.full((16, 16), 7.0, device="cuda")
    e = torch.empty((16, 0), dtype=torch.uint8, device="cuda")
    one = torch.ones(1, device="cuda")
    lib.fp4q_gemm_nvfp4(e, e, one, e, e, one, 16, 16, 0, out)
    torch.cuda.synchronize()
    assert (out == 0).all()
    with pytest.raises(lib.Fp4qError):
        z = torch.zeros((16, 64), dtype=torch.uint8, device="cuda")
        zs = torch.zeros((16, 8), dtype=torch.uint8, device="cuda")
        lib.fp4q_gemm_nvfp4(z, zs, one, z, zs, one, 16, 16, 128, out)    # K % 256


def test_linear_block_fprop_shape(lib):
    """The 8B-class out projection (8192 x 4096 x 4096) on UE4M3-quantised
    activations and weights, sampled stripes against the oracle."""
    X, W, _ = workloads.linear_block("out")
    qx = lib.quantize(to_dev(X), fmt=lib.UE4M3)
    qw = lib.quantize(to_dev(W), fmt=lib.UE4M3)
    C = lib.gemm_nvfp4(qx.payload_row, qx.scales_row, qx.T, qw.payload_row, qw.scales_row, qw.T,
                       dtype=torch.float32)
    torch.cuda.synchronize()
    pa, sa, pb, sb = (t.cpu().numpy() for t in (qx.payload_row, qx.scales_row, qw.payload_row, qw.scales_row))
    alpha = float(qx.T.item()) * float(qw.T.item())
    rng = np.random.default_rng(5)
    rows = np.unique(np.r_[0:128, 8192 - 128:8192, rng.choice(8192, 64, replace=False)])
    cols = np.unique(np.r_[0:256, 4096 - 256:4096, rng.choice(4096, 64, replace=False)])
    ea, eb = oracle.deq_es(pa[rows], sa[rows], UE4M3), oracle.deq_es(pb, sb, UE4M3)
    Rr, Sr = alpha * (ea @ eb.T), alpha * (np.abs(ea) @ np.abs(eb).T)
    ea, eb = oracle.deq_es(pa, sa, UE4M3), oracle.deq_es(pb[cols], sb[cols], UE4M3)
    Rc, Sc = alpha * (ea @ eb.T), alpha * (np.abs(ea) @ np.abs(eb).T)
    cr = C[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    cc = C[:, torch.from_numpy(cols).cuda()].cpu().numpy().astype(np.float64)
    scale = max(np.abs(Rr).max(), np.abs(Rc).max())
    assert np.abs(cr - Rr).max() / scale <= GEMM_TOL
    assert np.abs(cc - Rc).max() / scale <= GEMM_TOL
    check_gemm_elementwise(cr, Rr, Sr, 4096)
    check_gemm_elementwise(cc, Rc, Sc, 4096)


def test_persistent_tiles_with_ragged_edges(lib):
    """More 256 x 256 tiles (9 x 11 = 99) than there are resident clusters of
    two CTAs, so clusters walk several tiles and reuse TMEM and the stage ring
    across them; ragged last tiles in both M and N.  Every element against
    the oracle's exact e*s operands contracted in binary64, in FP32 and BF16."""
    rng = np.random.default_rng(6)
    M, N, K = 2200, 2600, 512
    pa, pb = _payload(rng, M, K), _payload(rng, N, K)
    sa = rng.integers(0x20, 0x60, (M, K // 16), dtype=np.uint8)
    sb = rng.integers(0x20, 0x60, (N, K // 16), dtype=np.uint8)
    ta, tb = 0.75, 1.5
    C32, C16 = _run(lib, pa, sa, ta, pb, sb, tb)
    ea, eb = oracle.deq_es(pa, sa, UE4M3), oracle.deq_es(pb, sb, UE4M3)
    alpha = ta * tb
    R = alpha * (ea @ eb.T)
    S = alpha * (np.abs(ea) @ np.abs(eb).T)
    assert gemm_error(C32, R) <= GEMM_TOL
    check_gemm_elementwise(C32, R, S, K)
    check_gemm_bf16(C16, R)


@pytest.mark.parametrize("M,N", [(200, 300), (200, 304), (96, 776)])
def test_result_written_at_every_alignment(lib, M, N):
    """The result's store paths (TMA stores of staged boxes when a tensor map
    describes the BF16 result, 256-bit stores where a row segment is 32-byte
    aligned, else 128-bit or scalar ones) write the same bits wherever the
    output starts: a result 16 bytes into a larger buffer (so that the
    32-byte alignment of its rows varies) equals the one in a fresh tensor,
    for the one-window and the two-window shapes, BF16 and binary32, ragged N
    included."""
    rng = np.random.default_rng(M * N)
    K = 512
    pa, pb = _payload(rng, M, K), _payload(rng, N, K)
    sa = rng.integers(0x30, 0x48, (M, K // 16), dtype=np.uint8)
    sb = rng.integers(0x30, 0x48, (N, K // 16), dtype=np.uint8)
    A = (_dev(pa), _dev(sa), torch.ones(1, device="cuda"))
    B = (_dev(pb), _dev(sb), torch.ones(1, device="cuda"))
    lo = torch.zeros((M, K // 16), dtype=torch.uint8, device="cuda")
    lo[:, ::7] = 0x70                                   # low-window codes ~2^-7 of the high ones: visible in BF16
    fa, fb = torch.ones(M, device="cuda"), torch.ones(1, device="cuda")
    for dtype, esz in ((torch.bfloat16, 2), (torch.float32, 4)):
        ref_n = torch.empty((M, N), dtype=dtype, device="cuda")
        ref_t = torch.empty((M, N), dtype=dtype, device="cuda")
        buf = torch.full((M * N + 64 // esz,), 7, dtype=dtype, device="cuda")
        off = 16 // esz
        out = buf[off:off + M * N].view(M, N)
        assert out.data_ptr() % 32 == 16
        lib.fp4q_gemm_nvfp4(*A, *B, M, N, K, ref_n)
        lib.fp4q_gemm_nvfp4(*A, *B, M, N, K, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_n), dtype
        lib.fp4q_gemm_nvfp4_two_windows(A[0], A[1], lo, fa, A[2], B[0], B[1], fb, B[2], M, N, K, None, ref_t)
        lib.fp4q_gemm_nvfp4_two_windows(A[0], A[1], lo, fa, A[2], B[0], B[1], fb, B[2], M, N, K, None, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_t), dtype
        assert (buf[:off] == 7).all() and (buf[off + M * N:] == 7).all()   # nothing outside the result
        assert not torch.equal(ref_t, ref_n)                                # the low window contributes

"""GPU parity of the UE5M3 GEMM through rebiased codes on the native MMA with
its result quantised in the epilogue (fp4q_gemm_nvfp4_rebiased_quantize,
and fp4q_gemm_quantize_if in its place when a group does not fit): the
payload and scales equal, byte for byte, the oracle's row-wise RNE
quantisation of the BF16 result the GPU wrote; the fused amax equals
max |bf16(C)|; the BF16 result meets the GEMM bound against the oracle's
binary64 UE5M3 contraction of the original operands; the fallback equals
the emulated fused GEMM bit for bit.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (UE5M3 emulated because the tensor cores take only E4M3/E8M0 block
scales; E2M1 + UE5M3 inputs of every FP4 linear) and Related papers
(quantisation fused into the producing GEMM)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import check_gemm_bf16, np_u8, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    yield fp4q
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def _operands(lib, a_bits, b_bits):
    qa, qb = lib.quantize(to_dev(a_bits)), lib.quantize(to_dev(b_bits))
    return (qa.payload_row, qa.scales_row, qa.T), (qb.payload_row, qb.scales_row, qb.T)


def _fits(A, B):
    return oracle.rebias_scales(np_u8(A[1]), True)[2] and oracle.rebias_scales(np_u8(B[1]), False)[2]


def _check(lib, A, B, T=None, full=True):
    M, N = A[0].shape[0], B[0].shape[0]
    if T is None:
        T = lib.tensor_scale(lib.amax(lib.gemm(*A, *B)))
    flag = torch.empty(1, dtype=torch.int32, device="cuda")
    q = lib.gemm_quantize_ue5m3_rebiased(*A, *B, T, nofit=flag)
    q2 = lib.gemm_quantize_ue5m3_rebiased(*A, *B, T, want_bf16=False, want_amax=False)
    torch.cuda.synchronize()
    assert int(flag.item()) == int(not _fits(A, B))
    cb = q.C.view(torch.int16).cpu().numpy().view(np.uint16)
    p, s, _ = oracle.quantize(cb, oracle.ROW, float(T.item()))
    gp, gs = np_u8(q.payload_row), np_u8(q.scales_row)
    if not np.array_equal(gp, p):
        bad = np.argwhere(gp != p)
        raise AssertionError(f"payload: {len(bad)} bytes differ, first {bad[:4].tolist()}")
    assert np.array_equal(gs, s)
    assert torch.equal(q2.payload_row, q.payload_row) and torch.equal(q2.scales_row, q.scales_row)
    assert float(q.amax.item()) == oracle.amax(cb)[0]
    if full:
        pa, sa, pb, sb = (np_u8(t) for t in (A[0], A[1], B[0], B[1]))
        R = oracle.gemm(pa, sa, float(A[2].item()), pb, sb, float(B[2].item()))
        check_gemm_bf16(workloads.bf16_bits_to_f32(cb).astype(np.float64), R)
    return q, int(flag.item())


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (208, 320, 512), (16, 32, 256), (384, 768, 768),
                                   (608, 544, 1280)])
def test_native_path_shapes(lib, M, N, K):
    A, B = _operands(lib, workloads.activations(M, K, M + 3 * K), workloads.weights(N, K, N + 5 * K))
    _, fell = _check(lib, A, B)
    assert fell == 0


def test_stale_tensor_scales(lib):
    """Tensor scales of C far from its amax: saturated and underflowed blocks
    are encoded as the quantiser encodes them."""
    A, B = _operands(lib, workloads.activations(256, 512, 11), workloads.weights(512, 512, 12))
    for T in (1e-9, 1e-6, 1e-3):
        _check(lib, A, B, T=torch.tensor([T], dtype=torch.float32, device="cuda"))


def test_fallback_equals_the_emulated_fused_gemm(lib):
    """A row of A outside its window: the native launch writes nothing, the
    emulated fused GEMM writes every output -- bit for bit what
    fp4q_gemm_quantize writes."""
    M, N, K = 256, 512, 512
    af = workloads.bf16_bits_to_f32(workloads.activations(M, K, 13))
    af[9, :16] *= np.float32(2.0 ** -20)
    A, B = _operands(lib, workloads.f32_to_bf16_bits(af), workloads.weights(N, K, 14))
    T = lib.tensor_scale(lib.amax(lib.gemm(*A, *B)))
    q, fell = _check(lib, A, B, T=T)
    assert fell == 1
    e = lib.gemm_quantize(*A, *B, T)
    torch.cuda.synchronize()
    assert torch.equal(q.C, e.C) and torch.equal(q.payload_row, e.payload_row)
    assert torch.equal(q.scales_row, e.scales_row) and torch.equal(q.amax, e.amax)


def test_skip_flags_leave_every_output_untouched(lib):
    M, N, K = 256, 256, 256
    A, B = _operands(lib, workloads.activations(M, K, 15), workloads.weights(N, K, 16))
    a4, fa, _ = lib.rebias_scales(A[1], True)
    b4, fb, _ = lib.rebias_scales(B[1], False)
    T = torch.ones(1, device="cuda")
    C = torch.full((M, N), 3.0, device="cuda").bfloat16()
    pay = torch.full((M, N // 2), 0xA5, dtype=torch.uint8, device="cuda")
    sc = torch.full((M, N // 16), 0x5A, dtype=torch.uint8, device="cuda")
    am = torch.full((1,), 7.0, device="cuda")
    one = torch.ones(1, dtype=torch.int32, device="cuda")
    zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.fp4q_gemm_nvfp4_rebiased_quantize(A[0], a4, fa, A[2], B[0], b4, fb, B[2], M, N, K, one, lib.UE5M3, T,
                                          C, pay, sc, am)
    lib.fp4q_gemm_quantize_if(*A, *B, M, N, K, lib.UE5M3, zero, T, C, pay, sc, am)
    torch.cuda.synchronize()
    assert (C.float() == 3.0).all() and (pay == 0xA5).all() and (sc == 0x5A).all() and float(am.item()) == 7.0


def test_full_fprop(lib):
    """Y = X W^T at 8192 x 16384 x 4096 on the native path, quantised for the
    next layer in the epilogue (the BF16 result is checked by the other
    full-size tests)."""
    X, W = workloads.fprop_operands()
    A, B = _operands(lib, X, W)
    _, fell = _check(lib, A, B, full=False)
    assert fell == 0

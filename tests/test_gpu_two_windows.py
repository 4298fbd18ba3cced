"""GPU parity of the two-window exponent rebias (fp4q_rebias_scales_two_windows)
and of the UE5M3 GEMM on the native block-scaled MMA with two accumulators
(fp4q_gemm_nvfp4_two_windows), for an A operand whose rows span more binades
than one UE4M3 window holds: the column-wise codes of a gradient whose
per-token magnitudes differ by many decades (wgrad's A).

The rebias is byte work: codes and factors equal the oracle's bit for bit on
every row, fitting or not, and the flag equals the oracle's decision.  The
GEMM meets the elementwise bound against the oracle's binary64 UE5M3
contraction of the ORIGINAL operands, including outputs made of low-window
products alone (a dropped or mis-scaled low accumulator fails there), and
the device-side fallback equals plain fp4q_gemm bit for bit.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract -- UE5M3 is emulated because the tensor cores take only E4M3/E8M0
block scales; two 14-binade windows of UE4M3 codes times powers of two hold
the 28 binades under a row's largest scale exactly."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import (GEMM_TOL, check_gemm_bf16, check_gemm_elementwise, gemm_abs_reference, gemm_error,
                         np_u8, sampled_check, stripes, to_dev)
from scale_codes import codes_with_span

pytestmark = pytest.mark.gpu
UE5M3 = oracle.UE5M3


@pytest.fixture(scope="module", autouse=True)
def lib():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    yield fp4q
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("rows,nb", [(1, 16), (37, 32), (300, 16), (9, 528), (130, 256)])
@pytest.mark.parametrize("span", [0, 13, 14, 20, 27, 28, 31])
def test_codes_factors_and_flag(lib, rows, nb, span):
    """Rows of one span each (28 and more do not fit), zero rows, subnormal
    codes; every row's codes and factors equal the oracle's, the flag its
    decision."""
    rng = np.random.default_rng(rows * 1000 + nb + span)
    codes = codes_with_span(rng, rows, nb, span)
    codes[rng.random(rows) < 0.1] = 0
    hi, lo, fh, fl, flag = lib.rebias_scales_two_windows(_dev(codes))
    torch.cuda.synchronize()
    rh, rl, rfh, rfl, fits = oracle.rebias_scales2(codes)
    assert int(flag.item()) == int(not fits)
    assert fits == (span <= 27 or not codes.any())
    np.testing.assert_array_equal(np_u8(hi), rh)
    np.testing.assert_array_equal(np_u8(lo), rl)
    np.testing.assert_array_equal(fh.cpu().numpy(), rfh)
    np.testing.assert_array_equal(fl.cpu().numpy(), rfl)


def test_every_top_binade_and_offset(lib):
    """Each of the 32 top exponent fields with codes at every offset below it
    (0 .. 31 binades, both sides of each window's edge), all 8 mantissas:
    the SIMD path (normal codes) and the code-by-code path (subnormals)."""
    rows = []
    for top in range(32):
        for m in range(8):
            row = [(top << 3) | (6 if top == 31 and m == 7 else m)]   # 0xFF is not a value
            row += [((top - d) << 3) | m for d in range(1, 32) if top - d >= 1]
            row += [m or 1] if top >= 1 and m % 2 == 0 else []     # a subnormal code in half the rows
            rows.append((row + [0] * 48)[:48])
    codes = np.array(rows, np.uint8)
    hi, lo, fh, fl, flag = lib.rebias_scales_two_windows(_dev(codes))
    torch.cuda.synchronize()
    rh, rl, rfh, rfl, fits = oracle.rebias_scales2(codes)
    assert int(flag.item()) == int(not fits) == 1
    np.testing.assert_array_equal(np_u8(hi), rh)
    np.testing.assert_array_equal(np_u8(lo), rl)
    np.testing.assert_array_equal(fh.cpu().numpy(), rfh)
    np.testing.assert_array_equal(fl.cpu().numpy(), rfl)


def test_flag_is_or_ed_not_cleared(lib):
    flag = torch.ones(1, dtype=torch.int32, device="cuda")
    lib.rebias_scales_two_windows(_dev(np.full((4, 16), 0x80, np.uint8)), flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 1


def _wgrad_operands(lib, T, F, H, seed, lo=-8.0, hi=2.0):
    """wgrad of a linear H -> F over T tokens: A = dY column-wise (SR, seed 7),
    B = X column-wise; M = F, N = H, K = T."""
    dY = workloads.gradients(T, F, seed, lo, hi)
    X = workloads.activations(T, H, seed + 1)
    qd = lib.quantize(to_dev(dY), lib.AXIS_COL, None, lib.UE5M3, lib.SR, 7)
    qx = lib.quantize(to_dev(X), lib.AXIS_COL)
    return (qd.payload_col, qd.scales_col, qd.T), (qx.payload_col, qx.scales_col, qx.T)


def _oracle_check(C32, C16, A, B):
    pa, sa, pb, sb = (np_u8(t) for t in (A[0], A[1], B[0], B[1]))
    ta, tb = float(A[2].item()), float(B[2].item())
    R = oracle.gemm(pa, sa, ta, pb, sb, tb, UE5M3)
    S = gemm_abs_reference(pa, sa, pb, sb, ta * tb, UE5M3)
    C32 = C32.cpu().numpy().astype(np.float64)
    assert gemm_error(C32, R) <= GEMM_TOL
    check_gemm_elementwise(C32, R, S, pa.shape[1] * 2)
    check_gemm_bf16(C16.float().cpu().numpy().astype(np.float64), R)


def _run(lib, A, B):
    flag = torch.empty(1, dtype=torch.int32, device="cuda")
    C32 = lib.gemm_ue5m3_two_windows(*A, *B, dtype=torch.float32, nofit=flag)
    C16 = lib.gemm_ue5m3_two_windows(*A, *B, dtype=torch.bfloat16, nofit=flag)
    torch.cuda.synchronize()
    return C32, C16, int(flag.item())


@pytest.mark.parametrize("T,F,H,seed,lo", [(768, 208, 304, 2, -8.0), (1280, 384, 784, 4, -8.0),
                                           (2048, 640, 512, 5, -8.0), (512, 256, 128, 1, -12.0),
                                           (256, 16, 48, 3, -12.0)])
def test_wgrad_shapes_match_the_ue5m3_oracle(lib, T, F, H, seed, lo):
    """Gradient operands whose rows need the low window (one window does not
    fit, two do); ragged M and N, several tiles and tile columns."""
    A, B = _wgrad_operands(lib, T, F, H, seed, lo)
    sa, sb = np_u8(A[1]), np_u8(B[1])
    assert not oracle.rebias_scales(sa, True)[2]
    assert oracle.rebias_scales2(sa)[4] and oracle.rebias_scales(sb, False)[2]
    C32, C16, flag = _run(lib, A, B)
    assert flag == 0
    _oracle_check(C32, C16, A, B)


def _low_only_operands(lib, M, N, K, seed):
    """A's rows: K block 0 near 1 (each row's top), blocks 1 and 2 eight
    binades down (high window), the rest twenty down (low window); B's rows:
    weights, K blocks 0..2 zero in every even row -- so C[m, even n] is made
    of low-window products alone."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K)).astype(np.float32)
    a[:, 16:48] *= np.float32(2.0 ** -8)
    a[:, 48:] *= np.float32(2.0 ** -20)
    b = workloads.bf16_bits_to_f32(workloads.weights(N, K, seed + 1))
    b[0::2, :48] = 0
    qa = lib.quantize(to_dev(workloads.f32_to_bf16_bits(a)))
    qb = lib.quantize(to_dev(workloads.f32_to_bf16_bits(b)))
    return (qa.payload_row, qa.scales_row, qa.T), (qb.payload_row, qb.scales_row, qb.T)


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (144, 208, 768)])
def test_outputs_of_low_window_products_alone(lib, M, N, K):
    A, B = _low_only_operands(lib, M, N, K, M + N + K)
    _, lo, _, _, fits = oracle.rebias_scales2(np_u8(A[1]))
    assert fits and (lo != 0).mean() > 0.8
    C32, C16, flag = _run(lib, A, B)
    assert flag == 0
    _oracle_check(C32, C16, A, B)
    # the even columns alone, with their own scale: every entry within the
    # elementwise bound of low-window products
    pa, sa, pb, sb = (np_u8(t) for t in (A[0], A[1], B[0], B[1]))
    ta, tb = float(A[2].item()), float(B[2].item())
    R = oracle.gemm(pa, sa, ta, pb[0::2], sb[0::2], tb, UE5M3)
    S = gemm_abs_reference(pa, sa, pb[0::2], sb[0::2], ta * tb, UE5M3)
    C = C32.cpu().numpy().astype(np.float64)[:, 0::2]
    assert np.abs(R).max() < 2.0 ** -12 * np.abs(oracle.gemm(pa, sa, ta, pb[1::2], sb[1::2], tb, UE5M3)).max()
    assert gemm_error(C, R) <= GEMM_TOL
    check_gemm_elementwise(C, R, S, K)


def test_one_window_rows_through_the_two_window_path(lib):
    """Operands that one window already holds (zero low codes): the same
    contraction, within the bound of the one-window result."""
    M, N, K = 256, 384, 512
    qa = lib.quantize(to_dev(workloads.activations(M, K, 21)))
    qb = lib.quantize(to_dev(workloads.weights(N, K, 22)))
    A, B = (qa.payload_row, qa.scales_row, qa.T), (qb.payload_row, qb.scales_row, qb.T)
    _, lo, _, _, fits = oracle.rebias_scales2(np_u8(A[1]))
    assert fits and not lo.any()
    C32, C16, flag = _run(lib, A, B)
    one = lib.gemm_ue5m3_rebiased(*A, *B, dtype=torch.float32)
    torch.cuda.synchronize()
    assert flag == 0
    assert gemm_error(C32.cpu().numpy().astype(np.float64), one.cpu().numpy().astype(np.float64)) <= 1e-5
    _oracle_check(C32, C16, A, B)


def test_fallback_below_both_windows(lib):
    """A block 30 binades under its row's top (UE5M3 still holds it; two
    windows do not): the flag is set, the native launch writes nothing and the
    emulated GEMM writes C -- fp4q_gemm's result bit for bit."""
    M, N, K = 256, 256, 512
    a = np.random.default_rng(31).standard_normal((M, K)).astype(np.float32)
    a[:, 16:] *= np.float32(2.0 ** -8)
    a[7, 32:48] *= np.float32(2.0 ** -22)
    qa = lib.quantize(to_dev(workloads.f32_to_bf16_bits(a)))
    qb = lib.quantize(to_dev(workloads.weights(N, K, 32)))
    A, B = (qa.payload_row, qa.scales_row, qa.T), (qb.payload_row, qb.scales_row, qb.T)
    assert np_u8(A[1])[7, 2] != 0 and not oracle.rebias_scales2(np_u8(A[1]))[4]
    C, C16, flag = _run(lib, A, B)
    E = lib.gemm(*A, *B, dtype=torch.float32)
    torch.cuda.synchronize()
    assert flag == 1
    assert torch.equal(C, E)
    _oracle_check(C, C16, A, B)


def test_skip_flag_leaves_out_untouched(lib):
    M, N, K = 256, 256, 512
    A, B = _low_only_operands(lib, M, N, K, 41)
    ah, al, fh, _, _ = lib.rebias_scales_two_windows(A[1])
    b4, fb, _ = lib.rebias_scales(B[1], False)
    sentinel = torch.full((M, N), 12345.0, device="cuda")
    one = torch.ones(1, dtype=torch.int32, device="cuda")
    zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sentinel.clone()
    lib.fp4q_gemm_nvfp4_two_windows(A[0], ah, al, fh, A[2], B[0], b4, fb, B[2], M, N, K, one, out)
    torch.cuda.synchronize()
    assert torch.equal(out, sentinel)
    lib.fp4q_gemm_nvfp4_two_windows(A[0], ah, al, fh, A[2], B[0], b4, fb, B[2], M, N, K, zero, out)
    n = out.clone()
    out.copy_(sentinel)
    lib.fp4q_gemm_nvfp4_two_windows(A[0], ah, al, fh, A[2], B[0], b4, fb, B[2], M, N, K, None, out)
    torch.cuda.synchronize()
    assert not torch.equal(n, sentinel) and torch.equal(out, n)


def test_empty_shapes_and_k0(lib):
    e = torch.empty((0, 16), dtype=torch.uint8, device="cuda")
    f = torch.empty(0, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.fp4q_rebias_scales_two_windows(e, 0, 16, e.clone(), e.clone(), f, f.clone(), flag)
    M, N = 64, 96
    z8 = torch.zeros((M, 0), dtype=torch.uint8, device="cuda")
    zb = torch.zeros((N, 0), dtype=torch.uint8, device="cuda")
    one = torch.ones(1, device="cuda")
    out = torch.full((M, N), 7.0, device="cuda")
    lib.fp4q_gemm_nvfp4_two_windows(z8, z8, z8, torch.ones(M, device="cuda"), one, zb, zb, one, one, M, N, 0,
                                    None, out)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0 and (out == 0).all()


def test_full_size_wgrad_takes_the_native_path(lib):
    """The 8B-class linear's wgrad (16384 x 4096 x 8192: A = dY column-wise
    with SR, seed 7; B = X column-wise) as the step runs it: one window does
    not hold dY's rows, two do (the flag agrees with the oracle's decision on
    the same codes), and sampled row and column stripes meet the bound
    against the oracle's UE5M3 contraction of the original operands."""
    X, _ = workloads.fprop_operands()
    dY = workloads.backward_gradient()
    qd = lib.quantize(to_dev(dY), lib.AXIS_BOTH, None, lib.UE5M3, lib.SR, 7)
    qx = lib.quantize(to_dev(X), lib.AXIS_BOTH)
    A = (qd.payload_col, qd.scales_col, qd.T)
    B = (qx.payload_col, qx.scales_col, qx.T)
    flag = torch.empty(1, dtype=torch.int32, device="cuda")
    C = lib.gemm_ue5m3_two_windows(*A, *B, dtype=torch.float32, nofit=flag)
    torch.cuda.synchronize()
    sa = np_u8(A[1])
    assert not oracle.rebias_scales(sa, True)[2]
    assert oracle.rebias_scales2(sa)[4] and oracle.rebias_scales(np_u8(B[1]), False)[2]
    assert int(flag.item()) == 0
    rng = np.random.default_rng(4)
    err = sampled_check(A, B, C, stripes(16384, rng, 128), stripes(4096, rng, 128))
    assert err <= GEMM_TOL, err

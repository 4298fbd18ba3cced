"""GPU parity of the UE5M3 -> UE4M3 exponent rebias and of the UE5M3 GEMM
run on the native block-scaled MMA through it.

fp4q_rebias_scales is byte work: codes and factors must equal the oracle's
bit for bit for every group that fits, and the "does not fit" flag must equal
the oracle's decision.  The rebiased GEMM (fp4q_gemm_nvfp4_rebiased) must meet
the GEMM bound against the oracle's binary64 UE5M3 contraction of the
ORIGINAL operands, and the device-side fallback (fp4q_gemm_if) must make the
whole sequence equal plain fp4q_gemm when a group does not fit.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract -- UE5M3 is emulated because the tensor cores take only E4M3/E8M0
block scales; the two formats share their mantissa bits, so a group of UE5M3
scales within 14 binades is a power of two times UE4M3 scales."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import (GEMM_TOL, check_gemm_bf16, check_gemm_elementwise, gemm_abs_reference,
                         extreme_rows, gemm_error, np_u8, sampled_check, stripes, to_dev)
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


def _rebias(lib, codes, per_row):
    c4, f, flag = lib.rebias_scales(_dev(codes), per_row)
    torch.cuda.synchronize()
    return np_u8(c4), f.cpu().numpy(), int(flag.item())


def _fitting_groups(codes, per_row):
    """Per row: which rows the oracle says fit (each row alone)."""
    if not per_row:
        return None
    return np.array([oracle.rebias_scales(codes[r:r + 1], True)[2] for r in range(codes.shape[0])])


@pytest.mark.parametrize("rows,nb", [(1, 16), (37, 32), (300, 16), (9, 528), (130, 256)])
@pytest.mark.parametrize("span", [0, 7, 13, 14, 19])
def test_per_row_codes_factors_and_flag(lib, rows, nb, span):
    """Rows of one span each (span 14 and 19 do not fit), plus zero rows; nb
    up to 528 codes makes a lane handle more than one 16-code chunk."""
    rng = np.random.default_rng(rows * 1000 + nb + span)
    codes = codes_with_span(rng, rows, nb, span)
    codes[rng.random(rows) < 0.1] = 0                      # all-zero rows: factor 1, zero codes
    c4, f, flag = _rebias(lib, codes, True)
    r4, rf, fits = oracle.rebias_scales(codes, per_row=True)
    assert flag == int(not fits)
    ok = _fitting_groups(codes, True)
    assert ok.any() or span > 13
    np.testing.assert_array_equal(c4[ok], r4[ok])
    np.testing.assert_array_equal(f[ok], rf[ok])


def test_per_row_mixed_fit(lib):
    """One row that does not fit among fitting ones sets the flag; the other
    rows are still exact."""
    rng = np.random.default_rng(5)
    codes = codes_with_span(rng, 64, 64, 10)
    codes[17] = codes_with_span(rng, 1, 64, 15)[0]
    c4, f, flag = _rebias(lib, codes, True)
    r4, rf, fits = oracle.rebias_scales(codes, per_row=True)
    assert flag == 1 and not fits
    ok = np.ones(64, bool)
    ok[17] = False
    np.testing.assert_array_equal(c4[ok], r4[ok])
    np.testing.assert_array_equal(f[ok], rf[ok])


@pytest.mark.parametrize("rows,nb", [(16, 16), (1000, 32), (77, 256)])
def test_per_tensor_window(lib, rows, nb):
    """Per tensor: codes in binades 3..16 (and zeros) fit with factor 2^9,
    bit-exact; one code below binade 3 anywhere sets the flag."""
    rng = np.random.default_rng(rows + nb)
    e = rng.integers(18, 32, (rows, nb))                     # exponent fields of binades 3..16
    m = rng.integers(0, 8, (rows, nb))
    codes = ((e << 3) | m).astype(np.uint8)
    codes[codes == 0xFF] = 0xFE
    codes[rng.random((rows, nb)) < 0.05] = 0
    c4, f, flag = _rebias(lib, codes, False)
    r4, rf, fits = oracle.rebias_scales(codes, per_row=False)
    assert fits and flag == 0
    np.testing.assert_array_equal(c4, r4)
    np.testing.assert_array_equal(f, rf)
    codes[rows // 2, nb - 1] = (17 << 3) | 3                # binade 2
    _, _, flag = _rebias(lib, codes, False)
    assert flag == 1 and not oracle.rebias_scales(codes, per_row=False)[2]


def test_flag_is_or_ed_not_cleared(lib):
    codes = codes_with_span(np.random.default_rng(1), 8, 16, 3)
    flag = torch.ones(1, dtype=torch.int32, device="cuda")
    lib.rebias_scales(_dev(codes), True, flag)
    assert int(flag.item()) == 1


def _quantised(lib, a_bits, b_bits):
    qa = lib.quantize(to_dev(a_bits))
    qb = lib.quantize(to_dev(b_bits))
    return (qa.payload_row, qa.scales_row, qa.T), (qb.payload_row, qb.scales_row, qb.T)


def _oracle_check(C32, C16, A, B):
    pa, sa, pb, sb = (np_u8(t) for t in (A[0], A[1], B[0], B[1]))
    ta, tb = float(A[2].item()), float(B[2].item())
    R = oracle.gemm(pa, sa, ta, pb, sb, tb, UE5M3)
    S = gemm_abs_reference(pa, sa, pb, sb, ta * tb, UE5M3)
    C32 = C32.cpu().numpy().astype(np.float64)
    assert gemm_error(C32, R) <= GEMM_TOL
    check_gemm_elementwise(C32, R, S, pa.shape[1] * 2)
    check_gemm_bf16(C16.float().cpu().numpy().astype(np.float64), R)


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (208, 304, 512), (16, 48, 256), (384, 784, 768),
                                   (608, 528, 1280)])
def test_rebiased_gemm_matches_the_ue5m3_oracle(lib, M, N, K):
    """Quantised activations (per-channel magnitudes) and weights: every A
    row and the whole of B fit, so the native MMA computes the UE5M3 GEMM."""
    a = workloads.activations(M, K, M + K)
    b = workloads.weights(N, K, N + K)
    A, B = _quantised(lib, a, b)
    flag = torch.empty(1, dtype=torch.int32, device="cuda")
    C32 = lib.gemm_ue5m3_rebiased(*A, *B, dtype=torch.float32, nofit=flag)
    C16 = lib.gemm_ue5m3_rebiased(*A, *B, dtype=torch.bfloat16, nofit=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    _oracle_check(C32, C16, A, B)


def test_fallback_when_a_row_does_not_fit(lib):
    """A row of A whose block scales span more than 14 binades: the flag is
    set, the native launch writes nothing and the emulated GEMM writes C --
    the result is fp4q_gemm's, bit for bit, and meets the oracle bound."""
    M, N, K = 256, 512, 512
    a = workloads.activations(M, K, 3)
    af = workloads.bf16_bits_to_f32(a)
    af[5, :16] *= 2.0 ** -20                                   # one tiny block in row 5
    a = workloads.f32_to_bf16_bits(af)
    b = workloads.weights(N, K, 4)
    A, B = _quantised(lib, a, b)
    assert not oracle.rebias_scales(np_u8(A[1]), per_row=True)[2]
    flag = torch.empty(1, dtype=torch.int32, device="cuda")
    C = lib.gemm_ue5m3_rebiased(*A, *B, dtype=torch.float32, nofit=flag)
    E = lib.gemm(*A, *B, dtype=torch.float32)
    C16 = lib.gemm_ue5m3_rebiased(*A, *B, dtype=torch.bfloat16, nofit=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    assert torch.equal(C, E)
    _oracle_check(C, C16, A, B)


def test_skip_and_run_flags_leave_out_untouched(lib):
    M, N, K = 256, 256, 256
    A, B = _quantised(lib, workloads.activations(M, K, 8), workloads.weights(N, K, 9))
    a4, fa, _ = lib.rebias_scales(A[1], True)
    b4, fb, _ = lib.rebias_scales(B[1], False)
    sentinel = torch.full((M, N), 12345.0, device="cuda")
    one = torch.ones(1, dtype=torch.int32, device="cuda")
    zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sentinel.clone()
    lib.fp4q_gemm_nvfp4_rebiased(A[0], a4, fa, A[2], B[0], b4, fb, B[2], M, N, K, one, out)
    lib.fp4q_gemm_if(*A, *B, M, N, K, lib.UE5M3, zero, out)
    torch.cuda.synchronize()
    assert torch.equal(out, sentinel)
    # the same calls with the flags the other way round write C
    lib.fp4q_gemm_nvfp4_rebiased(A[0], a4, fa, A[2], B[0], b4, fb, B[2], M, N, K, zero, out)
    n = out.clone()
    out.copy_(sentinel)
    lib.fp4q_gemm_if(*A, *B, M, N, K, lib.UE5M3, one, out)
    torch.cuda.synchronize()
    assert not torch.equal(n, sentinel) and not torch.equal(out, sentinel)
    assert gemm_error(n.cpu().numpy().astype(np.float64), out.cpu().numpy().astype(np.float64)) <= GEMM_TOL
    # no flag at all: the native launch always runs
    out.copy_(sentinel)
    lib.fp4q_gemm_nvfp4_rebiased(A[0], a4, fa, A[2], B[0], b4, fb, B[2], M, N, K, None, out)
    torch.cuda.synchronize()
    assert torch.equal(out, n)


def test_full_size_fprop_and_dgrad_take_the_native_path(lib):
    """The 8B-class linear's fprop (8192 x 16384 x 4096) and dgrad (8192 x
    4096 x 16384, dY with SR, seed 7) as the step runs them: every group fits
    (the flag agrees with the oracle's decision on the same codes), and
    sampled row and column stripes meet the bound against the oracle's UE5M3
    contraction of the original operands."""
    X, W = workloads.fprop_operands()
    dY = workloads.backward_gradient()
    qx = lib.quantize(to_dev(X))
    qw = lib.quantize(to_dev(W), 2)
    qd = lib.quantize(to_dev(dY), 2, None, 0, 1, 7)
    rng = np.random.default_rng(2)
    flag = torch.empty(1, dtype=torch.int32, device="cuda")
    for A, B, M, N, extra in (((qx.payload_row, qx.scales_row, qx.T), (qw.payload_row, qw.scales_row, qw.T), 8192,
                               16384, extreme_rows(X)),
                              ((qd.payload_row, qd.scales_row, qd.T), (qw.payload_col, qw.scales_col, qw.T), 8192,
                               4096, extreme_rows(dY))):
        C = lib.gemm_ue5m3_rebiased(*A, *B, dtype=torch.float32, nofit=flag)
        torch.cuda.synchronize()
        fits = oracle.rebias_scales(np_u8(A[1]), True)[2] and oracle.rebias_scales(np_u8(B[1]), False)[2]
        assert fits and int(flag.item()) == 0, (M, N)
        # rows of extreme magnitude carry the extreme per-row factors
        rows = np.unique(np.r_[stripes(M, rng, 128), extra])
        err = sampled_check(A, B, C, rows, stripes(N, rng, 256))
        assert err <= GEMM_TOL, (M, N, err)
        del C


def test_empty_shapes_and_k0(lib):
    """No rows: the per-tensor factor is still written (2^9) and the flag
    untouched; K = 0: both GEMM entry points write zeros whatever the flag;
    M = 0: nothing is launched."""
    e = torch.empty((0, 16), dtype=torch.uint8, device="cuda")
    f = torch.full((1,), -1.0, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.fp4q_rebias_scales(e, 0, 16, False, torch.empty_like(e), f, flag)
    torch.cuda.synchronize()
    assert float(f.item()) == 512.0 and int(flag.item()) == 0
    one = torch.ones(1, device="cuda")
    z = torch.empty((16, 0), dtype=torch.uint8, device="cuda")
    set_ = torch.ones(1, dtype=torch.int32, device="cuda")
    for out in (torch.full((16, 32), 7.0, device="cuda"), torch.full((16, 32), 7.0, device="cuda").bfloat16()):
        lib.fp4q_gemm_nvfp4_rebiased(z, z, torch.ones(16, device="cuda"), one, torch.empty((32, 0), dtype=torch.uint8,
                                     device="cuda"), torch.empty((32, 0), dtype=torch.uint8, device="cuda"), one, one,
                                     16, 32, 0, set_, out)
        torch.cuda.synchronize()
        assert (out == 0).all()
        out.fill_(7.0)
        lib.fp4q_gemm_if(z, z, one, torch.empty((32, 0), dtype=torch.uint8, device="cuda"),
                         torch.empty((32, 0), dtype=torch.uint8, device="cuda"), one, 16, 32, 0, lib.UE5M3,
                         torch.zeros(1, dtype=torch.int32, device="cuda"), out)
        torch.cuda.synchronize()
        assert (out == 0).all()
    out = torch.empty((0, 32), device="cuda")
    lib.fp4q_gemm_if(torch.empty((0, 128), dtype=torch.uint8, device="cuda"),
                     torch.empty((0, 16), dtype=torch.uint8, device="cuda"), one,
                     torch.empty((32, 128), dtype=torch.uint8, device="cuda"),
                     torch.empty((32, 16), dtype=torch.uint8, device="cuda"), one, 0, 32, 256, lib.UE5M3, set_, out)
    torch.cuda.synchronize()


def test_per_tensor_b_that_does_not_fit_falls_back(lib):
    """B's fixed window fails (one B block far below the tensor's amax):
    the sequence equals fp4q_gemm bit for bit, BF16 and FP32."""
    M, N, K = 256, 256, 512
    a = workloads.activations(M, K, 21)
    bf = workloads.bf16_bits_to_f32(workloads.weights(N, K, 22))
    bf[7, 32:48] *= np.float32(2.0 ** -24)
    A, B = _quantised(lib, a, workloads.f32_to_bf16_bits(bf))
    assert not oracle.rebias_scales(np_u8(B[1]), per_row=False)[2]
    flag = torch.empty(1, dtype=torch.int32, device="cuda")
    for dt in (torch.float32, torch.bfloat16):
        C = lib.gemm_ue5m3_rebiased(*A, *B, dtype=dt, nofit=flag)
        E = lib.gemm(*A, *B, dtype=dt)
        torch.cuda.synchronize()
        assert int(flag.item()) == 1 and torch.equal(C, E)


def test_full_size_rebias_bytes(lib):
    """The step's four rebias inputs at the 8B-class sizes, byte for byte
    against the oracle: X's and dY's row-wise codes per row (8192 x 256 and
    8192 x 1024), W's row-wise and column-wise codes per tensor (16384 x 256
    and 4096 x 1024)."""
    X, W = workloads.fprop_operands()
    dY = workloads.backward_gradient()
    qx = lib.quantize(to_dev(X))
    qw = lib.quantize(to_dev(W), 2)
    qd = lib.quantize(to_dev(dY), 2, None, 0, 1, 7)
    for codes, per_row in ((qx.scales_row, True), (qd.scales_row, True), (qw.scales_row, False),
                           (qw.scales_col, False)):
        c4, f, flag = lib.rebias_scales(codes, per_row)
        torch.cuda.synchronize()
        r4, rf, fits = oracle.rebias_scales(np_u8(codes), per_row=per_row)
        assert fits and int(flag.item()) == 0, (tuple(codes.shape), per_row)
        np.testing.assert_array_equal(np_u8(c4), r4)
        np.testing.assert_array_equal(f.cpu().numpy(), rf)


def test_rows_beyond_one_pass_of_the_grid(lib):
    """More rows than the per-row kernel's grid holds warps (each warp then
    takes several rows), mixed spans and zero rows."""
    rng = np.random.default_rng(77)
    codes = codes_with_span(rng, 30000, 16, 9)
    codes[rng.random(30000) < 0.02] = 0
    c4, f, flag = _rebias(lib, codes, True)
    r4, rf, fits = oracle.rebias_scales(codes, per_row=True)
    assert fits and flag == 0
    np.testing.assert_array_equal(c4, r4)
    np.testing.assert_array_equal(f, rf)


@pytest.mark.parametrize("name", ["qkv", "out", "down"])
def test_block_linears_through_the_native_path(lib, name):
    """The 8B-class block's other linears (qkv 4096->6144, out 4096->4096,
    down 16384->4096; up is the full-size case above), 8192 tokens: fprop
    and dgrad through rebiased codes, as the block step runs them -- the
    flag agrees with the oracle's fit decision and sampled row and column
    stripes meet the bound against the oracle's UE5M3 contraction."""
    X, W, dY = workloads.linear_block(name)
    fin, fout = workloads.LINEARS[name]
    qx = lib.quantize(to_dev(X))
    qw = lib.quantize(to_dev(W), 2)
    qd = lib.quantize(to_dev(dY), 2, None, 0, 1, 7)
    rng = np.random.default_rng(len(name) + 100)
    flag = torch.empty(1, dtype=torch.int32, device="cuda")
    for A, B, M, N in (((qx.payload_row, qx.scales_row, qx.T), (qw.payload_row, qw.scales_row, qw.T), 8192, fout),
                       ((qd.payload_row, qd.scales_row, qd.T), (qw.payload_col, qw.scales_col, qw.T), 8192, fin)):
        C = lib.gemm_ue5m3_rebiased(*A, *B, dtype=torch.float32, nofit=flag)
        torch.cuda.synchronize()
        fits = oracle.rebias_scales(np_u8(A[1]), True)[2] and oracle.rebias_scales(np_u8(B[1]), False)[2]
        assert int(flag.item()) == int(not fits), (name, M, N)
        err = sampled_check(A, B, C, stripes(M, rng, 128), stripes(N, rng, 256))
        assert err <= GEMM_TOL, (name, M, N, err)
        del C


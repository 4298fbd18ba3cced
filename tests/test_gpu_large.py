"""GPU parity past 2^31 elements: every quantiser layout and the GEMM
epilogue on tensors whose element index (and BF16 byte offset) no longer fits
32 bits, compared with the oracle on row bands at the start, around element
2^30 (byte offset 2^31), across element 2^31 and at the end.

The input is a seeded gradient-like block (per-row magnitudes 1e-8 .. 1e2)
repeated down the rows on the device, so each band's input is known on the
host; stochastic rounding still draws different bits in every repeat (its
counter is the element's logical index), which the oracle's band evaluation
reproduces.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (E2M1 + UE5M3 block-16 quantisation, stochastic rounding of
gradients, FP4 matrix multiplications)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import GEMM_TOL, bf16_ulp, check_gemm_elementwise, to_dev

pytestmark = pytest.mark.gpu

COLS = 16384
BASE_ROWS = 1024
ROWS = 128 * BASE_ROWS + 128          # 131200 rows: 2,149,580,800 elements > 2^31
BANDS = [(0, 128), (65536 - 64, 65536 + 64), (131072 - 64, 131072 + 64), (ROWS - 64, ROWS)]
ROW, COL, BOTH, BOTH_2D = 0, 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def lib():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    yield fp4q
    assert fp4q.fp4q_get_device_status() == fp4q.OK


@pytest.fixture(scope="module")
def base():
    return workloads.gradients(BASE_ROWS, COLS, seed=41)


@pytest.fixture(scope="module")
def big(base):
    b = to_dev(base)
    x = torch.empty((ROWS, COLS), dtype=torch.bfloat16, device="cuda")
    for k in range(ROWS // BASE_ROWS):
        x[k * BASE_ROWS:(k + 1) * BASE_ROWS] = b
    x[ROWS - ROWS % BASE_ROWS:] = b[:ROWS % BASE_ROWS]
    torch.cuda.synchronize()
    yield x
    del x
    torch.cuda.empty_cache()


def band_bits(base, r0, r1):
    return np.ascontiguousarray(base[np.arange(r0, r1) % BASE_ROWS])


def test_amax_and_scale(lib, big, base):
    a = lib.amax(big)
    T = lib.tensor_scale(a)
    a_or = oracle.amax(base)[0]
    assert float(a.item()) == a_or
    assert float(T.item()) == oracle.tensor_scale(a_or)


@pytest.mark.parametrize("axis,rnd", [(BOTH, 0), (BOTH, 1), (ROW, 1), (ROW, 0), (BOTH_2D, 0)])
def test_quantize_bands(lib, big, base, axis, rnd):
    T = lib.tensor_scale(lib.amax(big))
    Tf = float(T.item())
    q = lib.quantize(big, axis, T, 0, rnd, 7, stats=axis != BOTH_2D, want_amax=True)
    torch.cuda.synchronize()
    assert float(q.amax.item()) == oracle.amax(base)[0]
    for r0, r1 in BANDS:
        bits = band_bits(base, r0, r1)
        if axis == BOTH_2D:
            pr, sr, pc, sc, _ = oracle.quantize_2d(bits, Tf)
        else:
            pr, sr, _ = oracle.quantize(bits, ROW, Tf, rnd=rnd, seed=7, row_base=r0)
            pc = sc = None
            if axis != ROW:
                pc, sc, _ = oracle.quantize(bits, COL, Tf, rnd=rnd, seed=7, row_base=r0)
        assert np.array_equal(q.payload_row[r0:r1].cpu().numpy(), pr), (r0, "row payload")
        assert np.array_equal(q.scales_row[r0:r1].cpu().numpy(), sr), (r0, "row scales")
        if pc is not None:
            gpc = q.payload_col[:, r0 // 2:r1 // 2].contiguous().cpu().numpy()
            gsc = q.scales_col[:, r0 // 16:r1 // 16].contiguous().cpu().numpy()
            assert np.array_equal(gpc, pc), (r0, "column payload")
            assert np.array_equal(gsc, sc), (r0, "column scales")
    if axis != BOTH_2D:
        # counts: the repeats of the base plus the partial repeat at the end
        reps, tail = ROWS // BASE_ROWS, ROWS % BASE_ROWS
        gst = q.stats.cpu().numpy().astype(np.uint64)
        for k, ax in enumerate([ROW] if axis == ROW else [ROW, COL]):
            full = oracle.quantize(base, ax, Tf)[2]
            part = oracle.quantize(np.ascontiguousarray(base[:tail]), ax, Tf)[2]
            want = full * np.uint64(reps) + part
            if rnd:   # flushed counts depend on the random bits; the rest do not
                assert np.array_equal(gst[k][:3], want[:3]), (ax, gst[k], want)
            else:
                assert np.array_equal(gst[k], want), (ax, gst[k], want)
    del q
    torch.cuda.empty_cache()


def test_gemm_output_past_2_31(lib):
    """C [65792, 32768] (2,155,872,256 elements) with K = 64: FP32 and BF16
    results, and the epilogue-quantised result, on row stripes past element
    2^31 and on column stripes, against the oracle."""
    M, N, K = 65536 + 256, 32768, 64
    rng = np.random.default_rng(43)
    a = workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    b = workloads.f32_to_bf16_bits((rng.standard_normal((N, K)) *
                                    10.0 ** rng.uniform(-2, 2, (N, 1))).astype(np.float32))
    qa, qb = lib.quantize(to_dev(a)), lib.quantize(to_dev(b))
    A = (qa.payload_row, qa.scales_row, qa.T)
    B = (qb.payload_row, qb.scales_row, qb.T)
    pa, sa, pb, sb = (t.cpu().numpy() for t in (A[0], A[1], B[0], B[1]))
    alpha = float(A[2].item()) * float(B[2].item())
    rows = np.r_[0:64, 65536 - 32:65536 + 32, M - 64:M]
    cols = np.r_[0:32, N - 32:N]
    ea, eb = oracle.deq_es(pa[rows], sa[rows]), oracle.deq_es(pb, sb)
    Ra, Sa = alpha * (ea @ eb.T), alpha * (np.abs(ea) @ np.abs(eb).T)
    ea, eb = oracle.deq_es(pa, sa), oracle.deq_es(pb[cols], sb[cols])
    Rc, Sc = alpha * (ea @ eb.T), alpha * (np.abs(ea) @ np.abs(eb).T)
    del ea, eb
    scale = max(np.abs(Ra).max(), np.abs(Rc).max())
    for dtype in (torch.float32, torch.bfloat16):
        C = lib.gemm(*A, *B, dtype=dtype)
        torch.cuda.synchronize()
        ca = C[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64)
        cc = C[:, torch.from_numpy(cols).cuda()].float().cpu().numpy().astype(np.float64)
        if dtype == torch.float32:
            assert np.abs(ca - Ra).max() / scale <= GEMM_TOL
            assert np.abs(cc - Rc).max() / scale <= GEMM_TOL
            check_gemm_elementwise(ca, Ra, Sa, K)
            check_gemm_elementwise(cc, Rc, Sc, K)
        else:   # one BF16 ulp of R plus 1e-3 of the largest |R| of the stripes, per element
            assert (np.abs(ca - Ra) <= bf16_ulp(Ra) + GEMM_TOL * scale).all()
            assert (np.abs(cc - Rc) <= bf16_ulp(Rc) + GEMM_TOL * scale).all()
        del C
        torch.cuda.empty_cache()
    # epilogue quantisation: row bands against the oracle's quantisation of
    # the GPU's own BF16 result
    T = lib.tensor_scale(torch.tensor([float(scale)], dtype=torch.float32, device="cuda"))
    q = lib.gemm_quantize(*A, *B, T)
    torch.cuda.synchronize()
    for r0, r1 in ((0, 32), (65536 - 16, 65536 + 16), (M - 32, M)):
        cb = q.C[r0:r1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        p, s, _ = oracle.quantize(cb, ROW, float(T.item()))
        assert np.array_equal(q.payload_row[r0:r1].cpu().numpy(), p), r0
        assert np.array_equal(q.scales_row[r0:r1].cpu().numpy(), s), r0
    del q
    torch.cuda.empty_cache()

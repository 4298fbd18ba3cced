"""Pins of the oracle's re-expression of UE5M3 block scales as UE4M3 scales
times one power of two per row (or per tensor).

The two formats share their 3 mantissa bits ("UE5M3 FP4 Block Scaling for
Stable Language Model Pretraining", Abstract: UE5M3 is emulated because the
tensor cores take E4M3/E8M0 block scales), so a group of UE5M3 scales whose
non-zero values span at most 14 binades is exactly f * (UE4M3 values): the
dequantised operand, and hence the GEMM, is unchanged.  Checked here against
values decoded independently of the oracle's decoder (from the format
definitions), brute-force binade spans, and the oracle's own dequantised
operands and GEMM."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from scale_codes import codes_with_span as _codes_with_span


def _ue5m3(code):
    """Exact value of a UE5M3 code from the format definition (bias 15,
    exponent 0 subnormal, 0xFF not a value)."""
    e, m = code >> 3, code & 7
    return Fraction(m, 8) * Fraction(2) ** -14 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 15)


def _ue4m3(code):
    e, m = code >> 3, code & 7
    return Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


V5 = [_ue5m3(c) for c in range(255)]
V4 = [_ue4m3(c) for c in range(127)]


def _binade(v):
    """floor(log2 v) of a positive rational."""
    e = 0
    while v >= 2:
        v /= 2
        e += 1
    while v < 1:
        v *= 2
        e -= 1
    return e


@pytest.mark.parametrize("span", [0, 5, 13])
def test_fitting_rows_are_exact(span):
    rng = np.random.default_rng(span)
    codes = _codes_with_span(rng, 64, 48, span)
    c4, f, fits = oracle.rebias_scales(codes, per_row=True)
    assert fits
    for r in range(codes.shape[0]):
        fr = Fraction(float(f[r]))
        assert fr.numerator == 1 or fr.denominator == 1    # a power of two
        for i in range(codes.shape[1]):
            assert V4[c4[r, i]] * fr == V5[codes[r, i]], (r, i, codes[r, i], c4[r, i])
            assert c4[r, i] == 0 or 1 <= (c4[r, i] >> 3) <= 14   # UE4M3 normal, never the NaN code
        # the convention f = 2^(e_max - 7): the row's largest scale lands in
        # UE4M3's exponent field 14 (values in [128, 256))
        if (codes[r] != 0).any():
            assert (c4[r] >> 3).max() == 14


def test_fit_flag_is_the_binade_span():
    rng = np.random.default_rng(7)
    for span in range(10, 18):
        codes = _codes_with_span(rng, 8, 32, span)
        _, _, fits = oracle.rebias_scales(codes, per_row=True)
        spans = []
        for r in range(codes.shape[0]):
            b = [_binade(V5[c]) for c in codes[r] if c != 0]
            spans.append(max(b) - min(b))
        assert max(spans) == span
        assert fits == (span <= 13), span


def test_per_tensor_window_and_zero_group():
    """Per tensor: the fixed window of binades 3..16, f = 2^9, decided code by
    code."""
    rng = np.random.default_rng(3)
    for top, span in ((16, 6), (16, 13), (12, 9), (16, 14), (10, 9), (2, 0)):
        codes = _codes_with_span(np.random.default_rng(top * 100 + span), 16, 32, span)
        # move every row's window so that its top binade is `top`
        c = codes.astype(np.int32)
        e = c >> 3
        shift = top - max(_binade(V5[x]) for x in codes.ravel() if x != 0)
        normal = (c != 0) & (e > 0)
        codes = np.where(normal & (e + shift >= 1) & (e + shift <= 31), ((e + shift) << 3) | (c & 7), c)
        codes = np.where(codes == 0xFF, 0xFE, codes).astype(np.uint8)
        c4, f, fits = oracle.rebias_scales(codes, per_row=False)
        allb = [_binade(V5[x]) for x in codes.ravel() if x != 0]
        assert f.shape == (1,) and float(f[0]) == 512.0
        assert fits == (min(allb) >= 3 and max(allb) <= 16), (top, span)
        if fits:
            assert all(V4[a] * 512 == V5[b] for a, b in zip(c4.ravel(), codes.ravel()))
    z = np.zeros((3, 16), np.uint8)
    c4, f, fits = oracle.rebias_scales(z, per_row=True)
    assert fits and (c4 == 0).all() and (f == 1.0).all()
    # the largest UE5M3 scale (114688 = 1.75 * 2^16) lands on UE4M3 1.75 * 2^7
    top = np.array([[0xFE, 0xF0]], np.uint8)             # 1.75 * 2^16 and 2^15
    for per_row in (True, False):
        c4, f, fits = oracle.rebias_scales(top, per_row=per_row)
        assert fits and c4[0, 0] == (14 << 3 | 6) and float(f[0]) == 2.0 ** 9


def test_quantised_operand_and_gemm_are_unchanged():
    """deq(payload, UE4M3 codes) * f equals deq(payload, UE5M3 codes), element
    by element, and so does the binary64 GEMM scaled by the factors."""
    rng = np.random.default_rng(11)
    a = workloads.activations(64, 512, 5)
    b = workloads.weights(96, 512, 6)
    ta = oracle.tensor_scale(oracle.amax(a)[0])
    tb = oracle.tensor_scale(oracle.amax(b)[0])
    pa, sa, _ = oracle.quantize(a, oracle.ROW, ta)
    pb, sb, _ = oracle.quantize(b, oracle.ROW, tb)
    sa4, fa, oka = oracle.rebias_scales(sa, per_row=True)
    sb4, fb, okb = oracle.rebias_scales(sb, per_row=False)
    assert oka and okb
    ea5 = oracle.deq_es(pa, sa, oracle.UE5M3)
    ea4 = oracle.deq_es(pa, sa4, oracle.UE4M3) * fa.astype(np.float64)[:, None]
    assert np.array_equal(ea4, ea5)
    eb5 = oracle.deq_es(pb, sb, oracle.UE5M3)
    eb4 = oracle.deq_es(pb, sb4, oracle.UE4M3) * float(fb[0])
    assert np.array_equal(eb4, eb5)
    R5 = oracle.gemm(pa, sa, ta, pb, sb, tb, oracle.UE5M3)
    R4 = oracle.gemm(pa, sa4, ta, pb, sb4, tb, oracle.UE4M3) * fa.astype(np.float64)[:, None] * float(fb[0])
    assert np.array_equal(R4, R5)
    del rng


@pytest.mark.parametrize("span", [0, 9, 13, 14, 20, 27, 28, 31])
def test_two_windows_are_exact(span):
    """Two windows per row: every value is hi * f_hi + lo * f_lo exactly,
    with one of the two codes zero; a value sits in the hi window iff its
    binade is within 13 of the row's top (else the lo one, down to 27);
    the fit flag is "span <= 27"; factors 2^(e_top - 7) and 2^(e_top - 21)."""
    rng = np.random.default_rng(100 + span)
    codes = _codes_with_span(rng, 24, 64, span)
    hi, lo, fh, fl, fits = oracle.rebias_scales2(codes)
    spans = []
    for r in range(codes.shape[0]):
        vals = [V5[c] for c in codes[r] if c != 0]
        b = [_binade(v) for v in vals]
        spans.append(max(b) - min(b))
        top = max(b)
        assert Fraction(float(fh[r])) == Fraction(2) ** (top - 7)
        assert Fraction(float(fl[r])) == Fraction(2) ** (top - 21)
        for i, c in enumerate(codes[r]):
            if c == 0:
                assert hi[r, i] == 0 and lo[r, i] == 0
                continue
            e = _binade(V5[c])
            if e < top - 27:
                continue   # outside both windows: codes unspecified
            assert (hi[r, i] != 0) == (e >= top - 13) and (lo[r, i] != 0) == (e < top - 13)
            assert V4[hi[r, i]] * Fraction(float(fh[r])) + V4[lo[r, i]] * Fraction(float(fl[r])) == V5[c]
            for x in (hi[r, i], lo[r, i]):
                assert x == 0 or 1 <= (x >> 3) <= 14
    assert fits == (max(spans) <= 27)


def test_two_windows_reduce_to_one_within_fourteen_binades():
    """Rows spanning at most 13 binades: the hi codes and factor are the
    one-window rebias's, the lo codes all zero."""
    rng = np.random.default_rng(5)
    codes = _codes_with_span(rng, 40, 48, 11)
    codes[3] = 0
    hi, lo, fh, fl, fits = oracle.rebias_scales2(codes)
    c4, f, fits1 = oracle.rebias_scales(codes, per_row=True)
    assert fits and fits1
    assert np.array_equal(hi, c4) and np.array_equal(fh, f) and not lo.any()
    assert float(fh[3]) == 1.0 and float(fl[3]) == 2.0 ** -14


def test_two_window_gemm_is_the_ue5m3_gemm():
    """The UE5M3 GEMM of a wide-span operand equals f_hi * GEMM(hi codes) +
    f_lo * GEMM(lo codes) of the same payload (binary64; the two sides sum
    the same exact products in different orders)."""
    rng = np.random.default_rng(21)
    g = workloads.bf16_bits_to_f32(workloads.gradients(4096, 64, 9))   # per-token magnitudes over ten decades
    gt = workloads.f32_to_bf16_bits(np.ascontiguousarray(g.T))          # rows: features, K: tokens
    x = workloads.activations(96, 4096, 10)
    ta, tb = oracle.tensor_scale(oracle.amax(gt)[0]), oracle.tensor_scale(oracle.amax(x)[0])
    pa, sa, _ = oracle.quantize(gt, oracle.ROW, ta)
    pb, sb, _ = oracle.quantize(x, oracle.ROW, tb)
    hi, lo, fh, fl, fits = oracle.rebias_scales2(sa)
    assert fits and lo.any()                       # the span needs the second window
    R5 = oracle.gemm(pa, sa, ta, pb, sb, tb, oracle.UE5M3)
    del rng
    # B keeps its UE5M3 codes; A's dequantised values split exactly by window
    ea5 = oracle.deq_es(pa, sa, oracle.UE5M3)
    ea2 = (oracle.deq_es(pa, hi, oracle.UE4M3) * fh.astype(np.float64)[:, None]
           + oracle.deq_es(pa, lo, oracle.UE4M3) * fl.astype(np.float64)[:, None])
    assert np.array_equal(ea2, ea5)
    eb = oracle.deq_es(pb, sb, oracle.UE5M3)
    R2 = ta * tb * (fh.astype(np.float64)[:, None] * (oracle.deq_es(pa, hi, oracle.UE4M3) @ eb.T)
                    + fl.astype(np.float64)[:, None] * (oracle.deq_es(pa, lo, oracle.UE4M3) @ eb.T))
    assert np.abs(R2 - R5).max() <= 1e-12 * np.abs(R5).max()


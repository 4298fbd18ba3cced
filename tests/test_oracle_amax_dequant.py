"""Pins of three oracle steps that every GPU parity check leans on -- the
tensor amax, the dequantised operand matrix e*s that the full-size GEMM checks
contract, and the BF16 rounding of the dequantiser -- each against a model
written here from the format definitions, never by calling the oracle's own
arithmetic twice.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (current/periodic tensor scaling from an amax; E2M1 payloads with
UE5M3 block-16 scales; the FP4 matrix multiplications over the dequantised
operands).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

F = Fraction


# ------------------------------------------------------------------ amax
def _amax_model(bits: np.ndarray):
    """numpy's own view of the BF16 patterns as binary32 (bits << 16), max of
    |x| over the finite entries, and whether any entry is inf or NaN."""
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    fin = np.isfinite(x)
    m = float(np.abs(x[fin]).max()) if fin.any() else 0.0
    return m, bool((~fin).any())


def _bf16(values) -> np.ndarray:
    v = np.asarray(values, np.float32).view(np.uint32)
    assert not (v & 0xFFFF).any()
    return (v >> 16).astype(np.uint16)


POS_INF, NEG_INF, QNAN, NEG_NAN = 0x7F80, 0xFF80, 0x7FC0, 0xFFC1


@pytest.mark.parametrize("n", [0, 1, 2, 7, 8, 9, 16, 1023, 1024, 4097])
def test_amax_equals_numpy_max_of_magnitudes(n):
    rng = np.random.default_rng(n + 5)
    # random BF16 patterns of both signs over a wide range of magnitudes
    bits = (rng.standard_normal(n).astype(np.float32) * np.float32(3.0)).view(np.uint32) >> 16
    bits = bits.astype(np.uint16)
    got, bad = oracle.amax(bits)
    want, wbad = _amax_model(bits)
    assert (got, bad) == (want, wbad)


def test_amax_special_positions_and_values():
    # the largest magnitude in the last element, at odd and even lengths
    for n in (15, 16):
        x = np.arange(n, dtype=np.float32) / 8 - 1      # BF16-exact
        x[-1] = -5.0
        bits = _bf16(x)
        assert oracle.amax(bits) == (5.0, False) == _amax_model(bits)
    # a negative maximum magnitude in the first element
    bits = _bf16([-7.5, 1.0, 2.0, -3.0, 0.5])
    assert oracle.amax(bits) == (7.5, False)
    # -0 and +0 only
    assert oracle.amax(np.array([0x8000, 0x0000, 0x8000], np.uint16)) == (0.0, False)
    # BF16 subnormals: the smallest (2^-133) and the largest (127 * 2^-133)
    sub = np.array([0x0001, 0x807F, 0x0003], np.uint16)
    got, bad = oracle.amax(sub)
    assert not bad and F(got) == F(127, 2 ** 133)
    assert (got, bad) == _amax_model(sub)
    # the largest finite BF16 magnitude (negative) beside a smaller value
    big = np.array([0x3F80, 0xFF7F], np.uint16)
    assert oracle.amax(big) == (float(np.array([0x7F7F0000], np.uint32).view(np.float32)[0]), False)


@pytest.mark.parametrize("special", [POS_INF, NEG_INF, QNAN, NEG_NAN])
def test_amax_skips_non_finite_and_flags_them(special):
    for pos in (0, 3, 8):
        bits = _bf16([1.0, -2.0, 0.5, 1.5, 0.25, -0.75, 1.25, 0.125, 3.0])
        bits[pos] = special
        got, bad = oracle.amax(bits)
        assert bad
        want, _ = _amax_model(bits)
        assert got == want
        assert got == (2.0 if pos == 8 else 3.0)
    # nothing finite: amax 0, flagged
    assert oracle.amax(np.array([special] * 3, np.uint16)) == (0.0, True)


# ------------------------------------------------------------------ e * s
E2M1_MAG = [F(0), F(1, 2), F(1), F(3, 2), F(2), F(3), F(4), F(6)]


def _scale_value(code: int, fmt: int) -> Fraction:
    """The scale formats from their definition: 3 mantissa bits; UE5M3 has a
    5-bit exponent with bias 15, UE4M3 a 4-bit exponent with bias 7; exponent
    field 0 is subnormal (m/8 * 2^(1 - bias))."""
    bias = 15 if fmt == oracle.UE5M3 else 7
    e, m = code >> 3, code & 7
    if e == 0:
        return F(m, 8) * F(2) ** (1 - bias)
    return (1 + F(m, 8)) * F(2) ** (e - bias)


def _es_model(payload: np.ndarray, scales: np.ndarray, fmt: int):
    """Element k of row o: nibble k % 2 of byte k // 2 (even element in the
    low nibble), times the scale of block k // 16 of that row."""
    outer, inner = payload.shape[0], payload.shape[1] * 2
    out = [[None] * inner for _ in range(outer)]
    for o in range(outer):
        for k in range(inner):
            nib = (int(payload[o, k // 2]) >> (4 * (k % 2))) & 15
            e = E2M1_MAG[nib & 7] * (-1 if nib & 8 else 1)
            out[o][k] = e * _scale_value(int(scales[o, k // 16]), fmt)
    return out


@pytest.mark.parametrize("outer,inner,fmt", [(3 * 16, 32, oracle.UE5M3), (16, 80, oracle.UE5M3),
                                             (32, 48, oracle.UE4M3)])
def test_deq_es_matrix_layout_and_values(outer, inner, fmt):
    rng = np.random.default_rng(outer * 7 + inner)
    payload = rng.integers(0, 256, (outer, inner // 2), dtype=np.uint8)
    top = 0xFE if fmt == oracle.UE5M3 else 0x7E
    scales = rng.integers(0, top + 1, (outer, inner // 16), dtype=np.uint8)
    scales[0, 0] = 0          # zero scale
    scales[-1, -1] = top      # largest scale
    scales[outer // 2, 0] = 1  # smallest subnormal
    got = oracle.deq_es(payload, scales, fmt)
    assert got.shape == (outer, inner)
    want = _es_model(payload, scales, fmt)
    for o in range(outer):
        for k in range(inner):
            assert F(float(got[o, k])) == want[o][k], (o, k)


def test_deq_es_matrix_contracts_to_the_gemm():
    # orc_gemm over (A, B) equals T_A T_B (e s)_A (e s)_B^T built from the
    # model above, in exact rationals, on operands whose products sum exactly
    rng = np.random.default_rng(3)
    M, N, K = 16, 32, 48
    A = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    As = rng.integers(0x70, 0x80, (M, K // 16), dtype=np.uint8)   # scales near 1
    Bs = rng.integers(0x70, 0x80, (N, K // 16), dtype=np.uint8)
    TA, TB = 0.75, 2.0 ** -3
    got = oracle.gemm(A, As, TA, B, Bs, TB)
    ea, eb = _es_model(A, As, 0), _es_model(B, Bs, 0)
    for m in range(M):
        for n in range(N):
            exact = F(TA) * F(TB) * sum(ea[m][k] * eb[n][k] for k in range(K))
            assert F(float(got[m, n])) == exact


# ------------------------------------------------------------------ BF16 output
def _f32_rne(x: Fraction) -> Fraction:
    """Round a rational to binary32 (normal range), nearest, ties to even."""
    if x == 0:
        return F(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    q = round(a * 2 ** 23)          # Fraction rounding: half to even
    return sign * F(q, 2 ** 23) * F(2) ** e


def _bf16_rne_bits(v: Fraction) -> int:
    """BF16 nearest-even rounding of a rational in the normal/subnormal range:
    8 significant bits above 2^-126, a fixed quantum of 2^-133 below."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    quantum = F(2) ** (max(e, -126) - 7)
    r = round(abs(v) / quantum) * quantum       # half to even
    assert r < F(2) ** 128                       # stays finite in these tests
    f = np.array([float(r)], np.float32)
    assert F(float(f[0])) == r
    return sign | int(f.view(np.uint32)[0] >> 16)


@pytest.mark.parametrize("T", [1 + 2 ** -8, 1 + 3 * 2 ** -9, 0.1, 0.7071067690849304, 2.0 ** -120 * 1.3])
def test_dequantize_rounds_to_binary32_then_bf16_nearest_even(T):
    T = float(np.float32(T))
    rng = np.random.default_rng(int(T * 1e6) % 1000)
    outer, inner = 16, 64
    payload = rng.integers(0, 256, (outer, inner // 2), dtype=np.uint8)
    scales = rng.integers(0x60, 0x90, (outer, inner // 16), dtype=np.uint8)
    f, b = oracle.dequantize(payload, scales, T)
    es = _es_model(payload, scales, oracle.UE5M3)
    n_inexact = 0
    for o in range(outer):
        for k in range(inner):
            v = _f32_rne(es[o][k] * F(T))
            assert F(float(f[o, k])) == v, (o, k)
            neg_zero = es[o][k] == 0 and (int(payload[o, k // 2]) >> (4 * (k % 2))) & 8
            assert int(b[o, k]) == (0x8000 if neg_zero else _bf16_rne_bits(v)), (o, k)
            n_inexact += F(float((np.array([b[o, k]], np.uint32) << 16).view(np.float32)[0])) != v
    if T != 2.0 ** -120 * 1.3:
        assert n_inexact > 0      # the case really exercises the BF16 rounding


def test_dequantize_bf16_ties_go_to_even():
    # T = 1 + 2^-8 puts e*s*T exactly halfway between two BF16 neighbours for
    # e*s = 1, 2 and -1 (each goes to the even neighbour, here e*s itself);
    # e*s = 1.5 lands three quarters of the way up and rounds up
    T = 1 + 2 ** -8
    payload = np.zeros((16, 8), np.uint8)
    payload[0, 0] = 0x2 | (0x3 << 4)     # elements 1.0 and 1.5
    payload[0, 1] = 0x4 | (0xA << 4)     # elements 2.0 and -1.0
    scales = np.full((16, 1), 0x78, np.uint8)   # scale 1.0
    f, b = oracle.dequantize(payload, scales, T)
    want = {0: 1.0, 1: 1.5078125, 2: 2.0, 3: -1.0}
    for k, w in want.items():
        got = float((np.array([b[0, k]], np.uint32) << 16).view(np.float32)[0])
        assert got == w, (k, got, w)

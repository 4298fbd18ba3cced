"""Pins of the oracle's tensor-level steps: tensor scale, block-16
quantisation (row-wise and column-wise, RNE and SR), dequantisation and the
binary64 GEMM -- by invariants, crafted blocks with known answers, and brute
force in exact rationals.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (block-16 UE5M3 scales over E2M1 payloads, periodic tensor scaling,
stochastic rounding on backward gradients, FP4 matrix multiplications).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])


def bf16_bits(x):
    """float32 values that are exactly BF16 -> their uint16 patterns."""
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32)
    assert not (u & 0xFFFF).any(), "value is not exactly representable in BF16"
    return (u >> 16).astype(np.uint16)


def bf16_round(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bits_to_f32(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32)


def nib_values(payload):
    lo = payload & 15
    hi = payload >> 4
    n = np.stack([lo, hi], -1).reshape(payload.shape[0], -1)
    mag = E2M1[n & 7]
    return np.where(n & 8, -mag, mag)


# ------------------------------------------------------------ tensor scale
def test_tensor_scale_closed_forms():
    # T = amax / (6 * Smax / H): 6 * 114688 = 688128 for UE5M3, 6 * 448 = 2688
    assert oracle.tensor_scale(688128.0) == 1.0
    assert oracle.tensor_scale(2688.0, oracle.UE4M3) == 1.0
    assert oracle.tensor_scale(688128.0 * 2 ** -20) == 2 ** -20
    assert oracle.tensor_scale(0.0) == 1.0
    # one correctly rounded division: the exact quotient is within half an ulp
    for a in (1.0, 3.0, 6.5, 1234.5, 1e-8, 3e30):
        t = oracle.tensor_scale(a)
        q = Fraction(float(np.float32(a))) / 688128
        ulp = Fraction(float(np.spacing(np.float32(t))))
        assert abs(Fraction(t) - q) <= ulp / 2
    # power-of-two headroom scales T exactly
    for a in (3.0, 777.0):
        assert oracle.tensor_scale(a, headroom=16.0) == 16 * oracle.tensor_scale(a)
    # floor that keeps s * T normal
    assert oracle.tensor_scale(1e-35) == 2.0 ** -100


# ------------------------------------------------------------ quantisation
def _on_grid_tensor(rng, rows, cols, T):
    """Blocks whose values are exactly e_j * s * T with the block max equal to
    6 * s * T, so that RNE quantisation must reproduce them exactly."""
    codes = rng.integers(0x10, 0xE0, (rows, cols // 16))        # UE5M3 normal codes
    s = np.vectorize(oracle.scale_decode)(codes)
    e = E2M1[rng.integers(0, 8, (rows, cols))] * rng.choice([-1, 1], (rows, cols))
    e = e.reshape(rows, cols // 16, 16)
    e[:, :, 0] = np.where(e[:, :, 0] >= 0, 6.0, -6.0)              # block max hits 6
    x = (e * s[:, :, None] * T).reshape(rows, cols)
    return x.astype(np.float32), codes


def test_quantize_reproduces_on_grid_values_exactly():
    rng = np.random.default_rng(0)
    T = 2.0 ** -7
    x, codes = _on_grid_tensor(rng, 32, 64, T)
    p, s, st = oracle.quantize(bf16_bits(x), oracle.ROW, T)
    assert (s == codes).all()
    # no scale saturates or underflows and nothing flushes; an element equal to
    # 6 s T may count as clamped, because 1 / (s T) is rounded once before the
    # multiply and so |q| can land an ulp above 6 (it still encodes to 6)
    assert st[0] == st[1] == st[3] == 0
    assert st[2] <= (np.abs(x) == np.abs(x).reshape(32, 4, 16).max(-1).repeat(16, 1)).sum()
    f, b = oracle.dequantize(p, s, T)
    assert (f == x).all()
    assert (b == bf16_bits(x)).all()


def test_nibble_order_and_scale_position():
    # element (r, 2j) goes to the low nibble of payload[r, j]
    x = np.zeros((16, 32), np.float32)
    x[0, 0], x[0, 1] = 1.0, 2.0
    x[0, 16] = 6.0
    x[3, 5] = -6.0
    p, s, _ = oracle.quantize(bf16_bits(x), oracle.ROW, 1.0)
    # block amax 2 -> s* = 2/6 -> UE5M3 code nearest 1/3 = 0x6B (1.375 * 2^-2 = 0.34375)
    assert s[0, 0] == 0x6B
    sv = oracle.scale_decode(0x6B)
    assert p[0, 0] & 15 == int(oracle.e2m1_rne(np.float32(1.0) / np.float32(sv))[0])
    assert p[0, 0] >> 4 == int(oracle.e2m1_rne(np.float32(2.0) * (np.float32(1) / np.float32(sv)))[0])
    assert s[0, 1] == 0x78 and p[0, 8] == 0x07           # 6 / (1 * 1) -> code 7
    assert s[3, 0] == 0x78 and p[3, 2] == 0xF0           # element 5 -> high nibble, -6


def test_col_is_row_of_transpose():
    rng = np.random.default_rng(1)
    x = bf16_round(rng.standard_normal((64, 96)).astype(np.float32) * 3)
    T = oracle.tensor_scale(oracle.amax(x)[0])
    pc, sc, stc = oracle.quantize(x, oracle.COL, T)
    pr, sr, str_ = oracle.quantize(np.ascontiguousarray(x.T), oracle.ROW, T)
    assert pc.shape == (96, 32) and sc.shape == (96, 4)
    assert (pc == pr).all() and (sc == sr).all() and (stc == str_).all()


def test_sign_symmetry():
    rng = np.random.default_rng(2)
    x = bf16_round(rng.standard_normal((32, 64)).astype(np.float32))
    neg = x ^ np.uint16(0x8000)
    T = oracle.tensor_scale(oracle.amax(x)[0])
    p1, s1, _ = oracle.quantize(x, oracle.ROW, T)
    p2, s2, _ = oracle.quantize(neg, oracle.ROW, T)
    assert (s1 == s2).all()
    assert (p1 ^ 0x88 == p2).all()


def test_rne_error_bound():
    """Every non-saturated element lies within half a grid step (at its scale)
    of its reconstruction, up to binary32 rounding of the scale arithmetic."""
    rng = np.random.default_rng(3)
    xf = (rng.standard_normal((64, 256)) * np.exp(rng.standard_normal(256))).astype(np.float32)
    x = bf16_round(xf)
    xv = bits_to_f32(x).astype(np.float64)
    T = oracle.tensor_scale(oracle.amax(x)[0])
    p, s, st = oracle.quantize(x, oracle.ROW, T)
    # with no headroom the block holding the tensor amax sits on the top of
    # the scale range and may saturate by the rounding of T
    assert st[0] <= 1
    sv = np.vectorize(oracle.scale_decode)(s).repeat(16, 1) * T
    q = xv / sv
    e = nib_values(p)
    step = np.where(np.abs(q) < 2, 0.5, np.where(np.abs(q) < 4, 1.0, 2.0))
    clamp = np.abs(q) > 6
    err = np.abs(q - e)
    assert (err[~clamp] <= step[~clamp] / 2 * (1 + 2 ** -20) + 1e-12).all()
    # block amax rounds to within the grid: |q| never exceeds 6 by more than
    # the UE5M3 relative half-step
    assert (np.abs(q) <= 6 * (1 + 1 / 16) + 1e-9).all()


def test_stats_on_crafted_blocks():
    T = 1.0
    x = np.zeros((16, 64), np.float32)
    # block 0: all zero -> code 0, no stats
    # block 1: amax = 6 * 2^17 -> s* = 2^17 > 114688 -> saturates
    x[0, 16] = 6 * 2.0 ** 17
    x[0, 17] = 1.0
    # block 2: tiny -> s* < 2^-18 -> scale underflows, both nonzero values flushed
    x[0, 32] = 2.0 ** -22
    x[0, 33] = -(2.0 ** -23)
    # block 3: s* = amax/6 = 1.0625 -> rounds (tie) to code 1.0 -> 6.375 clamps
    x[0, 48] = 6.375
    x[0, 49] = 0.0625          # nonzero, flushes to 0 at scale 1
    p, s, st = oracle.quantize(bf16_bits(x), oracle.ROW, T)
    assert s[0, 0] == 0 and (p[0, 0:8] == 0).all()
    assert s[0, 1] == 0xFE
    assert s[0, 2] == 0 and p[0, 16] == 0x80
    assert s[0, 3] == 0x78 and p[0, 24] & 15 == 7
    # sat blocks, uflow blocks, clamped elements, flushed elements
    # block 1: 6*2^17 / 114688 = 6.857 clamps; 1.0/114688 flushes
    assert list(st) == [1, 1, 2, 4]


def test_sr_quantize_unbiased_and_scales_match_rne():
    rng = np.random.default_rng(4)
    x = bf16_round((rng.standard_normal((16, 64)) * 10 ** rng.uniform(-8, 2, (16, 1))).astype(np.float32))
    xv = bits_to_f32(x).astype(np.float64)
    T = oracle.tensor_scale(oracle.amax(x)[0])
    pr, sr_, _ = oracle.quantize(x, oracle.ROW, T)
    acc = np.zeros_like(xv)
    n = 400
    for seed in range(n):
        p, s, _ = oracle.quantize(x, oracle.ROW, T, rnd=oracle.SR, seed=seed)
        assert (s == sr_).all()                     # scales are never stochastic
        acc += nib_values(p)
    sv = np.vectorize(oracle.scale_decode)(sr_).repeat(16, 1) * T
    q = xv / sv
    mean = acc / n
    # unbiased: |mean - q| within 6 sigma of a Bernoulli over one grid step
    step = np.where(np.abs(q) < 2, 0.5, np.where(np.abs(q) < 4, 1.0, 2.0))
    ok = np.abs(q) <= 6
    assert (np.abs(mean - q)[ok] <= 6 * step[ok] * 0.5 / np.sqrt(n) + 1e-9).all()


def test_sr_row_and_col_axes_draw_independent_bits():
    rng = np.random.default_rng(5)
    x = bf16_round(rng.uniform(-1, 1, (64, 64)).astype(np.float32))
    T = oracle.tensor_scale(oracle.amax(x)[0])
    pr, _, _ = oracle.quantize(x, oracle.ROW, T, rnd=oracle.SR, seed=7)
    pc, _, _ = oracle.quantize(x, oracle.COL, T, rnd=oracle.SR, seed=7)
    pc2, _, _ = oracle.quantize(np.ascontiguousarray(x.T), oracle.ROW, T, rnd=oracle.SR, seed=7)
    # same tensor, different axis -> different random decisions somewhere
    assert (pc != pc2).any()
    assert (pr != pc2).any()


def test_row_band_equals_slice_of_full_tensor():
    """A band of rows quantised with its row offset gives exactly the full
    tensor's outputs for those rows (ROW) and that span of each column (COL),
    stochastic-rounding counters included (logical index r * cols + c)."""
    rng = np.random.default_rng(6)
    x = bf16_round((rng.standard_normal((96, 48)) * 10 ** rng.uniform(-3, 2, (96, 1))).astype(np.float32))
    T = oracle.tensor_scale(oracle.amax(x)[0])
    for rnd in (oracle.RNE, oracle.SR):
        fr = oracle.quantize(x, oracle.ROW, T, rnd=rnd, seed=11)
        fc = oracle.quantize(x, oracle.COL, T, rnd=rnd, seed=11)
        for r0, r1 in ((0, 16), (16, 48), (48, 96)):
            band = np.ascontiguousarray(x[r0:r1])
            br = oracle.quantize(band, oracle.ROW, T, rnd=rnd, seed=11, row_base=r0)
            bc = oracle.quantize(band, oracle.COL, T, rnd=rnd, seed=11, row_base=r0)
            assert np.array_equal(br[0], fr[0][r0:r1]) and np.array_equal(br[1], fr[1][r0:r1])
            assert np.array_equal(bc[0], fc[0][:, r0 // 2:r1 // 2])
            assert np.array_equal(bc[1], fc[1][:, r0 // 16:r1 // 16])
        if rnd == oracle.SR:
            # without the offset the band draws other random words
            b = np.ascontiguousarray(x[48:96])
            assert not np.array_equal(oracle.quantize(b, oracle.ROW, T, rnd=rnd, seed=11)[0], fr[0][48:96])


def test_periodic_scaler_refreshes_every_period():
    rng = np.random.default_rng(6)
    sc = oracle.PeriodicScaler(period=4)
    Ts = []
    amaxes = []
    for t in range(9):
        x = bf16_round((rng.standard_normal((16, 32)) * 1.3 ** t).astype(np.float32))
        sc.quantize(x)
        Ts.append(sc.T)
        amaxes.append(oracle.amax(x)[0])
    assert Ts[0] == oracle.tensor_scale(amaxes[0])
    assert Ts[1:4] == [Ts[0]] * 3
    assert Ts[4] == oracle.tensor_scale(amaxes[3])      # last observed amax
    assert Ts[8] == oracle.tensor_scale(amaxes[7])


# ------------------------------------------------------------ GEMM
def _random_quantised(rng, rows, K):
    x = bf16_round((rng.standard_normal((rows, K)) * np.exp(rng.standard_normal(K))).astype(np.float32))
    T = oracle.tensor_scale(oracle.amax(x)[0])
    p, s, _ = oracle.quantize(x, oracle.ROW, T)
    return p, s, T


@pytest.mark.parametrize("M,N,K", [(16, 16, 32), (16, 32, 64), (32, 16, 48)])
def test_gemm_matches_exact_rational_brute_force(M, N, K):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    A, As, TA = _random_quantised(rng, M, K)
    B, Bs, TB = _random_quantised(rng, N, K)
    got = oracle.gemm(A, As, TA, B, Bs, TB)
    ea, eb = nib_values(A), nib_values(B)
    sa = np.vectorize(oracle.scale_decode)(As).repeat(16, 1)
    sb = np.vectorize(oracle.scale_decode)(Bs).repeat(16, 1)
    alpha = Fraction(TA) * Fraction(TB)
    for m in range(M):
        for n in range(N):
            exact = alpha * sum(Fraction(ea[m, k]) * Fraction(sa[m, k]) *
                                Fraction(eb[n, k]) * Fraction(sb[n, k]) for k in range(K))
            assert abs(Fraction(got[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 200)


def test_gemm_transpose_sampling_and_dequant_consistency():
    rng = np.random.default_rng(9)
    A, As, TA = _random_quantised(rng, 32, 64)
    B, Bs, TB = _random_quantised(rng, 48, 64)
    C = oracle.gemm(A, As, TA, B, Bs, TB)
    Ct = oracle.gemm(B, Bs, TB, A, As, TA)
    assert np.allclose(C, Ct.T, rtol=1e-14, atol=0)
    ms = np.array([0, 31, 7]); ns = np.array([47, 0, 20])
    assert (oracle.gemm(A, As, TA, B, Bs, TB, ms=ms, ns=ns) == C[ms, ns]).all()
    # the dequantised operands reproduce the contraction
    fa, _ = oracle.dequantize(A, As, TA)
    fb, _ = oracle.dequantize(B, Bs, TB)
    ref = fa.astype(np.float64) @ fb.astype(np.float64).T
    assert np.abs(ref - C).max() <= 1e-5 * np.abs(C).max()

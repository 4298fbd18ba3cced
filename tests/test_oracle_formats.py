"""Pins of the oracle's element and scale formats against the format
definitions, by brute force over exact rationals -- never by re-typing the
oracle's own arithmetic.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (E2M1 payloads with unsigned E5M3 block scales).  The E2M1 element is
the OCP FP4 E2M1 format; UE5M3/UE4M3 are the unsigned 8-bit scale formats with
5 (4) exponent and 3 mantissa bits.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

F = Fraction


def f32(x):
    return np.float32(x)


def f32_neighbours(x):
    x = np.float32(x)
    return [np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))]


# --------------------------------------------------------------------- E2M1
E2M1_GRID = [F(0), F(1, 2), F(1), F(3, 2), F(2), F(3), F(4), F(6)]


def test_e2m1_grid_is_the_fp4_value_set():
    # The sixteen E2M1 codes decode to +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}; the
    # sign is bit 3.
    got = [F(oracle.e2m1_decode(c)) for c in range(16)]
    assert got[:8] == E2M1_GRID
    assert got[8:] == [-g for g in E2M1_GRID]
    assert np.signbit(oracle.e2m1_decode(8))   # code 8 is negative zero


def _e2m1_nearest_even(q: Fraction, neg: bool) -> int:
    """Brute force: the grid point nearest |q|, ties to the even code,
    saturating at 6; the sign bit follows q."""
    a = abs(q)
    if a >= 6:
        code = 7
    else:
        d = [abs(a - g) for g in E2M1_GRID]
        best = min(d)
        cands = [c for c in range(8) if d[c] == best]
        code = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
    return code | (8 if neg else 0)


def _e2m1_probe_points():
    pts = []
    for g in E2M1_GRID:
        pts += f32_neighbours(float(g))
    for a, b in zip(E2M1_GRID, E2M1_GRID[1:]):
        pts += f32_neighbours(float((a + b) / 2))
    pts += f32_neighbours(6.0) + [f32(7.0), f32(1e30), f32(1e-30), f32(0.0)]
    rng = np.random.default_rng(11)
    pts += list(rng.uniform(0, 7, 4000).astype(np.float32))
    pts = [p for p in pts if p >= 0]
    return np.array(pts + [-p for p in pts], np.float32)


def test_e2m1_rne_matches_brute_force_nearest_even():
    q = _e2m1_probe_points()
    got = oracle.e2m1_rne(q)
    want = [_e2m1_nearest_even(F(float(x)), bool(np.signbit(x))) for x in q]
    bad = [(float(x), int(g), w) for x, g, w in zip(q, got, want) if g != w]
    assert not bad, bad[:10]


def test_e2m1_rne_ties():
    # the seven ties of the grid and where each must go (even code)
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for t, code in ties.items():
        assert int(oracle.e2m1_rne(t)[0]) == code, t
        assert int(oracle.e2m1_rne(-t)[0]) == code | 8, -t
    assert int(oracle.e2m1_rne(-0.1)[0]) == 0x8      # sign kept on a flush to zero


# --------------------------------------------------------------------- scales
def _scale_props(fmt):
    return dict(ue5m3=(15, 0xFF, 0xFE), ue4m3=(7, 0x7F, 0x7E))["ue5m3" if fmt == oracle.UE5M3 else "ue4m3"]


@pytest.mark.parametrize("fmt", [oracle.UE5M3, oracle.UE4M3])
def test_scale_decode_structure(fmt):
    """The decode table is pinned by structure, not by its formula:
    strictly increasing over the finite codes, the NaN code is the all-ones
    pattern, uniform spacing inside each binade with 8 steps per binade,
    gradual underflow (the subnormal step equals the first binade's step),
    1.0 sits at code bias<<3, and every value has at most 4 significant bits."""
    bias, nan_code, max_code = _scale_props(fmt)
    vals = [oracle.scale_decode(c, fmt) for c in range(max_code + 1)]
    assert np.isnan(oracle.scale_decode(nan_code, fmt))
    fr = [F(v) for v in vals]
    assert fr[0] == 0
    assert all(b > a for a, b in zip(fr, fr[1:]))
    assert fr[bias << 3] == 1
    steps = [b - a for a, b in zip(fr, fr[1:])]
    # codes 0..8 are the subnormals plus the min normal: one uniform step
    assert len(set(steps[:8])) == 1
    for e in range(1, (max_code >> 3) + 1):
        lo = e << 3
        binade = steps[lo:lo + 7] if lo + 7 < len(steps) else steps[lo:]
        assert len(set(binade)) == 1, e
        assert fr[lo] * 2 == (fr[lo + 8] if lo + 8 <= max_code else fr[lo] * 2)
        assert binade[0] == fr[lo] / 8
    for v in fr[1:]:
        # at most 4 significant bits: v * 2^k is an integer < 16 for some k
        k = 0
        while (v * 2 ** k).denominator != 1:
            k += 1
        n = v * 2 ** k
        while n.numerator % 2 == 0 and n >= 16:
            n /= 2
        assert n < 16
    assert fr[-1] == (F(114688) if fmt == oracle.UE5M3 else F(448))
    assert oracle.scale_max(fmt) == float(fr[-1])


def _scale_nearest_even(x: Fraction, table):
    """Brute force: nearest finite code, ties to the even code; values above
    the largest finite value saturate to it."""
    if x > table[-1]:
        return len(table) - 1, 1
    d = [abs(x - t) for t in table]
    best = min(d)
    cands = [c for c, dd in enumerate(d) if dd == best]
    if len(cands) > 1:
        cands = [c for c in cands if c % 2 == 0]
    return cands[0], 0


@pytest.mark.parametrize("fmt", [oracle.UE5M3, oracle.UE4M3])
def test_scale_encode_matches_brute_force(fmt):
    bias, nan_code, max_code = _scale_props(fmt)
    table = [F(oracle.scale_decode(c, fmt)) for c in range(max_code + 1)]
    pts = []
    for t in table:
        pts += f32_neighbours(float(t))
    for a, b in zip(table, table[1:]):
        pts += f32_neighbours(float((a + b) / 2))
    top = float(table[-1])
    pts += [f32(top * 1.01), f32(top * 1.0625), f32(1e30), f32(float(table[1]) / 2),
            f32(float(table[1]) / 3), f32(1e-30), f32(0.0)]
    rng = np.random.default_rng(5)
    lo, hi = np.log2(float(table[1])) - 3, np.log2(top) + 2
    pts += list((2.0 ** rng.uniform(lo, hi, 20000)).astype(np.float32))
    pts = np.array([p for p in pts if p >= 0], np.float32)
    codes, sat = oracle.scale_encode(pts, fmt)
    for x, c, s in zip(pts, codes, sat):
        want, wsat = _scale_nearest_even(F(float(x)), table)
        assert (int(c), int(s)) == (want, wsat), (float(x), int(c), want)


def test_ue5m3_round_trip_all_codes():
    # encode(decode(c)) == c for all 255 finite codes; 0xFF is never produced
    for fmt, n in ((oracle.UE5M3, 255), (oracle.UE4M3, 127)):
        vals = np.array([oracle.scale_decode(c, fmt) for c in range(n)], np.float32)
        codes, sat = oracle.scale_encode(vals, fmt)
        assert list(codes) == list(range(n))
        assert not sat.any()
    codes, _ = oracle.scale_encode(np.float32([1e38, 3e5, 122880.0]), oracle.UE5M3)
    assert list(codes) == [0xFE] * 3


def test_ue5m3_range_is_wider_than_ue4m3():
    # the abstract's premise: UE5M3's dynamic range exceeds the E4M3 scale's
    r5 = oracle.scale_max(oracle.UE5M3) / oracle.scale_decode(1, oracle.UE5M3)
    r4 = oracle.scale_max(oracle.UE4M3) / oracle.scale_decode(1, oracle.UE4M3)
    assert np.log2(r5) > 33.7 and np.log2(r4) < 17.9

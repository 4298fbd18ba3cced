"""Pins of the oracle's 16 x 16 (two-dimensional) block scaling, the
transposition-invariant variant listed among the related work of "UE5M3 FP4
Block Scaling for Stable Language Model Pretraining" (Related papers:
"Stable FP4 Training via Transposition-Invariant Block Quantization").

Reading: one scale per 16 x 16 tile by the block rule applied to the tile's
amax; one quantisation per element with it; both layouts written.  The pins
tie it to the one-dimensional oracle (itself pinned elsewhere) and to the
invariants the variant exists for."""
import numpy as np
import pytest

import oracle
from fp4_block_scaled_bf16_gb300 import workloads


def _bits(shape, seed, spread=3.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    x *= (10.0 ** rng.uniform(-spread, spread, shape)).astype(np.float32)
    return workloads.f32_to_bf16_bits(x)


def _nibbles(payload):
    return np.stack([payload & 15, payload >> 4], -1).reshape(payload.shape[0], -1)


@pytest.mark.parametrize("rnd", [oracle.RNE, oracle.SR])
def test_transposition_invariance(rnd):
    """Quantising x^T gives the row and column outputs of x, swapped --
    except that SR draws its words by logical index, so only RNE is
    invariant byte for byte; SR keeps the scales invariant."""
    x = _bits((48, 80), 1)
    T = oracle.tensor_scale(oracle.amax(x)[0])
    pr, sr, pc, sc, _ = oracle.quantize_2d(x, T, rnd=rnd, seed=5)
    pr_t, sr_t, pc_t, sc_t, _ = oracle.quantize_2d(np.ascontiguousarray(x.T), T, rnd=rnd, seed=5)
    assert np.array_equal(sr, sc_t) and np.array_equal(sc, sr_t)
    if rnd == oracle.RNE:
        assert np.array_equal(pr, pc_t) and np.array_equal(pc, pr_t)


@pytest.mark.parametrize("rnd", [oracle.RNE, oracle.SR])
def test_column_layout_is_the_transpose(rnd):
    x = _bits((64, 32), 2)
    T = oracle.tensor_scale(oracle.amax(x)[0])
    pr, sr, pc, sc, _ = oracle.quantize_2d(x, T, rnd=rnd, seed=9)
    assert np.array_equal(_nibbles(pr), _nibbles(pc).T)
    # every row of a tile carries the tile's code, every column too
    for tr in range(4):
        for tc in range(2):
            code = sr[16 * tr, tc]
            assert (sr[16 * tr:16 * tr + 16, tc] == code).all()
            assert (sc[16 * tc:16 * tc + 16, tr] == code).all()


def test_scale_is_the_largest_row_block_scale():
    """The block rule is monotone in the amax, so the tile's code is the
    largest code of its sixteen one-dimensional row blocks."""
    x = _bits((64, 64), 3, spread=5.0)
    T = oracle.tensor_scale(oracle.amax(x)[0])
    _, s1, _ = oracle.quantize(x, oracle.ROW, T)
    _, s2, _, _, _ = oracle.quantize_2d(x, T)
    for tr in range(4):
        want = s1[16 * tr:16 * tr + 16].max(axis=0)
        assert np.array_equal(s2[16 * tr], want)


@pytest.mark.parametrize("rnd", [oracle.RNE, oracle.SR])
def test_reduces_to_row_wise_when_every_row_holds_the_tile_max(rnd):
    """If each row of every tile contains the tile's largest magnitude, the
    tile scale equals each row block's scale, and the 2-D quantisation must
    equal the row-wise one (same SR words: row stream) byte for byte."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((32, 48)).astype(np.float32)
    for tr in range(2):
        for tc in range(3):
            t = x[16 * tr:16 * tr + 16, 16 * tc:16 * tc + 16]
            m = np.float32(np.abs(t).max() * 1.5)
            cols = rng.integers(0, 16, 16)
            t[np.arange(16), cols] = m * np.sign(rng.standard_normal(16)).astype(np.float32)
    x = workloads.f32_to_bf16_bits(x)
    T = oracle.tensor_scale(oracle.amax(x)[0]) * np.float32(1.7)
    p1, s1, st1 = oracle.quantize(x, oracle.ROW, float(T), rnd=rnd, seed=11)
    p2, s2, _, _, st2 = oracle.quantize_2d(x, float(T), rnd=rnd, seed=11)
    assert np.array_equal(s1, s2) and np.array_equal(p1, p2)
    assert np.array_equal(st1[2:], st2[2:])


def test_closed_form_tile():
    """A tile whose amax is 6 T s for a representable scale s: the code is s's
    code and the element 6 T s encodes to 6 (0x7), half of it to 3 (0x5)."""
    T = 0.25
    s = 1.5                       # UE5M3 code 0x7c (bias 15: 2^0 * 1.5)
    x = np.zeros((16, 16), np.float32)
    x[3, 7] = 6 * T * s
    x[9, 2] = -3 * T * s
    x = workloads.f32_to_bf16_bits(x)
    pr, sr, pc, sc, st = oracle.quantize_2d(x, T)
    assert (sr == oracle.scale_encode(s)[0]).all() and (sc == sr[0, 0]).all()
    n = _nibbles(pr)
    assert n[3, 7] == 0x7 and n[9, 2] == 0x8 | 0x5
    assert n.sum() == 0x7 + 0xD
    assert list(st) == [0, 0, 0, 0]

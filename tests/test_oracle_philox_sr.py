"""Pins of the oracle's Philox generator and of E2M1 stochastic rounding.

Philox4x32-10 / 4x64-10: Salmon et al., "Parallel random numbers: as easy as
1, 2, 3" (SC 2011).  The oracle's round structure and key schedule are checked
against numpy's independent Philox4x64 bit generator, and its 32-bit variant
against Triton's Philox4x32 run in Triton's CPU interpreter.

Stochastic rounding of backward gradients ("UE5M3 FP4 Block Scaling for Stable
Language Model Pretraining", Abstract): it must be unbiased, E[round(q)] = q.
Reading (the abstract fixes no bit width): u = U * 2^-16 for a 16-bit uniform
U, round up iff u < p, so E[round(q)] is within 2^-16 of a grid step of q;
element i draws word i % 4 of Philox4x32-10 at counter (i/4, i/4 >> 32, 0, 0),
the row-wise layout its low 16 bits, the column-wise layout its high 16 bits.
"""
from fractions import Fraction
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle


def test_philox4x64_matches_numpy():
    rng = np.random.default_rng(3)
    for _ in range(8):
        key = rng.integers(0, 2**64, 2, dtype=np.uint64)
        ctr = rng.integers(0, 2**64, 4, dtype=np.uint64)
        bg = np.random.Philox(counter=ctr, key=key)
        # numpy advances the counter by one before producing a block
        got = np.array([bg.random_raw() for _ in range(4)], np.uint64)
        c1 = ctr.copy()
        c1[0] = (int(c1[0]) + 1) % 2**64
        if c1[0] == 0:
            c1[1] = (int(c1[1]) + 1) % 2**64
        want = oracle.philox4x64_10(c1, key)
        assert list(got) == list(want)


_TRITON_SCRIPT = textwrap.dedent(r"""
    import os, sys
    os.environ["TRITON_INTERPRET"] = "1"
    import numpy as np, torch, triton, triton.language as tl

    @triton.jit
    def k(out_ptr, c0p, c1p, c2p, c3p, seed, N: tl.constexpr):
        i = tl.arange(0, N)
        a, b, c, d = tl.philox(seed, tl.load(c0p + i), tl.load(c1p + i),
                               tl.load(c2p + i), tl.load(c3p + i))
        tl.store(out_ptr + 4 * i + 0, a)
        tl.store(out_ptr + 4 * i + 1, b)
        tl.store(out_ptr + 4 * i + 2, c)
        tl.store(out_ptr + 4 * i + 3, d)

    data = np.load(sys.argv[1])
    ctr, seed = data["ctr"], int(data["seed"])
    N = ctr.shape[0]
    cols = [torch.from_numpy(np.ascontiguousarray(ctr[:, j]).view(np.int32)) for j in range(4)]
    out = torch.zeros(4 * N, dtype=torch.int32)
    k[(1,)](out, *cols, seed, N=N)
    np.save(sys.argv[2], out.numpy().view(np.uint32).reshape(N, 4))
""")


def test_philox4x32_matches_triton_interpreter(tmp_path):
    pytest.importorskip("triton")
    rng = np.random.default_rng(4)
    N = 16
    ctr = rng.integers(0, 2**32, (N, 4), dtype=np.uint64).astype(np.uint32)
    ctr[0] = 0
    ctr[1] = 0xFFFFFFFF
    seed = 0x1234_5678_9ABC_DEF0
    inp, outp = tmp_path / "in.npz", tmp_path / "out.npy"
    np.savez(inp, ctr=ctr, seed=np.uint64(seed))
    script = tmp_path / "tri.py"
    script.write_text(_TRITON_SCRIPT)
    env = dict(os.environ, TRITON_INTERPRET="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, str(script), str(inp), str(outp)], env=env,
                       capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + r.stderr[-300:])
    want = np.load(outp)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    for j in range(N):
        assert list(oracle.philox4x32_10(ctr[j], key)) == list(want[j]), j


def test_sr_uniform_counter_map():
    # element i: word i % 4 of Philox((i/4, i/4 >> 32, 0, 0), seed); the
    # row-wise layout takes its low 16 bits, the column-wise its high 16
    seed = 0xDEADBEEF_00000007
    idx = np.array([0, 1, 2, 3, 4, 7, 2**33 + 5, 2**40 + 2], np.uint64)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    got0, got1 = oracle.sr_uniforms(seed, idx, 0), oracle.sr_uniforms(seed, idx, 1)
    for i, g0, g1 in zip(idx, got0, got1):
        i = int(i)
        w = int(oracle.philox4x32_10([(i >> 2) & 0xFFFFFFFF, i >> 34, 0, 0], key)[i & 3])
        assert int(g0) == w & 0xFFFF and int(g1) == w >> 16
    # the two halves behave as independent uniforms: uncorrelated, each uniform
    n = 1 << 18
    a0 = oracle.sr_uniforms(seed, np.arange(n, dtype=np.uint64), 0).astype(np.float64)
    a1 = oracle.sr_uniforms(seed, np.arange(n, dtype=np.uint64), 1).astype(np.float64)
    assert a0.max() < 2 ** 16 and a1.max() < 2 ** 16
    assert abs(np.corrcoef(a0, a1)[0, 1]) < 5 / np.sqrt(n)
    for a in (a0, a1):
        h = np.bincount((a.astype(np.int64) >> 12), minlength=16)
        assert (np.abs(h - n / 16) < 6 * np.sqrt(n / 16)).all()


E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])


def _decode(n):
    n = np.asarray(n)
    mag = E2M1[n & 7]
    return np.where(n & 8, -mag, mag)


@pytest.mark.parametrize("q", [0.1, 0.3, 0.49, 0.7, 1.2, 1.55, 1.9, 2.2, 2.9, 3.3,
                               3.999, 4.5, 5.9, -0.3, -2.6, -5.0])
def test_sr_is_unbiased_over_1e6_draws(q):
    n = 1_000_000
    rng = np.random.default_rng(abs(int(q * 1000)) + 17)
    u16 = rng.integers(0, 2**16, n, dtype=np.uint64).astype(np.uint32)
    out = _decode(oracle.e2m1_sr(np.full(n, q, np.float32), u16))
    a = abs(float(np.float32(q)))
    lo = E2M1[E2M1 <= a].max()
    hi = E2M1[E2M1 > a].min()
    p = (a - lo) / (hi - lo)
    sigma = (hi - lo) * np.sqrt(p * (1 - p) / n)
    assert set(np.unique(np.abs(out))) <= {lo, hi}
    assert abs(out.mean() - float(np.float32(q))) < 5 * sigma + 1e-12


def test_sr_unbiased_with_the_philox_stream():
    # same check, drawing the bits through the oracle's own counter map
    n = 1_000_000
    q = np.float32(2.7)
    for axis in (0, 1):
        u16 = oracle.sr_uniforms(7, np.arange(n, dtype=np.uint64), axis)
        out = _decode(oracle.e2m1_sr(np.full(n, q, np.float32), u16))
        p = (float(q) - 2.0) / 1.0
        assert abs(out.mean() - float(q)) < 5 * np.sqrt(p * (1 - p) / n)


@pytest.mark.parametrize("q", [0.0001, 0.1, 0.25, 0.3000001, 0.49999997, 0.5000001, 0.7, 0.99999994,
                               1.00000012, 1.2, 1.4999999, 1.75, 2.0000002, 2.6, 3.9999998, 4.5,
                               5.0, 5.9999995, -0.3, -4.2])
def test_sr_rounds_up_for_exactly_the_uniforms_below_p(q):
    # every one of the 2^16 uniforms: the ones that round up are exactly those
    # with U * 2^-16 < p, p the exact (rational) position of |q| between its
    # grid neighbours -- so P(up) = ceil(p 2^16) / 2^16, within 2^-16 of p
    qf = np.float32(q)
    a = abs(Fraction(float(qf)))
    grid = [Fraction(g) for g in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    lo = max(g for g in grid if g <= a)
    hi = min(g for g in grid if g > a)
    p = (a - lo) / (hi - lo)
    U = np.arange(2 ** 16, dtype=np.uint32)
    out = oracle.e2m1_sr(np.full(U.size, qf, np.float32), U)
    mag = E2M1[out & 7]
    up = mag == float(hi)
    assert ((mag == float(lo)) | up).all()
    want = np.array([Fraction(int(u), 2 ** 16) < p for u in range(2 ** 16)])
    assert np.array_equal(up, want)
    assert (out >> 3 == (1 if q < 0 else 0)).all()


def test_sr_edges():
    grid = np.float32([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for u in (0, 1, 2**15, 0xFFFF):
        # on-grid values never move, whatever the uniform
        assert list(oracle.e2m1_sr(grid, np.uint32(u))) == list(range(8))
        # at or above 6 saturates
        assert int(oracle.e2m1_sr(np.float32([7.5]), np.uint32(u))[0]) == 7
    # U = 0 rounds up whenever p > 0; U = 2^16 - 1 only when p > 1 - 2^-16
    assert int(oracle.e2m1_sr(np.float32([0.0001]), np.uint32(0))[0]) == 1
    assert int(oracle.e2m1_sr(np.float32([0.4999]), np.uint32(0xFFFF))[0]) == 0
    assert int(oracle.e2m1_sr(np.float32([0.49999997]), np.uint32(0xFFFF))[0]) == 1
    # only the low 16 bits of the argument are the uniform
    assert int(oracle.e2m1_sr(np.float32([0.25]), np.uint32(0x7FFF))[0]) == 1
    assert int(oracle.e2m1_sr(np.float32([0.25]), np.uint32(0x8000))[0]) == 0
    assert int(oracle.e2m1_sr(np.float32([0.25]), np.uint32(0xFFFF7FFF))[0]) == 1
    assert int(oracle.e2m1_sr(np.float32([0.25]), np.uint32(0x00018000))[0]) == 0
    # negative values round their magnitude and keep the sign
    assert int(oracle.e2m1_sr(np.float32([-0.0001]), np.uint32(0xFFFF))[0]) == 8

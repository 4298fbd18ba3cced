"""Seeded synthetic inputs for the five workloads, shared by the tests, the
bench and the oracle legs.

This module holds none of the method's arithmetic: it draws FP32 numbers with
numpy's PCG64 and rounds them to BF16 (round to nearest, ties to even) --
nothing else.  The shapes and value distributions stand in for the 8B-class
linear layers of the pretraining run described in "UE5M3 FP4 Block Scaling for
Stable Language Model Pretraining", Abstract (Nemotron-H 8B); no dataset or
trained weight is used.
"""
from __future__ import annotations

import numpy as np

HIDDEN = 4096
FFN = 16384
TOKENS = 8192
# the four internal linears of an 8B-class block (in_features, out_features)
LINEARS = {"qkv": (4096, 6144), "out": (4096, 4096), "up": (4096, 16384), "down": (16384, 4096)}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to BF16 (nearest, ties to even) -> uint16 patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    out = np.empty(u.shape, np.uint16)
    # process in slabs to bound the uint64 temporaries on large tensors
    flat_u, flat_o = u.reshape(-1), out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat_u.size, step):
        v = flat_u[i:i + step].astype(np.uint64)
        flat_o[i:i + step] = ((v + 0x7FFF + ((v >> 16) & 1)) >> 16).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint32) << 16).view(np.float32)


def to_torch_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _normal(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def tiny_operands(seed: int = 0, n: int = 256):
    """A, B: n x n ~ N(0, 1); entries where a separate uniform draw < 0.01 are
    multiplied by 100 (outliers)."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(2):
        x = _normal(rng, (n, n))
        mask = rng.random((n, n), dtype=np.float32) < 0.01
        x[mask] *= 100.0
        out.append(f32_to_bf16_bits(x))
    return out[0], out[1]


def activations(rows: int, cols: int, seed: int):
    """X = z * exp(g_c): z ~ N(0, 1), g_c ~ N(0, 1) per column (log-normal
    channel magnitudes, sigma = 1)."""
    rng = np.random.default_rng(seed)
    g = np.exp(_normal(rng, (1, cols)))
    x = _normal(rng, (rows, cols))
    x *= g
    return f32_to_bf16_bits(x)


def weights(rows: int, cols: int, seed: int, std: float = 0.02):
    rng = np.random.default_rng(seed)
    x = _normal(rng, (rows, cols))
    x *= np.float32(std)
    return f32_to_bf16_bits(x)


def gradients(rows: int, cols: int, seed: int, lo: float = -8.0, hi: float = 2.0):
    """dY = z * 10^u_r: z ~ N(0, 1), u_r ~ U(lo, hi) per row (per-row
    magnitudes log-uniform over 1e-8 .. 1e2)."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(lo, hi, (rows, 1)).astype(np.float32)
    x = _normal(rng, (rows, cols))
    x *= np.power(np.float32(10.0), u)
    return f32_to_bf16_bits(x)


def fprop_operands():
    """8B-class fprop linear: X 8192 x 4096 (seed 1), W 16384 x 4096 (seed 2)."""
    return activations(TOKENS, HIDDEN, 1), weights(FFN, HIDDEN, 2)


def backward_gradient():
    """dY 8192 x 16384 (seed 3)."""
    return gradients(TOKENS, FFN, 3)


def drift_amaxes(steps: int = 64, factor: float = 1.3, seed: int = 99, mode: str = "walk"):
    """Target amax per step: a_0 = 1 and a_t = a_{t-1} * factor^(+-1) with a
    fair random sign ("walk"), or a_t = factor^t ("monotone")."""
    if mode == "monotone":
        return [float(np.float32(factor) ** t) for t in range(steps)]
    rng = np.random.default_rng(seed)
    signs = rng.choice([-1, 1], steps)
    a = [1.0]
    for t in range(1, steps):
        a.append(a[-1] * factor ** int(signs[t]))
    return a


def drift_tensor(t: int, target_amax: float, n: int = 4096, flip_seed: int | None = None):
    """Step t of the drifting sequence: N(0, 1) (seed 100 + t) rescaled so
    that max |x| equals the target (before BF16 rounding); with flip_seed,
    element signs are flipped at random."""
    rng = np.random.default_rng(100 + t)
    x = _normal(rng, (n, n))
    x *= np.float32(target_amax) / np.abs(x).max()
    if flip_seed is not None:
        f = np.random.default_rng(flip_seed + t).random((n, n), dtype=np.float32) < 0.5
        x[f] = -x[f]
    return f32_to_bf16_bits(x)


def linear_block(name: str, tokens: int = TOKENS):
    """Inputs of one internal linear (in -> out) of the 8B-class block:
    X [tokens, in], W [out, in], dY [tokens, out], seeds 10+l, 20+l, 30+l."""
    l = list(LINEARS).index(name)
    fin, fout = LINEARS[name]
    return (activations(tokens, fin, 10 + l), weights(fout, fin, 20 + l),
            gradients(tokens, fout, 30 + l))

"""Shrinkage-bias diagnostic (the non-uniform E2M1 grid rounds magnitudes
toward zero on average; "Rethinking shrinkage bias in LLM FP4 pretraining",
summary, and the UE5M3 recipe's stochastic rounding of gradients in "UE5M3 FP4
Block Scaling for Stable Language Model Pretraining", Abstract).  On the
gradient distribution, RNE's mean signed magnitude error relative to the
magnitude is negative, while stochastic rounding's is zero within its
sampling error."""
import numpy as np

import oracle
from fp4_block_scaled_bf16_gb300 import workloads

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])


def _mags(payload):
    n = np.stack([payload & 15, payload >> 4], -1).reshape(payload.shape[0], -1)
    return E2M1[n & 7]


def test_rne_shrinks_sr_does_not():
    x = workloads.gradients(64, 1024, 3)
    xv = workloads.bf16_bits_to_f32(x).astype(np.float64)
    T = oracle.tensor_scale(oracle.amax(x)[0])
    p, s, _ = oracle.quantize(x, oracle.ROW, T)
    sv = np.vectorize(oracle.scale_decode)(s).repeat(16, 1) * T
    q = np.abs(xv) / sv
    ok = (q <= 6) & (q > 0)
    rel_rne = ((_mags(p) - q)[ok]).sum() / q[ok].sum()
    acc = np.zeros_like(q)
    n = 64
    for seed in range(n):
        ps, _, _ = oracle.quantize(x, oracle.ROW, T, rnd=oracle.SR, seed=seed)
        acc += _mags(ps)
    rel_sr = ((acc / n - q)[ok]).sum() / q[ok].sum()
    assert rel_rne < -1e-3            # systematic shrinkage under RNE
    assert abs(rel_sr) < 2e-3         # no systematic bias under SR
    assert abs(rel_sr) < abs(rel_rne) / 3

"""GPU parity of the 16 x 16 (transposition-invariant) block scaling against
the oracle, bit-exact: both payload layouts, both scale layouts, the counts
and the fused amax, RNE and stochastic rounding, UE5M3 and UE4M3, small
ragged sizes, edge values and the full 8B-class sizes; and a GEMM on such
operands.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Related papers ("Stable FP4 Training via Transposition-Invariant Block
Quantization": one scale per 2-D block, shared by the forward and the
transposed backward operand)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import GEMM_TOL, gemm_error, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    yield fp4q
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def rand_bits(shape, seed, spread=3.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    x *= (10.0 ** rng.uniform(-spread, spread, (shape[0], 1))).astype(np.float32)
    return workloads.f32_to_bf16_bits(x)


def check_2d(lib, bits, fmt=0, rnd=0, seed=0, T=None):
    x = to_dev(bits)
    if T is None:
        T_dev = lib.tensor_scale(lib.amax(x), fmt)
        T = float(T_dev.item())
    else:
        T_dev = torch.tensor([T], dtype=torch.float32, device="cuda")
        T = float(np.float32(T))
    q = lib.quantize(x, lib.AXIS_BOTH_2D, T_dev, fmt, rnd, seed, stats=True, want_amax=True)
    torch.cuda.synchronize()
    want = oracle.quantize_2d(bits, T, fmt, rnd, seed)
    got = [t.cpu().numpy() for t in (q.payload_row, q.scales_row, q.payload_col, q.scales_col)]
    for name, g, w in zip(("payload_row", "scales_row", "payload_col", "scales_col"), got, want[:4]):
        if not np.array_equal(g, w):
            bad = np.argwhere(g != w)
            raise AssertionError(f"{name}: {len(bad)} bytes differ, first {bad[:4].tolist()}")
    assert np.array_equal(q.stats.cpu().numpy()[0].astype(np.uint64), want[4])
    assert float(q.amax.item()) == oracle.amax(bits)[0]
    return q, want, T


@pytest.mark.parametrize("shape", [(16, 16), (48, 80), (128, 128), (272, 400), (144, 272), (384, 128)])
@pytest.mark.parametrize("rnd", [0, 1])
def test_small_and_ragged(lib, shape, rnd):
    check_2d(lib, rand_bits(shape, sum(shape) + rnd), rnd=rnd, seed=77)


@pytest.mark.parametrize("rnd", [0, 1])
def test_ue4m3_and_stale_scales(lib, rnd):
    bits = rand_bits((144, 272), 5, spread=5.0)
    check_2d(lib, bits, fmt=1, rnd=rnd, seed=3)
    for T in (1e-9, 1.0, 1e4):
        check_2d(lib, bits, rnd=rnd, seed=3, T=T)


def test_edge_values(lib):
    x = np.zeros((64, 64), np.float32)
    x[1, :16] = -0.0
    x[2, :16] = np.float32(2.0 ** -130)
    x[3, 0], x[3, 1] = 3e38, -3e38
    x[5, :16] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, 6.0, -6.0]
    x[16:, :] = np.random.default_rng(0).standard_normal((48, 64)).astype(np.float32)
    bits = workloads.f32_to_bf16_bits(x)
    bits[1, :16] = 0x8000
    for T in (None, 1.0, 1e-3, 2.0 ** -100):
        check_2d(lib, bits, T=T)
        check_2d(lib, bits, T=T, rnd=1, seed=4)


def test_full_size_weight_and_gradient(lib):
    _, W = workloads.fprop_operands()
    check_2d(lib, W)
    check_2d(lib, workloads.backward_gradient(), rnd=1, seed=7)


def test_gemm_on_2d_operands(lib):
    """C = A B^T with A the row layout of an SR-quantised gradient and B the
    column layout of a weight, both from 16 x 16 scaling, against the
    oracle's binary64 contraction of the same operands."""
    d = rand_bits((256, 512), 8)                          # A: rows of d, K = 512
    wt = rand_bits((512, 192), 10, spread=1.0)            # B: column layout of wt, K = 512
    qa = lib.quantize(to_dev(d), lib.AXIS_BOTH_2D, None, 0, 1, 7)
    qb = lib.quantize(to_dev(wt), lib.AXIS_BOTH_2D)
    C = lib.gemm(qa.payload_row, qa.scales_row, qa.T, qb.payload_col, qb.scales_col, qb.T,
                 dtype=torch.float32)
    torch.cuda.synchronize()
    pa, sa = qa.payload_row.cpu().numpy(), qa.scales_row.cpu().numpy()
    pb, sb = qb.payload_col.cpu().numpy(), qb.scales_col.cpu().numpy()
    R = oracle.gemm(pa, sa, float(qa.T.item()), pb, sb, float(qb.T.item()))
    assert gemm_error(C.cpu().numpy(), R) <= GEMM_TOL

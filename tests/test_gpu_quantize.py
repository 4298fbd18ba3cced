"""GPU parity of the quantisation path against the oracle, bit-exact:
amax, tensor scale, payload bytes, scale bytes, saturation/underflow counts
and the fused amax, for row-wise, column-wise and dual-axis blocking, RNE and
stochastic rounding, UE5M3 and UE4M3, at small ragged sizes, edge cases and
the full 8B-class sizes.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (E2M1 + UE5M3 block-16, periodic tensor scaling, stochastic rounding
on backward gradients)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import check_quantize, to_dev

pytestmark = pytest.mark.gpu

ROW, COL, BOTH = 0, 1, 2


def rand_bits(shape, seed, scale=1.0, spread=0.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32) * np.float32(scale)
    if spread:
        x *= (10.0 ** rng.uniform(-spread, spread, (shape[0], 1))).astype(np.float32)
    return workloads.f32_to_bf16_bits(x)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    yield fp4q
    assert fp4q.fp4q_get_device_status() == fp4q.OK


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 4096, 1000003])
def test_amax(n, lib):
    bits = rand_bits((1, max(n, 1)), n)[0][:n]
    x = workloads.to_torch_bf16(bits).cuda() if n else torch.empty(0, dtype=torch.bfloat16, device="cuda")
    a = lib.amax(x)
    assert float(a.item()) == oracle.amax(bits)[0]


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("headroom", [1.0, 16.0, 256.0])
def test_tensor_scale(fmt, headroom, lib):
    for amax in [0.0, 1e-38, 1e-30, 3.5, 688128.0, 3e38, 1.7e-5]:
        a = torch.tensor([amax], dtype=torch.float32, device="cuda")
        T = lib.tensor_scale(a, fmt, headroom)
        assert float(T.item()) == oracle.tensor_scale(float(np.float32(amax)), fmt, headroom), amax


SHAPES = [(16, 16), (48, 80), (256, 256), (272, 400), (128, 128), (144, 272), (384, 128)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("axis", [ROW, COL, BOTH])
@pytest.mark.parametrize("rnd", [0, 1])
def test_quantize_parity_small(shape, axis, rnd):
    bits = rand_bits(shape, hash((shape, axis, rnd)) % 1000, scale=3.0, spread=3.0)
    check_quantize(bits, axis, fmt=0, rnd=rnd, seed=1234567 + rnd)


@pytest.mark.parametrize("axis", [ROW, COL, BOTH])
@pytest.mark.parametrize("rnd", [0, 1])
def test_quantize_ue4m3(axis, rnd):
    bits = rand_bits((144, 272), 5, spread=4.0)
    check_quantize(bits, axis, fmt=1, rnd=rnd, seed=99)


def test_tiny_config_operands():
    a, b = workloads.tiny_operands(seed=0)
    for bits in (a, b):
        check_quantize(bits, ROW)
        check_quantize(bits, BOTH, rnd=1, seed=7)


@pytest.mark.parametrize("axis", [ROW, BOTH])
def test_edge_values(axis):
    x = np.zeros((64, 64), np.float32)
    x[0, :16] = 0.0                                    # all-zero block
    x[1, :16] = -0.0                                   # negative zeros
    x[2, :16] = np.float32(2.0 ** -130)                # BF16 subnormals
    x[3, 0], x[3, 1] = 3e38, -3e38                     # near BF16 max
    x[4, :16] = np.linspace(-6, 6, 16)                 # on-grid-ish
    x[5, :16] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0,
                 6.0, -6.0]                            # E2M1 ties at scale 1
    x[6, :16] = 1e-20
    x[6, 0] = 1.0                                      # block with huge internal range
    x[7:, :] = np.random.default_rng(0).standard_normal((57, 64)).astype(np.float32)
    bits = workloads.f32_to_bf16_bits(x)
    bits[1, :16] = 0x8000
    for T in (None, 1.0, 1e-3, 1e3, 2.0 ** -100):
        check_quantize(bits, axis, T=T)
        check_quantize(bits, axis, T=T, rnd=1, seed=3)


def test_saturation_and_underflow_counts():
    # a stale (too small / too large) tensor scale, as periodic scaling can
    # produce, must count saturated and underflowed blocks identically
    bits = rand_bits((256, 256), 11, spread=6.0)
    for T in (1e-9, 1e-6, 1.0, 1e4):
        out, _, _ = check_quantize(bits, BOTH, T=T)
        st = out[ROW][2]
        if T == 1e-9:
            assert st[0] > 0
        if T == 1e4:
            assert st[1] > 0


def test_empty_inputs(lib):
    for shape in [(0, 16), (16, 0), (0, 0)]:
        x = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        T = torch.ones(1, dtype=torch.float32, device="cuda")
        q = lib.quantize(x, BOTH, T, stats=True, want_amax=True)
        torch.cuda.synchronize()
        assert int(q.stats.abs().sum().item()) == 0 and float(q.amax.item()) == 0.0


def test_sr_seed_changes_bits_but_not_scales():
    bits = rand_bits((128, 256), 3)
    o1, _, _ = check_quantize(bits, ROW, rnd=1, seed=1)
    o2, _, _ = check_quantize(bits, ROW, rnd=1, seed=2)
    assert (o1[ROW][1] == o2[ROW][1]).all()
    assert (o1[ROW][0] != o2[ROW][0]).any()


@pytest.mark.parametrize("f32", [False, True])
@pytest.mark.parametrize("fmt", [0, 1])
def test_dequantize_parity(f32, fmt, lib):
    bits = rand_bits((272, 400), 8, spread=3.0)
    out, T, q = check_quantize(bits, ROW, fmt=fmt)
    p, s, _ = out[ROW]
    d = lib.dequantize(q.payload_row, q.scales_row, q.T, fmt,
                       dtype=torch.float32 if f32 else torch.bfloat16)
    torch.cuda.synchronize()
    of, ob = oracle.dequantize(p, s, T, fmt)
    if f32:
        assert np.array_equal(d.cpu().numpy().view(np.uint32), of.view(np.uint32))
    else:
        assert np.array_equal(d.cpu().view(torch.int16).numpy().view(np.uint16), ob)


def test_dequantize_empty_and_spans(lib):
    # empty; and sizes around the kernel's 128-word warp spans (ragged tails)
    T = torch.ones(1, dtype=torch.float32, device="cuda")
    for shape in [(0, 16), (16, 0)]:
        p = torch.empty((shape[0], shape[1] // 2), dtype=torch.uint8, device="cuda")
        s = torch.empty((shape[0], shape[1] // 16), dtype=torch.uint8, device="cuda")
        assert lib.dequantize(p, s, T).numel() == 0
    for shape in [(16, 16), (16, 2048), (16, 2064), (48, 1024 + 16), (1040, 1024)]:
        bits = rand_bits(shape, shape[1], spread=3.0)
        out, Tq, q = check_quantize(bits, ROW)
        d = lib.dequantize(q.payload_row, q.scales_row, q.T)
        torch.cuda.synchronize()
        _, ob = oracle.dequantize(out[ROW][0], out[ROW][1], Tq)
        assert np.array_equal(d.cpu().view(torch.int16).numpy().view(np.uint16), ob), shape


# ---------------------------------------------------------------- full sizes
def test_full_fprop_operands_row_rne():
    X, W = workloads.fprop_operands()
    check_quantize(X, ROW)
    check_quantize(W, ROW)


def test_full_backward_operands():
    X, W = workloads.fprop_operands()
    dY = workloads.backward_gradient()
    check_quantize(dY, BOTH, rnd=1, seed=7)      # SR gradient, both blockings
    check_quantize(W, COL)                      # dgrad B operand
    check_quantize(X, COL)                      # wgrad B operand


def test_dequantize_full_size(lib):
    """W's row payload (16384 x 4096) to BF16 and dY's SR column payload
    (16384 x 8192) to binary32, bit for bit against the oracle."""
    X, W = workloads.fprop_operands()
    for bits, axis, rnd, f32 in ((W, ROW, 0, False), (workloads.backward_gradient(), COL, 1, True)):
        x = to_dev(bits)
        q = lib.quantize(x, axis, None, 0, rnd, 7)
        pay, sc = (q.payload_row, q.scales_row) if axis == ROW else (q.payload_col, q.scales_col)
        d = lib.dequantize(pay, sc, q.T, dtype=torch.float32 if f32 else torch.bfloat16)
        torch.cuda.synchronize()
        of, ob = oracle.dequantize(pay.cpu().numpy(), sc.cpu().numpy(), float(q.T.item()))
        if f32:
            assert np.array_equal(d.cpu().numpy().view(np.uint32), of.view(np.uint32))
        else:
            assert np.array_equal(d.cpu().view(torch.int16).numpy().view(np.uint16), ob)
        del x, q, d


def test_periodic_scaling_sequence(lib):
    """64 steps of a 4096 x 4096 tensor whose amax drifts by x1.3 per step
    (random direction), tensor scale refreshed every 16 steps from the last
    observed amax; every step's payload and scale bytes and counts, for UE5M3
    and UE4M3, equal the oracle's."""
    amaxes = workloads.drift_amaxes(64)
    for fmt in (0, 1):
        ref = oracle.PeriodicScaler(period=16, fmt=fmt)
        last = torch.zeros(1, dtype=torch.float32, device="cuda")
        T = torch.zeros(1, dtype=torch.float32, device="cuda")
        for t in range(64):
            bits = workloads.drift_tensor(t, amaxes[t])
            x = to_dev(bits)
            if t == 0:
                lib.fp4q_amax(x, last)
            if t % 16 == 0:
                lib.fp4q_tensor_scale(last, fmt, 1.0, T)
            q = lib.quantize(x, ROW, T, fmt, stats=True, want_amax=True)
            last = q.amax
            p, s, st = ref.quantize(bits)
            torch.cuda.synchronize()
            assert float(T.item()) == ref.T, t
            assert np.array_equal(q.payload_row.cpu().numpy(), p), t
            assert np.array_equal(q.scales_row.cpu().numpy(), s), t
            assert np.array_equal(q.stats.cpu().numpy()[0].astype(np.uint64), st), t


def test_tile_pipeline_is_deterministic(lib):
    """The persistent tile quantiser's double-buffered column stage (and the
    prefetched next piece) must never be overwritten while still being read:
    repeated full-size dual-axis quantisations are byte-identical."""
    dY = workloads.backward_gradient()
    x = to_dev(dY)
    T = lib.tensor_scale(lib.amax(x))
    ref = lib.quantize(x, BOTH, T, rnd=1, seed=7)
    refr = lib.quantize(x, BOTH, T, rnd=0)
    for _ in range(6):
        q = lib.quantize(x, BOTH, T, rnd=1, seed=7)
        r = lib.quantize(x, BOTH, T, rnd=0)
        for a, b in ((q, ref), (r, refr)):
            assert torch.equal(a.payload_row, b.payload_row)
            assert torch.equal(a.payload_col, b.payload_col)
            assert torch.equal(a.scales_col, b.scales_col)

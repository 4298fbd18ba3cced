"""Failure detection on the GPU without faulting it: a GEMM whose operand loads
are withheld must give up its bounded pipeline waits, latch FP4Q_ERR_TIMEOUT
in the device status word and exit, leaving the context usable; a non-finite
input must latch FP4Q_ERR_NONFINITE.  Nothing here traps, faults or hangs."""
import numpy as np
import pytest
import torch

from fp4_block_scaled_bf16_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    assert fp4q.fp4q_get_device_status() in (fp4q.OK, fp4q.ERR_TIMEOUT, fp4q.ERR_NONFINITE)
    return fp4q


def _operands(lib, M=256, N=256, K=256):
    rng = np.random.default_rng(0)
    a = workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    b = workloads.f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    qa = lib.quantize(workloads.to_torch_bf16(a).cuda())
    qb = lib.quantize(workloads.to_torch_bf16(b).cuda())
    return (qa.payload_row, qa.scales_row, qa.T), (qb.payload_row, qb.scales_row, qb.T)


def test_gemm_wait_timeout_is_reported_and_context_survives(lib, monkeypatch):
    A, B = _operands(lib)
    ref = lib.gemm(*A, *B, dtype=torch.float32)
    torch.cuda.synchronize()
    assert lib.fp4q_get_device_status() == lib.OK
    monkeypatch.setenv("FP4Q_TEST_GEMM_SKIP_LOADS", "1")
    monkeypatch.setenv("FP4Q_TEST_GEMM_WAIT_CYCLES", "2000000")     # about 1 ms
    lib.gemm(*A, *B, dtype=torch.float32)
    assert lib.fp4q_get_device_status() == lib.ERR_TIMEOUT
    assert lib.fp4q_get_device_status() == lib.OK                   # read clears it
    monkeypatch.delenv("FP4Q_TEST_GEMM_SKIP_LOADS")
    monkeypatch.delenv("FP4Q_TEST_GEMM_WAIT_CYCLES")
    again = lib.gemm(*A, *B, dtype=torch.float32)
    torch.cuda.synchronize()
    assert lib.fp4q_get_device_status() == lib.OK
    assert torch.equal(again, ref)


def test_native_gemm_wait_timeout_is_reported_and_context_survives(lib, monkeypatch):
    """The native NVFP4 GEMM (persistent CTA pairs): with the operand loads
    withheld every wait of both CTAs runs out, the kernel winds down (no
    load or MMA in flight, both CTAs through the cluster barrier before
    TMEM is freed) and reports FP4Q_ERR_TIMEOUT; the next call is exact."""
    rng = np.random.default_rng(9)
    M, N, K = 512, 768, 512
    a = workloads.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    b = workloads.f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    qa = lib.quantize(workloads.to_torch_bf16(a).cuda(), fmt=lib.UE4M3)
    qb = lib.quantize(workloads.to_torch_bf16(b).cuda(), fmt=lib.UE4M3)
    A, B = (qa.payload_row, qa.scales_row, qa.T), (qb.payload_row, qb.scales_row, qb.T)
    ref = lib.gemm_nvfp4(*A, *B, dtype=torch.float32)
    torch.cuda.synchronize()
    assert lib.fp4q_get_device_status() == lib.OK
    monkeypatch.setenv("FP4Q_TEST_GEMM_SKIP_LOADS", "1")
    monkeypatch.setenv("FP4Q_TEST_GEMM_WAIT_CYCLES", "2000000")     # about 1 ms
    lib.gemm_nvfp4(*A, *B, dtype=torch.float32)
    assert lib.fp4q_get_device_status() == lib.ERR_TIMEOUT
    assert lib.fp4q_get_device_status() == lib.OK
    monkeypatch.delenv("FP4Q_TEST_GEMM_SKIP_LOADS")
    monkeypatch.delenv("FP4Q_TEST_GEMM_WAIT_CYCLES")
    again = lib.gemm_nvfp4(*A, *B, dtype=torch.float32)
    torch.cuda.synchronize()
    assert lib.fp4q_get_device_status() == lib.OK
    assert torch.equal(again, ref)


def test_nonfinite_input_is_reported(lib):
    x = torch.randn(64, 64, device="cuda").to(torch.bfloat16)
    x[3, 7] = float("inf")
    lib.amax(x)
    assert lib.fp4q_get_device_status() == lib.ERR_NONFINITE
    x[3, 7] = float("nan")
    T = torch.ones(1, device="cuda")
    lib.quantize(x, lib.AXIS_BOTH, T)
    assert lib.fp4q_get_device_status() == lib.ERR_NONFINITE
    x[3, 7] = 1.0
    lib.quantize(x, lib.AXIS_BOTH, T)
    assert lib.fp4q_get_device_status() == lib.OK


def test_status_is_read_in_the_order_of_the_given_stream(lib):
    # a condition latched by work on a side stream is reported by a read on
    # that stream (which waits for that stream only), and the read clears it
    x = torch.randn(64, 64, device="cuda").to(torch.bfloat16)
    x[5, 9] = float("-inf")
    out = torch.empty(1, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        lib.fp4q_amax(x, out)
    assert lib.fp4q_get_device_status(side) == lib.ERR_NONFINITE
    assert lib.fp4q_get_device_status(side) == lib.OK
    assert lib.fp4q_get_device_status() == lib.OK

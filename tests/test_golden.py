"""Stored oracle outputs (tests/golden/oracle_snapshot.txt, written by
tests/golden/make_golden.py from the CPU oracle alone) for the tiny
configuration: the oracle must still reproduce them exactly (a change of its
arithmetic shows up here), and the CUDA path must match the stored bytes,
counts and tensor scales without the oracle running.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (E2M1 + UE5M3 block-16 quantisation, SR on gradients, FP4 GEMMs)."""
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))
import make_golden  # noqa: E402

from parity_util import GEMM_TOL  # noqa: E402


def test_oracle_reproduces_snapshot():
    stored = make_golden.parse()
    fresh = {}
    for line in make_golden.snapshot():
        kind, name, *fields = line.split()
        fresh[(kind, name)] = dict(fv.split("=", 1) for fv in fields)
    assert fresh == stored


@pytest.mark.gpu
def test_cuda_path_matches_snapshot():
    import torch
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    from parity_util import to_dev
    stored = make_golden.parse()
    for name, x, axis, rnd, fmt, seed in make_golden.cases():
        want = stored[("quantize", name)]
        q = fp4q.quantize(to_dev(x), axis, None, fmt, rnd, seed, stats=True)
        torch.cuda.synchronize()
        pay, sc = (q.payload_row, q.scales_row) if axis == 0 else (q.payload_col, q.scales_col)
        assert float(q.T.item()) == float.fromhex(want["T"]), name
        assert make_golden.h(pay.cpu().numpy()) == want["payload"], name
        assert make_golden.h(sc.cpu().numpy()) == want["scales"], name
        assert ",".join(str(int(v)) for v in q.stats.cpu().numpy()[0]) == want["stats"], name
    a, b = make_golden.workloads.tiny_operands(seed=0)
    for fmt in (0, 1):
        want = stored[("gemm", f"tiny_fmt{fmt}")]
        qa, qb = fp4q.quantize(to_dev(a), 0, None, fmt), fp4q.quantize(to_dev(b), 0, None, fmt)
        C = fp4q.gemm(qa.payload_row, qa.scales_row, qa.T, qb.payload_row, qb.scales_row, qb.T, fmt,
                      dtype=torch.float32).cpu().numpy().astype(np.float64)
        scale = float.fromhex(want["absmax"])
        assert abs(np.abs(C).max() - scale) <= GEMM_TOL * scale
        assert abs(C[0, 0] - float.fromhex(want["r00"])) <= GEMM_TOL * scale
        assert abs(C[-1, -1] - float.fromhex(want["r_last"])) <= GEMM_TOL * scale
        # the sum of 65536 entries: each within 1e-3 * scale, so the sum within 65536 times that
        assert abs(C.sum() - float.fromhex(want["sum"])) <= C.size * GEMM_TOL * scale
    assert fp4q.fp4q_get_device_status() == fp4q.OK

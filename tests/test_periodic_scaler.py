"""The package's periodic tensor-scale policy (fp4_block_scaled_bf16_gb300.
periodic.PeriodicScaler): its schedule and state, checked on CPU against the
oracle's PeriodicScaler through a stand-in library whose every call is the
oracle's; on GPU the same sequence through libfp4q.so, bit for bit.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (periodic tensor scaling, possible because of UE5M3's range)."""
import types

import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from fp4_block_scaled_bf16_gb300.periodic import PeriodicScaler


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_lib():
    """The binding's interface with the oracle behind it (CPU tensors)."""
    def fp4q_amax(x, out):
        out[0] = oracle.amax(_bits(x))[0]

    def fp4q_tensor_scale(a, fmt, headroom, out):
        out[0] = oracle.tensor_scale(float(a[0]), fmt, headroom)

    def quantize(x, axis, T, fmt, rnd, seed, stats=False, want_amax=False):
        b = _bits(x)
        p, s, st = oracle.quantize(b, axis, float(T[0]), fmt, rnd, seed)
        return types.SimpleNamespace(payload_row=torch.from_numpy(p), scales_row=torch.from_numpy(s),
                                     stats=torch.from_numpy(st.astype(np.int64))[None], T=T,
                                     amax=torch.tensor([oracle.amax(b)[0]], dtype=torch.float32))
    return types.SimpleNamespace(fp4q_amax=fp4q_amax, fp4q_tensor_scale=fp4q_tensor_scale, quantize=quantize)


def drift_inputs(steps, n=64):
    amaxes = workloads.drift_amaxes(steps)
    return [workloads.to_torch_bf16(workloads.drift_tensor(t, amaxes[t], n)) for t in range(steps)]


@pytest.mark.parametrize("fmt,headroom", [(0, 1.0), (0, 16.0), (1, 1.0)])
def test_schedule_matches_oracle_scaler(fmt, headroom):
    xs = drift_inputs(40)
    ours = PeriodicScaler(period=16, fmt=fmt, headroom=headroom, device="cpu", lib=oracle_lib())
    ref = oracle.PeriodicScaler(period=16, fmt=fmt, headroom=headroom)
    Ts = []
    for t, x in enumerate(xs):
        q = ours.quantize(x)
        p, s, st = ref.quantize(_bits(x))
        assert float(q.T[0]) == ref.T, t
        assert np.array_equal(q.payload_row.numpy(), p) and np.array_equal(q.scales_row.numpy(), s)
        Ts.append(float(q.T[0]))
    # refreshed on steps 0, 16, 32 only
    for t in range(1, len(Ts)):
        if t % 16:
            assert Ts[t] == Ts[t - 1]


def test_returned_scale_is_a_snapshot():
    xs = drift_inputs(18)
    sc = PeriodicScaler(period=16, device="cpu", lib=oracle_lib())
    qs = [sc.quantize(x) for x in xs]
    assert float(qs[0].T[0]) == float(qs[15].T[0])
    assert float(qs[0].T[0]) != float(qs[16].T[0])     # the step-16 refresh left step 0's copy alone


def test_state_round_trip_resumes_identically():
    xs = drift_inputs(40)
    full = PeriodicScaler(period=16, device="cpu", lib=oracle_lib())
    t_full = [float(full.quantize(x).T[0]) for x in xs]
    first = PeriodicScaler(period=16, device="cpu", lib=oracle_lib())
    t_first = [float(first.quantize(x).T[0]) for x in xs[:21]]
    state = first.state_dict()
    resumed = PeriodicScaler(period=16, device="cpu", lib=oracle_lib())
    resumed.load_state_dict(state)
    t_rest = [float(resumed.quantize(x).T[0]) for x in xs[21:]]
    assert t_first + t_rest == t_full
    with pytest.raises(ValueError):
        PeriodicScaler(period=8, device="cpu", lib=oracle_lib()).load_state_dict(state)


@pytest.mark.gpu
def test_gpu_scaler_matches_oracle_scaler():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    xs = drift_inputs(34, n=256)
    ours = PeriodicScaler(period=16)
    ref = oracle.PeriodicScaler(period=16)
    for t, x in enumerate(xs):
        q = ours.quantize(x.cuda(), stats=True)
        p, s, st = ref.quantize(_bits(x))
        torch.cuda.synchronize()
        assert float(q.T.item()) == ref.T, t
        assert np.array_equal(q.payload_row.cpu().numpy(), p), t
        assert np.array_equal(q.scales_row.cpu().numpy(), s), t
        assert np.array_equal(q.stats.cpu().numpy()[0].astype(np.uint64), st), t
    state = ours.state_dict()
    again = PeriodicScaler(period=16)
    again.load_state_dict(state)
    assert again.state_dict() == state
    assert fp4q.fp4q_get_device_status() == fp4q.OK


@pytest.mark.parametrize("mode", ["walk", "monotone"])
def test_periodic_report_counts_match_oracle(mode):
    from fp4_block_scaled_bf16_gb300 import periodic_report
    steps, period, n = 20, 8, 64
    res = periodic_report.run(mode, steps=steps, period=period, n=n, device="cpu", lib=oracle_lib())
    amaxes = workloads.drift_amaxes(steps, mode=mode)
    for key, fmt, h in (("UE5M3_H1", 0, 1.0), ("UE5M3_H16", 0, 16.0), ("UE5M3_H256", 0, 256.0),
                        ("UE4M3_H1", 1, 1.0)):
        ref = oracle.PeriodicScaler(period=period, fmt=fmt, headroom=h)
        for t in range(steps):
            _, _, st = ref.quantize(workloads.drift_tensor(t, amaxes[t], n))
            row = res[key][t]
            assert row["T"] == ref.T
            assert [row["scale_sat_blocks"], row["scale_uflow_blocks"], row["elem_clamped"],
                    row["elem_flushed"]] == [int(v) for v in st], (key, t)

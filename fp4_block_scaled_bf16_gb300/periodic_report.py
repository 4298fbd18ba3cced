"""Periodic tensor scaling report: per-step saturation and underflow counts
of UE5M3 block scales next to the UE4M3 scale of the TE NVFP4 recipe.

Workload: 64 steps of a 4096 x 4096 BF16 tensor whose amax drifts by x1.3 per
step in a seeded random direction; the tensor scale is refreshed every 16
steps from the last observed amax ("UE5M3 FP4 Block Scaling for Stable
Language Model Pretraining", Abstract: the wider UE5M3 range permits periodic
rather than current tensor scaling).  Everything runs through libfp4q.so.

  python -m fp4_block_scaled_bf16_gb300.periodic_report [--mode walk|monotone] [--json]
"""
from __future__ import annotations

import argparse
import json

from . import fp4q, workloads
from .periodic import PeriodicScaler


def run(mode: str = "walk", steps: int = 64, period: int = 16, n: int = 4096, device: str = "cuda",
        lib=None):
    """Per-step counts of every variant.  `lib` replaces the binding (tests
    run the schedule through a stand-in on `device`)."""
    amaxes = workloads.drift_amaxes(steps, mode=mode)
    variants = [("UE5M3", fp4q.UE5M3, 1.0), ("UE5M3", fp4q.UE5M3, 16.0), ("UE5M3", fp4q.UE5M3, 256.0),
                ("UE4M3", fp4q.UE4M3, 1.0)]
    out = {f"{name}_H{int(h)}": [] for name, _, h in variants}
    scalers = {f"{name}_H{int(h)}": PeriodicScaler(period, fmt, h, device=device, lib=lib)
               for name, fmt, h in variants}
    for t in range(steps):
        x = workloads.to_torch_bf16(workloads.drift_tensor(t, amaxes[t], n)).to(device)
        for key, sc in scalers.items():
            q = sc.quantize(x, fp4q.AXIS_ROW, stats=True)
            st = q.stats[0].tolist()
            out[key].append({"step": t, "amax": amaxes[t], "T": float(q.T.item()),
                             "scale_sat_blocks": st[0], "scale_uflow_blocks": st[1],
                             "elem_clamped": st[2], "elem_flushed": st[3]})
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--mode", default="walk", choices=["walk", "monotone"])
    ap.add_argument("--json", action="store_true")
    a = ap.parse_args()
    res = run(a.mode)
    if a.json:
        print(json.dumps(res))
        return
    keys = list(res)
    print("step  amax      " + "  ".join(f"{k:>24s}" for k in keys))
    print("                " + "  ".join(f"{'sat blk / uflow blk / flush':>24s}" for _ in keys))
    for t in range(len(res[keys[0]])):
        row = [res[k][t] for k in keys]
        cells = "  ".join(f"{r['scale_sat_blocks']:>6d}/{r['scale_uflow_blocks']:>8d}/{r['elem_flushed']:>8d}" for r in row)
        print(f"{t:4d}  {row[0]['amax']:9.3g} {cells}")
    tot = {k: {m: sum(r[m] for r in res[k]) for m in ("scale_sat_blocks", "scale_uflow_blocks", "elem_clamped", "elem_flushed")} for k in keys}
    print(json.dumps(tot))


if __name__ == "__main__":
    main()

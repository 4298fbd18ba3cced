"""Times one libfp4q.so kernel on a synthetic input: CUDA events around
`--reps` launches on the current stream after `--warmup` launches, two
distinct inputs alternating so that no launch reads what the previous one
left in L2.  Prints one JSON line: milliseconds per launch and the rate in
algorithmic bytes (quantisers: 2 B read + 0.5625 B written per element and
axis; amax 2 B; dequantiser 0.5625 B read + 2 B written) or 2MNK flops.

Small cases of this command are what the committed ncu summaries capture.

  python -m fp4_block_scaled_bf16_gb300.kernel_bench --case dual_sr --rows 2048 --cols 16384
  cases: amax, row_rne, row_sr, dual_rne, dual_sr, 2d_rne, 2d_sr, dequant, gemm and gemm_nvfp4
  (--m --n --k; gemm_nvfp4 on UE4M3-scaled operands), gemm_rebias (the UE5M3
  GEMM through rebiased codes: two rebias launches, the native GEMM, the
  conditional emulated one), gemm_two_windows (the same for wgrad's shape of
  operands -- A a gradient column-wise with SR, B activations column-wise, K
  the tokens -- with A's codes in two windows: two rebias launches, the
  two-accumulator native GEMM, the conditional emulated one), and step: the
  whole linear fwd+bwd step of the
  bench (X [m, k], W [n, k], dY [m, n]) under periodic tensor scaling on
  three streams, one "launch" per step (its first step launches 12 kernels --
  amax and tensor scale of X, W, dY, three quantisations, three GEMMs -- every
  later one 6, plus a tensor scale per tensor every 16 steps); step_rebias:
  the same step with fprop and dgrad through rebiased codes (6 more launches
  per step: two rebias kernels and a conditional emulated GEMM each);
  step_rebias_wgrad: that step with wgrad through two-window codes as well
  (3 more launches per step).
"""
from __future__ import annotations

import argparse
import json

import torch

from . import build, fp4q, workloads

CASES = ("amax", "row_rne", "row_sr", "dual_rne", "dual_sr", "2d_rne", "2d_sr", "dequant", "gemm", "gemm_nvfp4",
         "gemm_rebias", "gemm_two_windows", "step", "step_rebias", "step_rebias_wgrad")


def _inputs(case, rows, cols, dev):
    gen = workloads.gradients if case.endswith("_sr") else workloads.weights
    return [workloads.to_torch_bf16(gen(rows, cols, 50 + i)).to(dev) for i in range(2)]


def run(case, rows=16384, cols=4096, m=8192, n=16384, k=4096, reps=10, warmup=3):
    build.build()
    dev = torch.device("cuda")
    u8 = dict(dtype=torch.uint8, device=dev)
    if case.startswith("step"):
        from .linear_step import LinearStep

        X = workloads.to_torch_bf16(workloads.activations(m, k, 1)).to(dev)
        W = workloads.to_torch_bf16(workloads.weights(n, k, 2)).to(dev)
        dY = workloads.to_torch_bf16(workloads.gradients(m, n, 3)).to(dev)
        st = LinearStep(X, W, dY, seed=7, rebias=case != "step", rebias_wgrad=case == "step_rebias_wgrad")
        launch = lambda j: st.run_overlapped(periodic=True)
        work, unit = 3 * 2.0 * m * n * k, "TFLOP/s"
    elif case == "gemm_two_windows":
        qa = fp4q.quantize(workloads.to_torch_bf16(workloads.gradients(k, m, 62)).to(dev), fp4q.AXIS_COL, None,
                           fp4q.UE5M3, fp4q.SR, 7)
        qb = fp4q.quantize(workloads.to_torch_bf16(workloads.activations(k, n, 63)).to(dev), fp4q.AXIS_COL)
        A = (qa.payload_col, qa.scales_col, qa.T)
        B = (qb.payload_col, qb.scales_col, qb.T)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        ah, al, b4 = torch.empty_like(A[1]), torch.empty_like(A[1]), torch.empty_like(B[1])
        fh, fl = (torch.empty(m, dtype=torch.float32, device=dev) for _ in range(2))
        fb = torch.empty(1, dtype=torch.float32, device=dev)
        flag = torch.zeros(1, dtype=torch.int32, device=dev)

        def launch(j):
            fp4q.fp4q_rebias_scales_two_windows(A[1], m, k // 16, ah, al, fh, fl, flag)
            fp4q.fp4q_rebias_scales(B[1], n, k // 16, False, b4, fb, flag)
            fp4q.fp4q_gemm_nvfp4_two_windows(A[0], ah, al, fh, A[2], B[0], b4, fb, B[2], m, n, k, flag, out)
            fp4q.fp4q_gemm_if(*A, *B, m, n, k, fp4q.UE5M3, flag, out)
        work, unit = 2.0 * m * n * k, "TFLOP/s"
    elif case in ("gemm", "gemm_nvfp4", "gemm_rebias"):
        fmt = fp4q.UE4M3 if case == "gemm_nvfp4" else fp4q.UE5M3
        xs = [fp4q.quantize(workloads.to_torch_bf16(workloads.activations(m, k, 60)).to(dev), fmt=fmt),
              fp4q.quantize(workloads.to_torch_bf16(workloads.weights(n, k, 61)).to(dev), fmt=fmt)]
        A = (xs[0].payload_row, xs[0].scales_row, xs[0].T)
        B = (xs[1].payload_row, xs[1].scales_row, xs[1].T)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        if case == "gemm":
            launch = lambda j: fp4q.fp4q_gemm(*A, *B, m, n, k, fmt, out)
        elif case == "gemm_rebias":
            a4, b4 = torch.empty_like(A[1]), torch.empty_like(B[1])
            fa = torch.empty(m, dtype=torch.float32, device=dev)
            fb = torch.empty(1, dtype=torch.float32, device=dev)
            flag = torch.zeros(1, dtype=torch.int32, device=dev)

            def launch(j):
                fp4q.fp4q_rebias_scales(A[1], m, k // 16, True, a4, fa, flag)
                fp4q.fp4q_rebias_scales(B[1], n, k // 16, False, b4, fb, flag)
                fp4q.fp4q_gemm_nvfp4_rebiased(A[0], a4, fa, A[2], B[0], b4, fb, B[2], m, n, k, flag, out)
                fp4q.fp4q_gemm_if(*A, *B, m, n, k, fmt, flag, out)
        else:
            launch = lambda j: fp4q.fp4q_gemm_nvfp4(*A, *B, m, n, k, out)
        work, unit = 2.0 * m * n * k, "TFLOP/s"
    else:
        xs = _inputs(case, rows, cols, dev)
        T = fp4q.tensor_scale(fp4q.amax(xs[0]))
        pr, sr = torch.empty((rows, cols // 2), **u8), torch.empty((rows, cols // 16), **u8)
        pc, sc = torch.empty((cols, rows // 2), **u8), torch.empty((cols, rows // 16), **u8)
        rnd = fp4q.SR if case.endswith("_sr") else fp4q.RNE
        unit = "GB/s"
        if case == "amax":
            a = torch.empty(1, dtype=torch.float32, device=dev)
            launch = lambda j: fp4q.fp4q_amax(xs[j % 2], a)
            work = 2.0 * rows * cols
        elif case.startswith("row"):
            launch = lambda j: fp4q.fp4q_quantize(xs[j % 2], fp4q.AXIS_ROW, fp4q.UE5M3, T, rnd, 7, pr, sr,
                                                  None, None)
            work = 2.5625 * rows * cols
        elif case.startswith("dual") or case.startswith("2d"):
            axis = fp4q.AXIS_BOTH if case.startswith("dual") else fp4q.AXIS_BOTH_2D
            launch = lambda j: fp4q.fp4q_quantize(xs[j % 2], axis, fp4q.UE5M3, T, rnd, 7, pr, sr, pc, sc)
            work = 3.125 * rows * cols
        elif case == "dequant":
            qs = [fp4q.quantize(x, fp4q.AXIS_ROW, T) for x in xs]
            o = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
            launch = lambda j: fp4q.fp4q_dequantize(qs[j % 2].payload_row, qs[j % 2].scales_row, rows, cols,
                                                    fp4q.UE5M3, T, o)
            work = 2.5625 * rows * cols
        else:
            raise ValueError(f"unknown case {case}")
    for j in range(warmup):
        launch(j)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for j in range(reps):
        launch(j)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    rate = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    status = fp4q.fp4q_get_device_status()
    extra = {"fallback": int(flag.item())} if case == "gemm_two_windows" else {}
    shape = {"m": m, "n": n, "k": k} if case.startswith(("gemm", "step")) else {"rows": rows, "cols": cols}
    return {"case": case, **shape, "reps": reps, "ms_per_launch": ms, "rate": rate, "unit": unit,
            "device_status": status, **extra}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=CASES, required=True)
    ap.add_argument("--rows", type=int, default=16384)
    ap.add_argument("--cols", type=int, default=4096)
    ap.add_argument("--m", type=int, default=8192)
    ap.add_argument("--n", type=int, default=16384)
    ap.add_argument("--k", type=int, default=4096)
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    a = ap.parse_args()
    print(json.dumps(run(a.case, a.rows, a.cols, a.m, a.n, a.k, a.reps, a.warmup)))


if __name__ == "__main__":
    main()

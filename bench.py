"""Benchmark of the UE5M3 FP4 hot path on one GB300.

One step = one 8B-class internal linear (in 4096 -> out 16384, 8192 tokens)
through the whole path of "UE5M3 FP4 Block Scaling for Stable Language Model
Pretraining" (Abstract): the tensor scales of X, W, dY under periodic tensor
scaling (refreshed every 16 steps from the amax each quantisation fuses in;
an amax pass only on the very first step); dual-axis block-16 E2M1/UE5M3
quantisation of X and W (RNE) and of dY (Philox SR, seed 7); the three
training GEMMs on the block-scaled operands (fprop Y = X W^T, dgrad
dX = dY W, wgrad dW = dY^T X), each 8192 x 16384 x 4096 multiply-adds.
All three run on the tensor cores' block-scaled MMA with their UE5M3 scale
codes rebiased to UE4M3 codes times powers of two (exact; the emulated GEMM
takes over on the device when a group does not fit): fprop and dgrad with
one window per A row, wgrad -- whose A rows run over tokens of very
different gradient magnitude -- with two windows per row and two
accumulators.  The same step with wgrad emulated, with all three GEMMs
emulated, and under current scaling (amax pass + scale before every
quantisation), are timed beside it.

value = the three GEMMs' 2MNK flops / step time (quantisation included),
TFLOP/s.  Per-kernel CUDA-event times give the quantiser GB/s and the GEMM
TFLOP/s against the measured rooflines (MEASURED_PEAKS.json).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle on a bounded sample of the same step.
Multi-GPU: replicas only (every rank runs its own independent step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_TOK, HID, FFN = 8192, 4096, 16384
GEMM_FLOPS = 2.0 * M_TOK * FFN * HID          # each of fprop, dgrad, wgrad
STEP_FLOPS = 3 * GEMM_FLOPS
METRIC = "E2M1/UE5M3 quantize GB/s & block-scaled GEMM TFLOP/s, % of roofline"
WORKLOAD = ("8B-class linear 4096->16384, 8192 tokens: periodic tensor scales (refresh every 16 steps "
            "from the fused amax), dual-axis quantise X/W (RNE) and dY (SR seed 7), fprop+dgrad+wgrad "
            "block-scaled GEMMs")
# algorithmic bytes per element: read BF16 (2) + payload 0.5 + scale 1/16 per axis
DUAL_BYTES_PER_ELEM = 2 + 2 * (0.5 + 1 / 16)
ROW_BYTES_PER_ELEM = 2 + 0.5 + 1 / 16
AMAX_BYTES_PER_ELEM = 2


def kernel_sources_sha(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "fp4_block_scaled_bf16_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ["gemm.cu", "fp4q_device.cuh", "fp4q_pipeline.cuh", "fp4q_tcgen05.cuh"]
NATIVE_SOURCES = ["gemm_native.cu", "fp4q_device.cuh", "fp4q_pipeline.cuh", "fp4q_tcgen05.cuh"]


def committed_traffic(name, sources, launch=None):
    """DRAM bytes per launch from a committed ncu capture (of the launch
    whose "gemm" entry starts with `launch`, else the mean), or None when the
    kernel's sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_sha") != kernel_sources_sha(sources):
        return None
    if launch is not None:
        for l in d.get("launches", []):
            if l.get("gemm", "").startswith(launch):
                return l["dram_read_bytes"] + l["dram_write_bytes"]
        return None
    return d.get("dram_bytes_per_launch")


QUANT_SOURCES = ["quantize.cu", "fp4q_device.cuh"]
SMS, SCHEDULERS_PER_SM = 152, 4   # GB300: warp instructions issued per SM and clock


def issue_roofline(q_gbs, sm_mhz):
    """The dual-axis quantisers against the instruction-issue rate: at n
    thread instructions per element (committed ncu counts, used only while
    the quantiser sources hash to the captured version) the SMs' schedulers
    (one warp instruction per clock each) cap the rate at
    SMs x schedulers x 32 x clock / n elements per second, 3.125 B each."""
    p = os.path.join(ROOT, "profiles", "quantize_instructions.json")
    if not os.path.exists(p) or not sm_mhz:
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_sha") != kernel_sources_sha(QUANT_SOURCES):
        return None
    per = d["thread_instructions_per_element"]
    n_rne = next(v for k, v in per.items() if k.startswith("quantize_tile_kernel"))
    n_sr = next(v for k, v in per.items() if k.startswith("quantize_tile4_kernel"))
    thread_ips = SMS * SCHEDULERS_PER_SM * 32 * sm_mhz * 1e6
    peak = {"X_dual_rne": thread_ips / n_rne * DUAL_BYTES_PER_ELEM / 1e9,
            "W_dual_rne": thread_ips / n_rne * DUAL_BYTES_PER_ELEM / 1e9,
            "dY_dual_sr": thread_ips / n_sr * DUAL_BYTES_PER_ELEM / 1e9}
    ach = dict(zip(("X_dual_rne", "W_dual_rne", "dY_dual_sr"), q_gbs))
    return {"bound": "alu", "unit": "GB/s", "achieved": ach, "peak": peak,
            "frac": {k: ach[k] / peak[k] for k in ach},
            "instructions_per_element": {"dual_rne": n_rne, "dual_sr": n_sr},
            "peak_source": f"{SMS} SMs x {SCHEDULERS_PER_SM} schedulers x 32 lanes x {sm_mhz:.0f} MHz (median SM "
                           "clock of the timed region) / ncu instructions per element (profiles/quantize_instructions.json)"}


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over the ranks of the initialised process group (the
    job time of N replicas is the slowest rank's); x itself with one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every one of `world` replicas runs the step."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _peak(d, *keys):
    for k in keys:
        v = d.get(k)
        if isinstance(v, (int, float)):
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "median", "peak"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # nvidia-smi's start-up (NVML initialisation) takes CPU and driver
            # time; the timed regions begin only once it is sampling
            t0 = time.time()
            while not self.rows and self.proc.poll() is None and time.time() - t0 < 5.0:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(2)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
                for n, v in zip(names, r[3:7]):
                    if v.lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def parse_cpulist(text: str) -> set:
    """CPU numbers of a sysfs list such as "0-3,8,10-11"."""
    cpus = set()
    for part in text.strip().split(","):
        part = part.strip()
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus


def bind_to_gpu_node(torch, index):
    """Restricts this process to the CPUs local to the GPU (its PCI device's
    local_cpulist), so that the pinned host buffers of the end-to-end
    measurement are allocated next to it, as `numactl --cpunodebind` would.
    Returns the CPU list, or None when it cannot be determined."""
    try:
        p = torch.cuda.get_device_properties(index)
        addr = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{addr}/local_cpulist") as f:
            text = f.read().strip()
        cpus = parse_cpulist(text)
        if cpus and cpus != set(os.sched_getaffinity(0)):
            os.sched_setaffinity(0, cpus & set(range(os.cpu_count() or 1)) or cpus)
        return text
    except Exception:
        return None


# ---------------------------------------------------------------- GPU path
def rebias_parts(torch, fp4q, st, steps):
    """Per-launch times of the pieces of the step's rebiased fprop, one
    stream, CUDA events between them: the per-row rebias of X's codes, the
    per-tensor rebias of W's, the native GEMM, and the emulated GEMM's launch
    when the flag tells it not to run (the operands and buffers of the
    step's last one-stream run; the flag is zeroed once before the region)."""
    tokens, hid, out = st.dims
    a4, fa, b4, fb, flag = st.rb[0]
    TX, TW = st.tensor_scales(periodic=False)[:2]   # the last run() quantised under current scaling
    flag.zero_()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        ev[k][0].record()
        fp4q.fp4q_rebias_scales(st.Xrs, tokens, hid // 16, True, a4, fa, flag)
        ev[k][1].record()
        fp4q.fp4q_rebias_scales(st.Wrs, out, hid // 16, False, b4, fb, flag)
        ev[k][2].record()
        fp4q.fp4q_gemm_nvfp4_rebiased(st.Xr, a4, fa, TX, st.Wr, b4, fb, TW, tokens, out, hid, flag, st.Y)
        ev[k][3].record()
        fp4q.fp4q_gemm_if(st.Xr, st.Xrs, TX, st.Wr, st.Wrs, TW, tokens, out, hid, fp4q.UE5M3, flag, st.Y)
        ev[k][4].record()
    torch.cuda.synchronize()
    seg = lambda a, b: sum(e[a].elapsed_time(e[b]) for e in ev) / steps
    return {"rebias_rows_X_ms": seg(0, 1), "rebias_tensor_W_ms": seg(1, 2), "native_gemm_ms": seg(2, 3),
            "skipped_emulated_launch_ms": seg(3, 4), "flag": int(flag.item())}


def wgrad_parts(torch, fp4q, st, steps):
    """The same for the step's wgrad through two-window codes: the per-row
    two-window rebias of dY's column-wise codes, the per-tensor rebias of X's,
    the two-accumulator native GEMM, and the emulated GEMM's skipped launch."""
    tokens, hid, out = st.dims
    ah, al, fh, fl, b4, fb, flag = st.rb[2]
    TX, TD = st.tensor_scales(periodic=False)[0], st.tensor_scales(periodic=False)[2]
    flag.zero_()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        ev[k][0].record()
        fp4q.fp4q_rebias_scales_two_windows(st.Dcs, out, tokens // 16, ah, al, fh, fl, flag)
        ev[k][1].record()
        fp4q.fp4q_rebias_scales(st.Xcs, hid, tokens // 16, False, b4, fb, flag)
        ev[k][2].record()
        fp4q.fp4q_gemm_nvfp4_two_windows(st.Dc, ah, al, fh, TD, st.Xc, b4, fb, TX, out, hid, tokens, flag, st.dW)
        ev[k][3].record()
        fp4q.fp4q_gemm_if(st.Dc, st.Dcs, TD, st.Xc, st.Xcs, TX, out, hid, tokens, fp4q.UE5M3, flag, st.dW)
        ev[k][4].record()
    torch.cuda.synchronize()
    seg = lambda a, b: sum(e[a].elapsed_time(e[b]) for e in ev) / steps
    return {"rebias_two_windows_dY_ms": seg(0, 1), "rebias_tensor_X_ms": seg(1, 2), "native_gemm_ms": seg(2, 3),
            "skipped_emulated_launch_ms": seg(3, 4), "flag": int(flag.item())}


def run_gpu(args, rank, world):
    import torch
    from fp4_block_scaled_bf16_gb300 import build, fp4q, workloads
    from fp4_block_scaled_bf16_gb300.linear_step import LinearStep

    build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    affinity = bind_to_gpu_node(torch, dev.index)
    if M_TOK == workloads.TOKENS:
        Xb, Wb = workloads.fprop_operands()
        dYb = workloads.backward_gradient()
    else:
        Xb, Wb = workloads.activations(M_TOK, HID, 1), workloads.weights(FFN, HID, 2)
        dYb = workloads.gradients(M_TOK, FFN, 3)
    hX = workloads.to_torch_bf16(Xb).pin_memory()
    hW = workloads.to_torch_bf16(Wb).pin_memory()
    hD = workloads.to_torch_bf16(dYb).pin_memory()
    X, W, dY = hX.to(dev), hW.to(dev), hD.to(dev)
    # the step as the library runs it: the three GEMMs on the block-scaled
    # MMA through rebiased UE5M3 scale codes (wgrad's A in two windows;
    # emulated fallback decided on the device); the same step with wgrad
    # emulated; and with all three GEMMs emulated
    rstep = LinearStep(X, W, dY, seed=7, rebias=True, rebias_wgrad=True)
    wstep = LinearStep(X, W, dY, seed=7, rebias=True)
    step = LinearStep(X, W, dY, seed=7)
    for _ in range(args.warmup):
        for st_w in (rstep, wstep, step):
            st_w.run_overlapped(periodic=True)
            st_w.run_overlapped()
            st_w.run()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    # ---- device-resident timed regions, K steps each: the method's step
    # (periodic tensor scaling, three streams) -- the headline; the same step
    # with all three GEMMs emulated; the headline step under current scaling
    # (an amax pass before every quantisation); and both current-scaling
    # steps launched one kernel after another on one stream with events
    # between the pieces, for the per-kernel times
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    evr = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]

    def timed(fn):
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for k in range(args.steps):
            fn(k)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    with ClockSampler(dev.index) as clk:
        rstep.launches = 0
        ms = timed(lambda k: rstep.run_overlapped(periodic=True))
        launches = rstep.launches
        fallbacks = rstep.fallbacks()
        refreshes = [sc.step for sc in rstep.scalers]
        ms_emulated = timed(lambda k: step.run_overlapped(periodic=True))
        ms_wgrad_emulated = timed(lambda k: wstep.run_overlapped(periodic=True))
        ms_current = timed(lambda k: rstep.run_overlapped())
        ms_serial = timed(lambda k: step.run(evs[k]))
        ms_serial_r = timed(lambda k: rstep.run(evr[k]))
        parts = rebias_parts(torch, fp4q, rstep, args.steps)
        wparts = wgrad_parts(torch, fp4q, rstep, args.steps)
    del wstep
    if world > 1:
        ms = max_over_ranks(ms, dev)
        ms_emulated = max_over_ranks(ms_emulated, dev)
        ms_current = max_over_ranks(ms_current, dev)
        ms_wgrad_emulated = max_over_ranks(ms_wgrad_emulated, dev)
    seg = lambda a, b: sum(e[a].elapsed_time(e[b]) for e in evs) / args.steps
    segr = lambda a, b: sum(e[a].elapsed_time(e[b]) for e in evr) / args.steps
    t_scale, t_qx, t_qw, t_qd = seg(0, 1), seg(1, 2), seg(2, 3), seg(3, 4)
    t_g = [seg(4, 5), seg(5, 6), seg(6, 7)]
    t_gr = [segr(4, 5), segr(5, 6), segr(6, 7)]
    status = fp4q.fp4q_get_device_status()

    # ---- end to end through the API with host buffers: every step copies its
    # inputs host -> device and its results device -> host.  Copies run on
    # their own streams and overlap the neighbouring steps' kernels (NSETS
    # device buffer sets in turn), which is how a training loop feeds the GPU.
    NSETS = args.e2e_sets
    hY = [torch.empty(step.Y.shape, dtype=torch.bfloat16).pin_memory() for _ in range(NSETS)]
    hdX = [torch.empty(step.dX.shape, dtype=torch.bfloat16).pin_memory() for _ in range(NSETS)]
    hdW = [torch.empty(step.dW.shape, dtype=torch.bfloat16).pin_memory() for _ in range(NSETS)]
    steps2 = [rstep] + [LinearStep(torch.empty_like(X), torch.empty_like(W), torch.empty_like(dY), seed=7,
                                   rebias=True, rebias_wgrad=True) for _ in range(NSETS - 1)]
    s_h2d, s_cmp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    e2e_warm = NSETS + 1
    e2e_steps = max(2, args.steps)
    n_e2e = e2e_warm + e2e_steps
    ev_in = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_done = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_out = [torch.cuda.Event() for _ in range(n_e2e)]

    def e2e_step(i):
        st_i = steps2[i % NSETS]
        with torch.cuda.stream(s_h2d):
            if i >= NSETS:
                s_h2d.wait_event(ev_done[i - NSETS])      # buffer set free again
            st_i.X.copy_(hX, non_blocking=True)
            st_i.W.copy_(hW, non_blocking=True)
            st_i.dY.copy_(hD, non_blocking=True)
            ev_in[i].record(s_h2d)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[i])
            if i >= NSETS:
                s_cmp.wait_event(ev_out[i - NSETS])      # outputs read back
            st_i.run_overlapped(periodic=True)
            ev_done[i].record(s_cmp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev_done[i])
            hY[i % NSETS].copy_(st_i.Y, non_blocking=True)
            hdX[i % NSETS].copy_(st_i.dX, non_blocking=True)
            hdW[i % NSETS].copy_(st_i.dW, non_blocking=True)
            ev_out[i].record(s_d2h)

    # warm-up: every buffer set and both copy directions once through the
    # pipeline, untimed (each set's first step also runs its amax pass)
    for i in range(e2e_warm):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(s_h2d)
    for i in range(e2e_warm, n_e2e):
        e2e_step(i)
    s_h2d.wait_event(ev_out[n_e2e - 1])
    s1.record(s_h2d)
    torch.cuda.synchronize()
    e2e_ms = s0.elapsed_time(s1) / e2e_steps
    h2d = (hX.numel() + hW.numel() + hD.numel()) * 2
    # the host link on its own: one 256 MiB copy each way from pinned memory
    link = {}
    for name, src, dst in (("h2d_gbs", hD, steps2[0].dY), ("d2h_gbs", steps2[0].dY, hD)):
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record()
        dst.copy_(src, non_blocking=True)
        c1.record()
        torch.cuda.synchronize()
        link[name] = src.numel() * 2 / (c0.elapsed_time(c1) * 1e-3) / 1e9
    d2h = (hY[0].numel() + hdX[0].numel() + hdW[0].numel()) * 2
    del steps2

    # ---- quantiser rates outside the step.  Each is timed as the replay of a
    # CUDA graph of its launches, so that the host's per-call cost does not
    # enter the device time of these short kernels; inputs larger than L2.
    def _graph_ms(fn, calls, replays=5):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()                                    # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record()
        for _ in range(replays):
            g.replay()
        b1.record()
        torch.cuda.synchronize()
        del g
        return b0.elapsed_time(b1) / (replays * calls)

    rates = {}
    # every rate alternates two distinct inputs of the same shape (each at
    # least as large as L2), so that no launch reads what the previous one
    # left in L2: W and a row-reversed copy of it, dY and a row-reversed copy
    W2 = torch.flip(step.W, dims=(0,)).contiguous()
    dY2 = torch.flip(step.dY, dims=(0,)).contiguous()
    rot = {id(step.W): (step.W, W2), id(step.dY): (step.dY, dY2)}
    # single-axis: W row-wise RNE and dY row-wise SR, 10 launches
    for name, x, rnd, pay, sc in (("W_row_rne", step.W, fp4q.RNE, step.Wr, step.Wrs),
                                  ("dY_row_sr", step.dY, fp4q.SR, step.Dr, step.Drs)):
        Tn = step.T[1:2] if x is step.W else step.T[2:3]

        def run(x=x, rnd=rnd, pay=pay, sc=sc, Tn=Tn):
            for j in range(10):
                fp4q.fp4q_quantize(rot[id(x)][j % 2], fp4q.AXIS_ROW, fp4q.UE5M3, Tn, rnd, 7, pay, sc, None, None)
        rates[name] = x.numel() * ROW_BYTES_PER_ELEM / (_graph_ms(run, 10) * 1e-3) / 1e9
    # dequantisation (support op): W's and W2's row-wise payload and scales -> BF16
    Wd = torch.empty_like(step.W)
    q2 = fp4q.quantize(W2, fp4q.AXIS_ROW, step.T[1:2])
    deq_in = ((step.Wr, step.Wrs), (q2.payload_row, q2.scales_row))

    def run_deq():
        for j in range(10):
            fp4q.fp4q_dequantize(*deq_in[j % 2], FFN, HID, fp4q.UE5M3, step.T[1:2], Wd)
    rates["W_dequant_bf16"] = step.W.numel() * ROW_BYTES_PER_ELEM / (_graph_ms(run_deq, 10) * 1e-3) / 1e9
    del Wd, q2, deq_in
    # 16 x 16 (transposition-invariant) scaling: both layouts from one
    # quantisation, same algorithmic bytes as the dual-axis quantisers
    for name, x, rnd, outs in (("W_2d_rne", step.W, fp4q.RNE, (step.Wr, step.Wrs, step.Wc, step.Wcs)),
                               ("dY_2d_sr", step.dY, fp4q.SR, (step.Dr, step.Drs, step.Dc, step.Dcs))):
        Tn = step.T[1:2] if x is step.W else step.T[2:3]

        def run2d(x=x, rnd=rnd, outs=outs, Tn=Tn):
            for j in range(10):
                fp4q.fp4q_quantize(rot[id(x)][j % 2], fp4q.AXIS_BOTH_2D, fp4q.UE5M3, Tn, rnd, 7, *outs)
        rates[name] = x.numel() * DUAL_BYTES_PER_ELEM / (_graph_ms(run2d, 10) * 1e-3) / 1e9
    # the step's dual-axis quantisers on their own (graph replays, as above):
    # X (64 MiB) rotates through four distinct copies, W and dY through two,
    # so every rotation spans at least twice the L2
    Xs = [step.X] + [torch.roll(step.X, shifts=1024 * i, dims=0).contiguous() for i in (1, 2, 3)]
    dual = {}
    for name, xs, rnd, outs, Ti in (("X_dual_rne", Xs, fp4q.RNE, (step.Xr, step.Xrs, step.Xc, step.Xcs), 0),
                                    ("W_dual_rne", rot[id(step.W)], fp4q.RNE, (step.Wr, step.Wrs, step.Wc, step.Wcs), 1),
                                    ("dY_dual_sr", rot[id(step.dY)], fp4q.SR, (step.Dr, step.Drs, step.Dc, step.Dcs), 2)):
        Tn = step.T[Ti:Ti + 1]

        def run_dual(xs=xs, rnd=rnd, outs=outs, Tn=Tn):
            for j in range(8):
                fp4q.fp4q_quantize(xs[j % len(xs)], fp4q.AXIS_BOTH, fp4q.UE5M3, Tn, rnd, 7, *outs)
        dual[name] = xs[0].numel() * DUAL_BYTES_PER_ELEM / (_graph_ms(run_dual, 8) * 1e-3) / 1e9
    del W2, dY2, rot, Xs
    # periodic scaling (config 4's per-step quantisation): a 4096 x 4096
    # tensor quantised row-wise (RNE) with the fused amax that the next
    # refresh uses, the tensor scale taken from an earlier step (no amax
    # pass); eight distinct tensors in turn, 256 MB in all, so that inputs do
    # not stay in L2.  The block and element counts (a report, not needed by
    # the scaling) are timed separately.
    per = [torch.randn(4096, 4096, device=dev).bfloat16() for _ in range(8)]
    Tp = fp4q.tensor_scale(fp4q.amax(per[0]))
    pp = torch.empty((4096, 2048), dtype=torch.uint8, device=dev)
    sp = torch.empty((4096, 256), dtype=torch.uint8, device=dev)
    stp = torch.empty((1, 4), dtype=torch.int64, device=dev)
    ap = torch.empty(1, dtype=torch.float32, device=dev)
    for name, st in (("periodic_4096sq_row_rne_amax", None), ("periodic_4096sq_row_rne_amax_counts", stp)):
        def run_per(st=st):
            for x in per:
                fp4q.fp4q_quantize(x, fp4q.AXIS_ROW, fp4q.UE5M3, Tp, fp4q.RNE, 0, pp, sp, None, None, st, ap)
        rates[name] = 4096 * 4096 * ROW_BYTES_PER_ELEM / (_graph_ms(run_per, len(per)) * 1e-3) / 1e9
    del per
    # ---- fprop with the quantisation of Y for the next layer: separate
    # (GEMM, then row-wise RNE quantisation of Y) versus fused into the GEMM's
    # epilogue, with and without writing Y in BF16; 10 launches each
    def _timed(fn, n=10):
        fn()
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record()
        for _ in range(n):
            fn()
        b1.record()
        torch.cuda.synchronize()
        return b0.elapsed_time(b1) / n
    T0, T1 = step.T[0:1], step.T[1:2]
    TY = fp4q.tensor_scale(fp4q.amax(step.Y))
    pY = torch.empty((M_TOK, FFN // 2), dtype=torch.uint8, device=dev)
    sY = torch.empty((M_TOK, FFN // 16), dtype=torch.uint8, device=dev)
    aY = torch.empty(1, dtype=torch.float32, device=dev)
    g_args = (step.Xr, step.Xrs, T0, step.Wr, step.Wrs, T1, M_TOK, FFN, HID, fp4q.UE5M3)
    fused = {
        "gemm_ms": _timed(lambda: fp4q.fp4q_gemm(*g_args, step.Y)),
        "gemm_then_quantize_ms": _timed(lambda: (fp4q.fp4q_gemm(*g_args, step.Y), fp4q.fp4q_quantize(
            step.Y, fp4q.AXIS_ROW, fp4q.UE5M3, TY, fp4q.RNE, 0, pY, sY, None, None))),
        "fused_ms": _timed(lambda: fp4q.fp4q_gemm_quantize(*g_args, TY, step.Y, pY, sY, aY)),
        "fused_without_bf16_ms": _timed(lambda: fp4q.fp4q_gemm_quantize(*g_args, TY, None, pY, sY, aY)),
    }
    # the same on the step's fast path: rebias of X's and W's codes, the
    # native GEMM (quantising in its epilogue) and the conditional fallback
    a4, fa, b4, fb, flag = step_rb = rstep.rb[0]
    nat = (step.Xr, a4, fa, T0, step.Wr, b4, fb, T1, M_TOK, FFN, HID, flag)

    def fast(quantize, bf16=True):
        flag.zero_()
        fp4q.fp4q_rebias_scales(step.Xrs, M_TOK, HID // 16, True, a4, fa, flag)
        fp4q.fp4q_rebias_scales(step.Wrs, FFN, HID // 16, False, b4, fb, flag)
        if quantize:
            aY.zero_()
            fp4q.fp4q_gemm_nvfp4_rebiased_quantize(*nat, fp4q.UE5M3, TY, step.Y if bf16 else None, pY, sY, aY)
            fp4q.fp4q_gemm_quantize_if(*g_args, flag, TY, step.Y if bf16 else None, pY, sY, aY)
        else:
            fp4q.fp4q_gemm_nvfp4_rebiased(*nat, step.Y)
            fp4q.fp4q_gemm_if(*g_args, flag, step.Y)

    fused.update({
        "rebiased_gemm_ms": _timed(lambda: fast(False)),
        "rebiased_gemm_then_quantize_ms": _timed(lambda: (fast(False), fp4q.fp4q_quantize(
            step.Y, fp4q.AXIS_ROW, fp4q.UE5M3, TY, fp4q.RNE, 0, pY, sY, None, None))),
        "rebiased_fused_ms": _timed(lambda: fast(True)),
        "rebiased_fused_without_bf16_ms": _timed(lambda: fast(True, False)),
    })
    del step_rb

    # ---- the full 8B-class linear block: the four internal linears (QKV,
    # out, up, down) each through the same fwd+bwd step, one after another
    block = None
    if M_TOK == workloads.TOKENS and not args.no_block:
        lin = []
        for name in workloads.LINEARS:
            xb, wb, db = workloads.linear_block(name)
            lin.append(LinearStep(workloads.to_torch_bf16(xb).to(dev), workloads.to_torch_bf16(wb).to(dev),
                                  workloads.to_torch_bf16(db).to(dev), seed=7, rebias=True, rebias_wgrad=True))
        for _ in range(2):
            for st_l in lin:
                st_l.run_overlapped(periodic=True)
        torch.cuda.synchronize()
        nb = max(2, args.steps // 4)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record()
        for _ in range(nb):
            for st_l in lin:
                st_l.run_overlapped(periodic=True)
        c1.record()
        torch.cuda.synchronize()
        bms = c0.elapsed_time(c1) / nb
        bflops = sum(3 * 2.0 * workloads.TOKENS * fi * fo for fi, fo in workloads.LINEARS.values())
        block = {"ms_per_block_step": bms, "TFLOP/s": bflops / (bms * 1e-3) / 1e12, "steps": nb,
                 "fallbacks_fprop_dgrad_wgrad": [st_l.fallbacks() for st_l in lin],
                 "linears": ", ".join(f"{k} {fi}->{fo}" for k, (fi, fo) in workloads.LINEARS.items()),
                 "tokens": workloads.TOKENS}
        del lin

    # ---- the native NVFP4 path on the same shapes: UE4M3-scaled operands,
    # the three GEMMs on the tensor cores' block-scaled MMA; the step as
    # scheduled (periodic scaling, three streams) and per-kernel times (one
    # stream), then the four-linear block
    nstep = LinearStep(step.X, step.W, step.dY, seed=7, fmt=fp4q.UE4M3, native=True)
    for _ in range(args.warmup):
        nstep.run_overlapped(periodic=True)
        nstep.run(periodic=True)
    evn = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    ms_native = timed(lambda k: nstep.run_overlapped(periodic=True))
    timed(lambda k: nstep.run(evn[k], periodic=True))
    segn = lambda a, b: sum(e[a].elapsed_time(e[b]) for e in evn) / args.steps
    native = {"ms_per_step": ms_native / args.steps, "gemm_ms": [segn(4, 5), segn(5, 6), segn(6, 7)],
              "quantize_ms": [segn(1, 2), segn(2, 3), segn(3, 4)]}
    del nstep
    if block is not None:
        lin = []
        for name in workloads.LINEARS:
            xb, wb, db = workloads.linear_block(name)
            lin.append(LinearStep(workloads.to_torch_bf16(xb).to(dev), workloads.to_torch_bf16(wb).to(dev),
                                  workloads.to_torch_bf16(db).to(dev), seed=7, fmt=fp4q.UE4M3, native=True))
        for _ in range(2):
            for st_l in lin:
                st_l.run_overlapped(periodic=True)
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record()
        for _ in range(block["steps"]):
            for st_l in lin:
                st_l.run_overlapped(periodic=True)
        c1.record()
        torch.cuda.synchronize()
        bms = c0.elapsed_time(c1) / block["steps"]
        native["block_ms_per_step"] = bms
        native["block_TFLOP/s"] = block["TFLOP/s"] * block["ms_per_block_step"] / bms
        del lin

    return dict(ms=ms, ms_emulated=ms_emulated, ms_current=ms_current, refreshes=refreshes, ms_serial=ms_serial,
                ms_serial_r=ms_serial_r, t_gr=t_gr, parts=parts, wparts=wparts, fallbacks=fallbacks, dual=dual,
                ms_wgrad_emulated=ms_wgrad_emulated,
                native=native, fused=fused, block=block, t_scale=t_scale, t_q=(t_qx, t_qw, t_qd), t_g=t_g, launches=launches, rates=rates,
                clocks=clk.summary(), status=status, e2e_ms=e2e_ms, e2e_steps=e2e_steps, e2e_sets=NSETS,
                h2d=h2d, d2h=d2h, link=link, affinity=affinity,
                elems=(X.numel(), W.numel(), dY.numel()))


# ---------------------------------------------------------------- oracle path
# The oracle runs as it stands (single-threaded C behind numpy) in one process
# per host core, started with `spawn` (never forked from a process that has
# used the GPU); each worker holds its own slice of the step's inputs, and a
# phase's wall time is taken in the parent around all workers' share of it.
_ORC = {}


def _oracle_worker_setup(qrows, grows, gcols, seed):
    """Builds this worker's inputs (untimed): qrows rows of X and of dY, and
    the quantised operands of a grows x gcols slice of fprop."""
    import oracle
    from fp4_block_scaled_bf16_gb300 import workloads

    oracle.build()
    x = workloads.activations(qrows, HID, 1 + 10 * seed)
    d = workloads.gradients(qrows, FFN, 3 + 10 * seed)
    w = workloads.weights(gcols, HID, 2 + 10 * seed)
    Tx = oracle.tensor_scale(oracle.amax(x)[0])
    Tw = oracle.tensor_scale(oracle.amax(w)[0])
    pa, sa, _ = oracle.quantize(x[:max(grows, 16)], oracle.ROW, Tx)
    pb, sb, _ = oracle.quantize(w, oracle.ROW, Tw)
    _ORC.update(x=x, d=d, ga=(pa[:grows], sa[:grows], Tx), gb=(pb, sb, Tw))
    time.sleep(0.5)   # hold this worker so that every worker takes one slice
    return os.getpid()


def _oracle_worker_quantise(_):
    """Seconds for amax + tensor scale + row and column quantisation of the
    worker's X (RNE) and dY (SR) slices, and the elements quantised."""
    import oracle

    x, d = _ORC["x"], _ORC["d"]
    t0 = time.perf_counter()
    Tx = oracle.tensor_scale(oracle.amax(x)[0])
    Td = oracle.tensor_scale(oracle.amax(d)[0])
    oracle.quantize(x, oracle.ROW, Tx)
    oracle.quantize(x, oracle.COL, Tx)
    oracle.quantize(d, oracle.ROW, Td, rnd=oracle.SR, seed=7)
    oracle.quantize(d, oracle.COL, Td, rnd=oracle.SR, seed=7)
    return time.perf_counter() - t0, x.size + d.size


def _oracle_worker_gemm(_):
    """Seconds for the worker's binary64 GEMM slice, and its multiply-adds."""
    import oracle

    (pa, sa, Ta), (pb, sb, Tb) = _ORC["ga"], _ORC["gb"]
    t0 = time.perf_counter()
    oracle.gemm(pa, sa, Ta, pb, sb, Tb)
    return time.perf_counter() - t0, pa.shape[0] * pb.shape[0] * HID


class OracleSample:
    """A pool of `workers` oracle processes, each holding a bounded slice of
    the step (qrows rows of X and dY quantised on both axes; a grows x gcols
    slice of fprop in binary64).  `run()` times one sample: each phase on all
    workers at once, wall time taken in the parent."""

    def __init__(self, qrows, grows, gcols, workers=None):
        import multiprocessing as mp

        self.workers = workers or len(os.sched_getaffinity(0))
        # the oracle is single-threaded C; keep numpy's own pools to one thread
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ.setdefault(v, "1")
        self.pool = mp.get_context("spawn").Pool(self.workers)
        pids = self.pool.starmap(_oracle_worker_setup,
                                 [(qrows, grows, gcols, i) for i in range(self.workers)], chunksize=1)
        if len(set(pids)) != self.workers:
            self.close()
            raise RuntimeError("oracle pool: a worker took two slices")
        self.shape = (qrows, grows, gcols)

    def run(self):
        """(estimated seconds for the whole step, measured seconds, elements
        quantised, multiply-adds) for one sample."""
        t0 = time.perf_counter()
        q = self.pool.map(_oracle_worker_quantise, range(self.workers), chunksize=1)
        wall_q = time.perf_counter() - t0
        t0 = time.perf_counter()
        g = self.pool.map(_oracle_worker_gemm, range(self.workers), chunksize=1)
        wall_g = time.perf_counter() - t0
        q_elems = sum(n for _, n in q)
        macs = sum(n for _, n in g)
        step_elems = M_TOK * HID + FFN * HID + M_TOK * FFN
        est = wall_q / q_elems * step_elems + wall_g / macs * (STEP_FLOPS / 2)
        return est, wall_q + wall_g, q_elems, macs

    def describe(self, q_elems, macs, spent):
        qrows, grows, gcols = self.shape
        return (f"{self.workers} oracle processes at once, each quantising {qrows} rows of X and of dY on both "
                f"axes (RNE / SR) and a {grows} x {gcols} x {HID} binary64 GEMM slice: {q_elems} elements and "
                f"{macs} MACs in {spent:.2f} s of wall time; scaled to the full step "
                f"({M_TOK * HID + FFN * HID + M_TOK * FFN} elements quantised on two axes, "
                f"{STEP_FLOPS / 2:.3e} MACs)")

    def close(self):
        self.pool.close()
        self.pool.join()


# dense FP4 against dense BF16 tensor throughput on GB300 (13.5 / 2.25 PFLOP/s nominal)
FP4_OVER_BF16 = 6.0


def native_line(nat, world, bf16_peak, src):
    """The native NVFP4 path's numbers: the whole step (UE4M3 quantisation and
    three block-scaled-MMA GEMMs), the GEMMs against the FP4 peak derived
    from the measured BF16 one by the nominal dense ratio."""
    g = GEMM_FLOPS / (sum(nat["gemm_ms"]) / 3 * 1e-3) / 1e12
    peak = bf16_peak * FP4_OVER_BF16 if bf16_peak else None
    out = {"ms_per_step": nat["ms_per_step"], "TFLOP/s": job_tflops(world, STEP_FLOPS, nat["ms_per_step"]),
           "gemm_ms": nat["gemm_ms"], "quantize_ms_one_stream": nat["quantize_ms"],
           "roofline": {"bound": "tensor", "achieved": g, "peak": peak, "unit": "TFLOP/s",
                        "frac": g / peak if peak else None,
                        "kernel": "fp4q gemm_nvfp4_kernel (mean of fprop/dgrad/wgrad)",
                        "peak_source": f"{src} bf16 x {FP4_OVER_BF16:g} (nominal dense fp4 / bf16)"}}
    if "block_ms_per_step" in nat:
        out["linear_block_ms_per_step"] = nat["block_ms_per_step"]
        out["linear_block_TFLOP/s"] = nat["block_TFLOP/s"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="fp4q", choices=["fp4q", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-block", action="store_true",
                    help="skip the four-linear block measurement (profiling captures)")
    ap.add_argument("--e2e-sets", type=int, default=2,
                    help="device buffer sets the end-to-end pipeline rotates through")
    ap.add_argument("--tokens", type=int, default=8192,
                    help="rows of X and dY; smaller values only for profiling captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    global M_TOK, GEMM_FLOPS, STEP_FLOPS
    if args.tokens != M_TOK:
        M_TOK = args.tokens
        GEMM_FLOPS = 2.0 * M_TOK * FFN * HID
        STEP_FLOPS = 3 * GEMM_FLOPS

    if args.impl == "reference":
        if rank != 0:
            return
        # each step is one bounded sample of the workload on every host core
        # (about 1 s of wall time); ms_per_step is that sample's measured time
        orc = OracleSample(qrows=256, grows=2, gcols=4096)
        try:
            for _ in range(args.warmup):
                orc.run()
            est_total, spent = 0.0, 0.0
            for _ in range(args.steps):
                est, dt, q_elems, macs = orc.run()
                est_total += est
                spent += dt
        finally:
            orc.close()
        est = est_total / args.steps
        v = STEP_FLOPS / est / 1e12
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": spent / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "inputs larger than L2",
                       "step": "a bounded sample of the workload (value = its rate, scaled to the whole step)",
                       "ms_per_full_step_estimate": est * 1e3},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": orc.workers, "kind": "oracle",
                             "sample": f"per step: {orc.describe(q_elems, macs, spent / args.steps)}"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_gpu(args, rank, world)
    if rank != 0:
        return
    pk, src = peaks()
    hbm = _peak(pk, "hbm_gbs", "hbm_GBps", "hbm")
    # the per-kernel GEMM times come from the one-stream region: a burst of
    # tens of milliseconds is held to the burst peak, a region of seconds to
    # the sustained one
    burst = r["ms_serial"] < 1000.0
    bf16 = _peak(pk, "bf16_tflops", "bf16_tflops_sustained") if burst else _peak(pk, "bf16_tflops_sustained", "bf16_tflops")
    ms = r["ms"] / args.steps
    value = job_tflops(world, STEP_FLOPS, ms)
    t_gemm = sum(r["t_g"]) / 3
    gemm_tflops = GEMM_FLOPS / (t_gemm * 1e-3) / 1e12
    # the dominant kernel of the headline step: the two-window native GEMM of
    # its wgrad (CUDA events around its launch, one stream); algorithmic
    # flops are the UE5M3 GEMM's 2MNK (its two MMAs per K step are the cost
    # of the second window, not work of the method)
    pr, pw = r["parts"], r["wparts"]
    fp4_peak = bf16 * FP4_OVER_BF16 if bf16 else None
    two_tflops = GEMM_FLOPS / (pw["native_gemm_ms"] * 1e-3) / 1e12
    native_tflops = GEMM_FLOPS / (pr["native_gemm_ms"] * 1e-3) / 1e12
    # the emulated GEMM on the same wgrad (the all-emulated one-stream step)
    wgrad_tflops = GEMM_FLOPS / (r["t_g"][2] * 1e-3) / 1e12
    nX, nW, nD = r["elems"]
    q_bytes = [n * DUAL_BYTES_PER_ELEM for n in (nX, nW, nD)]
    # the dual-axis quantisers: their own rate (graph replays), and the rate
    # of their launch inside the one-stream pass of the step (CUDA events
    # around each call, so the host's gaps between calls count too)
    q_gbs_step = [b / (t * 1e-3) / 1e9 for b, t in zip(q_bytes, r["t_q"])]
    q_gbs = [r["dual"][k] for k in ("X_dual_rne", "W_dual_rne", "dY_dual_sr")]
    cpu = None
    if not args.no_cpu_baseline:
        # about 30 s of CPU work spread over the host cores
        orc = OracleSample(qrows=512, grows=4, gcols=4096)
        try:
            orc.run()                                   # warm caches and pages
            est, spent, q_elems, macs = orc.run()
        finally:
            orc.close()
        cpu = {"value": STEP_FLOPS / est / 1e12, "unit": "TFLOP/s", "cores": orc.workers, "kind": "oracle",
               "sample": orc.describe(q_elems, macs, spent)}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_periodic": ms,
        "ms_per_step_current_scaling": r["ms_current"] / args.steps,
        "ms_per_step_all_gemms_emulated": r["ms_emulated"] / args.steps,
        "ms_per_step_wgrad_emulated": r["ms_wgrad_emulated"] / args.steps,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "E2M1/UE5M3 operands; e2m1 x e2m1 block-scaled MMA -> f32 (UE5M3 scales as UE4M3 codes x 2^k, "
                 "exact; wgrad's A in two windows, two f32 accumulators)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_TOK, "hidden": HID, "ffn": FFN,
                   "l2": "inputs larger than L2 (dY 256 MiB, step working set ~1 GiB)",
                   "schedule": "three streams: X/W scale, quantise and fprop; dY scale, SR "
                               "quantise and dgrad; wgrad once dY and X are quantised",
                   "tensor_scaling": "periodic: T refreshed every 16 steps from the amax fused into the "
                                     "previous quantisation; amax pass on the first step only "
                                     f"(scaler steps after the timed region: {r['refreshes']})",
                   "gemm_paths": "scale codes rebiased (A per row, B per tensor) + native block-scaled MMA, "
                                 "emulated GEMM launched after it and run on the device only if a group does not "
                                 "fit: fprop, dgrad one window (14 binades) per A row; wgrad two windows (28 "
                                 "binades) per A row, two accumulators",
                   "fallbacks_fprop_dgrad_wgrad": r["fallbacks"],
                   "wgrad_emulated_TFLOP/s": job_tflops(world, STEP_FLOPS, r["ms_wgrad_emulated"] / args.steps),
                   "current_scaling_TFLOP/s": job_tflops(world, STEP_FLOPS, r["ms_current"] / args.steps),
                   "all_gemms_emulated_TFLOP/s": job_tflops(world, STEP_FLOPS, r["ms_emulated"] / args.steps),
                   "ms_per_step_one_stream_current_scaling": r["ms_serial_r"] / args.steps,
                   "ms_per_step_one_stream_current_scaling_all_emulated": r["ms_serial"] / args.steps,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": two_tflops, "peak": fp4_peak,
                     "unit": "TFLOP/s", "frac": two_tflops / fp4_peak if fp4_peak else None,
                     "traffic": committed_traffic("gemm_nvfp4_two_windows_traffic_wgrad.json", NATIVE_SOURCES),
                     "kernel": "fp4q gemm_nvfp4_kernel, two windows (the step's wgrad, 16384 x 4096 x 8192)",
                     "peak_source": f"{src} bf16 x {FP4_OVER_BF16:g} (nominal dense fp4 / bf16; "
                                    f"{'burst' if burst else 'sustained'}: the per-kernel region ran "
                                    f"{r['ms_serial_r']:.0f} ms)",
                     "mma_work": {"achieved": 2 * two_tflops, "frac": 2 * two_tflops / fp4_peak if fp4_peak else None,
                                  "note": "the same launch counting both MMAs of each K step (high and low "
                                          "window): the tensor cores' own throughput"},
                     "parts_ms": pw},
        "roofline_emulated_wgrad": {
            "bound": "tensor", "achieved": wgrad_tflops, "peak": bf16, "unit": "TFLOP/s",
            "frac": wgrad_tflops / bf16 if bf16 else None,
            "traffic": committed_traffic("gemm_kernel_traffic_8B_linear.json", GEMM_SOURCES, "wgrad"),
            "kernel": "fp4q gemm_kernel (emulated UE5M3 GEMM; the same wgrad, all-emulated step)",
            "peak_source": f"{src} bf16 ({'burst' if burst else 'sustained'})",
            "all_three_emulated": {"achieved": gemm_tflops, "frac": gemm_tflops / bf16 if bf16 else None,
                                   "traffic": committed_traffic("gemm_kernel_traffic_8B_linear.json", GEMM_SOURCES),
                                   "note": "mean over fprop/dgrad/wgrad of the all-emulated one-stream step"}},
        "roofline_native_rebiased": {"bound": "tensor", "achieved": native_tflops, "peak": fp4_peak,
                                     "unit": "TFLOP/s", "frac": native_tflops / fp4_peak if fp4_peak else None,
                                     "kernel": "fp4q gemm_nvfp4_kernel on rebiased UE5M3 operands (fprop)",
                                     "peak_source": f"{src} bf16 x {FP4_OVER_BF16:g} (nominal dense fp4 / bf16)",
                                     "parts_ms": pr},
        "roofline_quantize": {"bound": "hbm", "unit": "GB/s", "peak": hbm,
                              "achieved": dict({"X_dual_rne": q_gbs[0], "W_dual_rne": q_gbs[1], "dY_dual_sr": q_gbs[2]}, **r["rates"]),
                              "frac": dict({k: g / hbm for k, g in zip(("X_dual_rne", "W_dual_rne", "dY_dual_sr"), q_gbs)},
                                           **{k: g / hbm for k, g in r["rates"].items()}) if hbm else None,
                              "peak_source": f"{src} hbm",
                              "dual_axis_in_step_gbs": dict(zip(("X_dual_rne", "W_dual_rne", "dY_dual_sr"),
                                                                q_gbs_step)),
                              "issue_roofline": issue_roofline(q_gbs, (r["clocks"] or {}).get("sm_mhz"))},
        "breakdown_ms": {"amax_scale": r["t_scale"], "quantize_X": r["t_q"][0], "quantize_W": r["t_q"][1],
                         "quantize_dY": r["t_q"][2], "fprop": r["t_gr"][0], "dgrad": r["t_gr"][1],
                         "wgrad": r["t_gr"][2], "fprop_emulated": r["t_g"][0], "dgrad_emulated": r["t_g"][1],
                         "wgrad_emulated": r["t_g"][2]},
        "e2e": {"value": job_tflops(world, STEP_FLOPS, r["e2e_ms"]), "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms_per_step": r["e2e_ms"],
                "steps": r["e2e_steps"], "device_buffer_sets": r["e2e_sets"],
                "host_link_gbs": {k: round(v, 1) for k, v in r["link"].items()},
                "cpu_affinity": r["affinity"]},
        "native_nvfp4": native_line(r["native"], world, bf16, src),
        "fused_epilogue_fprop": r["fused"],
        "linear_block_fwd_bwd": r["block"],
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "device_status": r["status"],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()

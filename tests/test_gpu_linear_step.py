"""The method's own step on the GPU: one linear layer's fprop, dgrad and
wgrad on block-scaled operands under periodic tensor scaling (the step that
bench.py times as its headline), checked step by step against the oracle.

Over 20 steps whose X, W and dY drift in magnitude (x1.3 per step, seeded
direction), the step's tensor scales must be exactly the oracle
PeriodicScaler's (refresh every 16 steps from the previous step's amax, an
amax pass only on step 0), every payload and scale byte of the six
quantised operands must equal the oracle's, and the three GEMM results must
meet the stated tolerance on the refresh steps and the last one.

Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Abstract (periodic tensor scaling made possible by UE5M3's range; stochastic
rounding on backward gradients; the FP4 matrix multiplications of every
internal linear)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_block_scaled_bf16_gb300 import workloads
from parity_util import check_gemm_bf16

pytestmark = pytest.mark.gpu

TOK, HID, OUT, STEPS, PERIOD = 256, 256, 512, 20, 16


def _inputs(t, amaxes):
    """X, W, dY of step t: the generators' distributions, scaled by the
    drift factor of the step (W drifts the other way)."""
    def scaled(bits, f):
        return workloads.f32_to_bf16_bits(workloads.bf16_bits_to_f32(bits) * np.float32(f))
    X = scaled(workloads.activations(TOK, HID, 200 + t), amaxes[t])
    W = scaled(workloads.weights(OUT, HID, 300 + t), 1.0 / amaxes[t])
    dY = scaled(workloads.gradients(TOK, OUT, 400 + t), amaxes[t])
    return X, W, dY


def _u8(t):
    return t.cpu().numpy()


def test_periodic_step_matches_oracle_every_step():
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    from fp4_block_scaled_bf16_gb300.linear_step import LinearStep

    dev = torch.device("cuda")
    amaxes = workloads.drift_amaxes(STEPS)
    X = torch.empty((TOK, HID), dtype=torch.bfloat16, device=dev)
    W = torch.empty((OUT, HID), dtype=torch.bfloat16, device=dev)
    dY = torch.empty((TOK, OUT), dtype=torch.bfloat16, device=dev)
    step = LinearStep(X, W, dY, seed=7, period=PERIOD)
    refs = [oracle.PeriodicScaler(period=PERIOD) for _ in range(3)]
    Ts = []
    for t in range(STEPS):
        xb, wb, db = _inputs(t, amaxes)
        X.copy_(workloads.to_torch_bf16(xb))
        W.copy_(workloads.to_torch_bf16(wb))
        dY.copy_(workloads.to_torch_bf16(db))
        step.launches = 0
        step.run_overlapped(periodic=True)
        torch.cuda.synchronize()
        # 3 dual-axis quantisations + 3 GEMMs, plus the refreshes (and the
        # amax passes of step 0)
        assert step.launches == 6 + (3 if t % PERIOD == 0 else 0) + (3 if t == 0 else 0), t
        gT = [float(T.item()) for T in step.tensor_scales(periodic=True)]
        outs = ((step.Xr, step.Xrs, step.Xc, step.Xcs), (step.Wr, step.Wrs, step.Wc, step.Wcs),
                (step.Dr, step.Drs, step.Dc, step.Dcs))
        for i, (bits, rnd) in enumerate(((xb, oracle.RNE), (wb, oracle.RNE), (db, oracle.SR))):
            seed = 7 if rnd else 0
            pr, sr, _ = refs[i].quantize(bits, oracle.ROW, rnd, seed)
            assert gT[i] == refs[i].T, (t, i, gT[i], refs[i].T)
            pc, sc, _ = oracle.quantize(bits, oracle.COL, refs[i].T, oracle.UE5M3, rnd, seed)
            for name, g, w in zip(("row payload", "row scales", "col payload", "col scales"),
                                  outs[i], (pr, sr, pc, sc)):
                assert np.array_equal(_u8(g), w), (t, i, name)
            # the quantiser's fused amax is the one the next refresh uses
            assert float(step.scalers[i].last_amax.item()) == oracle.amax(bits)[0], (t, i)
        Ts.append(gT)
        if t % PERIOD == 0 or t == STEPS - 1:
            for C, A, B, Ta, Tb in ((step.Y, (step.Xr, step.Xrs), (step.Wr, step.Wrs), gT[0], gT[1]),
                                    (step.dX, (step.Dr, step.Drs), (step.Wc, step.Wcs), gT[2], gT[1]),
                                    (step.dW, (step.Dc, step.Dcs), (step.Xc, step.Xcs), gT[2], gT[0])):
                R = oracle.gemm(_u8(A[0]), _u8(A[1]), Ta, _u8(B[0]), _u8(B[1]), Tb)
                Cf = C.float().cpu().numpy().astype(np.float64)
                check_gemm_bf16(Cf, R)
    # T held between refreshes, refreshed at steps 0 and 16
    for t in range(1, STEPS):
        if t % PERIOD:
            assert Ts[t] == Ts[t - 1], t
    assert Ts[PERIOD] != Ts[PERIOD - 1]
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def test_native_nvfp4_step_matches_oracle():
    """The same step with UE4M3 scales and the three GEMMs on the native
    block-scaled MMA: tensor scales and every quantised byte equal the
    oracle's, GEMM results within the BF16 bound, over the first refresh."""
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    from fp4_block_scaled_bf16_gb300.linear_step import LinearStep

    steps, period = 3, 2
    amaxes = workloads.drift_amaxes(steps)
    dev = torch.device("cuda")
    X = torch.empty((TOK, HID), dtype=torch.bfloat16, device=dev)
    W = torch.empty((OUT, HID), dtype=torch.bfloat16, device=dev)
    dY = torch.empty((TOK, OUT), dtype=torch.bfloat16, device=dev)
    step = LinearStep(X, W, dY, seed=7, period=period, fmt=fp4q.UE4M3, native=True)
    refs = [oracle.PeriodicScaler(period=period, fmt=oracle.UE4M3) for _ in range(3)]
    for t in range(steps):
        xb, wb, db = _inputs(t, amaxes)
        X.copy_(workloads.to_torch_bf16(xb))
        W.copy_(workloads.to_torch_bf16(wb))
        dY.copy_(workloads.to_torch_bf16(db))
        step.run_overlapped(periodic=True)
        torch.cuda.synchronize()
        gT = [float(T.item()) for T in step.tensor_scales(periodic=True)]
        outs = ((step.Xr, step.Xrs, step.Xc, step.Xcs), (step.Wr, step.Wrs, step.Wc, step.Wcs),
                (step.Dr, step.Drs, step.Dc, step.Dcs))
        for i, (bits, rnd) in enumerate(((xb, oracle.RNE), (wb, oracle.RNE), (db, oracle.SR))):
            seed = 7 if rnd else 0
            pr, sr, _ = refs[i].quantize(bits, oracle.ROW, rnd, seed)
            assert gT[i] == refs[i].T, (t, i)
            pc, sc, _ = oracle.quantize(bits, oracle.COL, refs[i].T, oracle.UE4M3, rnd, seed)
            for g, w in zip(outs[i], (pr, sr, pc, sc)):
                assert np.array_equal(_u8(g), w), (t, i)
        for C, A, B, Ta, Tb in ((step.Y, (step.Xr, step.Xrs), (step.Wr, step.Wrs), gT[0], gT[1]),
                                (step.dX, (step.Dr, step.Drs), (step.Wc, step.Wcs), gT[2], gT[1]),
                                (step.dW, (step.Dc, step.Dcs), (step.Xc, step.Xcs), gT[2], gT[0])):
            R = oracle.gemm(_u8(A[0]), _u8(A[1]), Ta, _u8(B[0]), _u8(B[1]), Tb, oracle.UE4M3)
            check_gemm_bf16(C.float().cpu().numpy().astype(np.float64), R)
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def test_rebiased_step_matches_oracle():
    """The UE5M3 step with fprop and dgrad on the native MMA through rebiased
    scale codes: quantised bytes as in the emulated step, the fallback flags
    equal to the oracle's fit decisions on the same codes, and all three GEMM
    results within the BF16 bound of the oracle's UE5M3 contraction, on the
    refresh steps of a drifting sequence."""
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    from fp4_block_scaled_bf16_gb300.linear_step import LinearStep

    steps, period = 3, 2
    amaxes = workloads.drift_amaxes(steps)
    dev = torch.device("cuda")
    X = torch.empty((TOK, HID), dtype=torch.bfloat16, device=dev)
    W = torch.empty((OUT, HID), dtype=torch.bfloat16, device=dev)
    dY = torch.empty((TOK, OUT), dtype=torch.bfloat16, device=dev)
    step = LinearStep(X, W, dY, seed=7, period=period, rebias=True)
    assert step.rb[0] is not None and step.rb[1] is not None and step.rb[2] is None   # wgrad emulated
    for t in range(steps):
        xb, wb, db = _inputs(t, amaxes)
        X.copy_(workloads.to_torch_bf16(xb))
        W.copy_(workloads.to_torch_bf16(wb))
        dY.copy_(workloads.to_torch_bf16(db))
        step.launches = 0
        step.run_overlapped(periodic=True)
        torch.cuda.synchronize()
        # each of fprop and dgrad: two rebias launches, the native GEMM and
        # the conditional emulated one
        assert step.launches == 12 + (3 if t % period == 0 else 0) + (3 if t == 0 else 0), t
        gT = [float(T.item()) for T in step.tensor_scales(periodic=True)]
        fell = step.fallbacks()
        for g, (A, B) in enumerate((((step.Xr, step.Xrs), (step.Wr, step.Wrs)),
                                    ((step.Dr, step.Drs), (step.Wc, step.Wcs)))):
            fits = oracle.rebias_scales(_u8(A[1]), True)[2] and oracle.rebias_scales(_u8(B[1]), False)[2]
            assert fell[g] == (not fits), (t, g)
        for C, A, B, Ta, Tb in ((step.Y, (step.Xr, step.Xrs), (step.Wr, step.Wrs), gT[0], gT[1]),
                                (step.dX, (step.Dr, step.Drs), (step.Wc, step.Wcs), gT[2], gT[1]),
                                (step.dW, (step.Dc, step.Dcs), (step.Xc, step.Xcs), gT[2], gT[0])):
            R = oracle.gemm(_u8(A[0]), _u8(A[1]), Ta, _u8(B[0]), _u8(B[1]), Tb)
            check_gemm_bf16(C.float().cpu().numpy().astype(np.float64), R)
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def test_rebiased_step_falls_back_to_the_emulated_step_exactly():
    """A W whose block scales span more than the per-tensor window (one
    16 x 16 tile 2^-24 of the rest, so a row block and a column block):
    both rebiased GEMMs' flags are set, the native
    launches write nothing and the emulated ones run -- Y, dX and dW equal
    the all-emulated step's bit for bit; with W back in range both flags
    clear and the results stay within the BF16 bound of the emulated step."""
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    from fp4_block_scaled_bf16_gb300.linear_step import LinearStep

    dev = torch.device("cuda")
    xb = workloads.activations(TOK, HID, 7)
    wf = workloads.bf16_bits_to_f32(workloads.weights(OUT, HID, 8))
    db = workloads.gradients(TOK, OUT, 9)
    for tiny, want in ((True, [True, True]), (False, [False, False])):
        w = wf.copy()
        if tiny:
            w[0:16, 16:32] *= np.float32(2.0 ** -24)
        wb = workloads.f32_to_bf16_bits(w)
        X = workloads.to_torch_bf16(xb).to(dev)
        W = workloads.to_torch_bf16(wb).to(dev)
        dY = workloads.to_torch_bf16(db).to(dev)
        fast = LinearStep(X, W, dY, seed=7, rebias=True)
        ref = LinearStep(X, W, dY, seed=7)
        fast.run_overlapped(periodic=True)
        ref.run_overlapped(periodic=True)
        torch.cuda.synchronize()
        assert fast.fallbacks() == want
        for a, b in ((fast.Y, ref.Y), (fast.dX, ref.dX), (fast.dW, ref.dW)):
            if tiny:
                assert torch.equal(a, b)
            else:
                R = b.float().cpu().numpy().astype(np.float64)
                check_gemm_bf16(a.float().cpu().numpy().astype(np.float64), R)
        assert torch.equal(fast.dW, ref.dW)   # wgrad is emulated in both
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def test_full_size_step_fallback_is_the_emulated_step():
    """The 8B-class step (8192 tokens, 4096 -> 16384) with one 16 x 16 tile of
    W 2^-24 of the rest: both rebiased GEMMs fall back on the device and the
    step's Y, dX, dW equal the all-emulated step's bit for bit (every cluster
    of both launches took the same decision)."""
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    from fp4_block_scaled_bf16_gb300.linear_step import LinearStep

    dev = torch.device("cuda")
    X, Wb = workloads.fprop_operands()
    w = workloads.bf16_bits_to_f32(Wb)
    w[4096:4112, 1024:1040] *= np.float32(2.0 ** -24)
    Xd = workloads.to_torch_bf16(X).to(dev)
    Wd = workloads.to_torch_bf16(workloads.f32_to_bf16_bits(w)).to(dev)
    Dd = workloads.to_torch_bf16(workloads.backward_gradient()).to(dev)
    fast = LinearStep(Xd, Wd, Dd, seed=7, rebias=True)
    ref = LinearStep(Xd, Wd, Dd, seed=7)
    for _ in range(2):
        fast.run_overlapped(periodic=True)
        ref.run_overlapped(periodic=True)
    torch.cuda.synchronize()
    assert fast.fallbacks() == [True, True]
    for a, b in ((fast.Y, ref.Y), (fast.dX, ref.dX), (fast.dW, ref.dW)):
        assert torch.equal(a, b)
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def test_two_steps_on_two_caller_streams():
    """Two rebiased steps (separate inputs, buffers and internal streams)
    issued from two caller streams at once give the results each gives
    alone."""
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    from fp4_block_scaled_bf16_gb300.linear_step import LinearStep

    dev = torch.device("cuda")
    steps = []
    for k in range(2):
        X = workloads.to_torch_bf16(workloads.activations(TOK, HID, 50 + k)).to(dev)
        W = workloads.to_torch_bf16(workloads.weights(OUT, HID, 60 + k)).to(dev)
        dY = workloads.to_torch_bf16(workloads.gradients(TOK, OUT, 70 + k)).to(dev)
        steps.append(LinearStep(X, W, dY, seed=7, rebias=True))
    alone = []
    for st in steps:
        st.run_overlapped()
        torch.cuda.synchronize()
        alone.append([t.clone() for t in (st.Y, st.dX, st.dW)])
    callers = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        for st, cs in zip(steps, callers):
            with torch.cuda.stream(cs):
                st.run_overlapped()
    torch.cuda.synchronize()
    for st, ref in zip(steps, alone):
        for a, b in zip((st.Y, st.dX, st.dW), ref):
            assert torch.equal(a, b)
    assert fp4q.fp4q_get_device_status() == fp4q.OK


def test_wgrad_through_the_native_path_when_it_fits():
    """rebias_wgrad: wgrad's A operand (dY column-wise) in two windows per
    row.  Gradients whose per-token magnitudes stay within a decade fit; with
    one block of 16 tokens 2^-20 smaller every row needs the low window and
    still fits (the bench's ten-decade gradients span up to 20 binades per row
    at 8192 tokens) -- dW within the BF16 bound of the oracle's UE5M3
    contraction, flag clear; 2^-30 smaller lies below both windows, wgrad falls
    back and dW equals the all-emulated step's bit for bit."""
    from fp4_block_scaled_bf16_gb300 import build
    build.build()
    from fp4_block_scaled_bf16_gb300 import fp4q
    from fp4_block_scaled_bf16_gb300.linear_step import LinearStep

    dev = torch.device("cuda")
    X = workloads.to_torch_bf16(workloads.activations(TOK, HID, 81)).to(dev)
    W = workloads.to_torch_bf16(workloads.weights(OUT, HID, 82)).to(dev)
    for tiny, want_one, want_fall in ((None, True, False), (-20, False, False), (-30, False, True)):
        g = workloads.bf16_bits_to_f32(workloads.gradients(TOK, OUT, 83, -1.0, 0.0))
        if tiny is not None:
            g[32:48] *= np.float32(2.0 ** tiny)
        dY = workloads.to_torch_bf16(workloads.f32_to_bf16_bits(g)).to(dev)
        fast = LinearStep(X, W, dY, seed=7, rebias=True, rebias_wgrad=True)
        ref = LinearStep(X, W, dY, seed=7)
        fast.run_overlapped()
        ref.run_overlapped()
        torch.cuda.synchronize()
        fell = fast.fallbacks()
        dcs = _u8(fast.Dcs)
        assert oracle.rebias_scales(dcs, True)[2] == want_one
        assert dcs[:, 2].all()                                   # the small block's codes are not zero
        fits = oracle.rebias_scales2(dcs)[4] and oracle.rebias_scales(_u8(fast.Xcs), False)[2]
        assert fell[2] == (not fits) == want_fall, (tiny, fell)
        assert fell[:2] == [False, False]
        if want_fall:
            assert torch.equal(fast.dW, ref.dW)
        else:
            TD, TX = float(fast.T[2].item()), float(fast.T[0].item())
            R = oracle.gemm(_u8(fast.Dc), _u8(fast.Dcs), TD, _u8(fast.Xc), _u8(fast.Xcs), TX)
            check_gemm_bf16(fast.dW.float().cpu().numpy().astype(np.float64), R)
    assert fp4q.fp4q_get_device_status() == fp4q.OK


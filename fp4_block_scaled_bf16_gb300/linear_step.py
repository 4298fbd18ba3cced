"""One internal linear layer's training step on the block-scaled FP4 path of
"UE5M3 FP4 Block Scaling for Stable Language Model Pretraining" (Abstract):
every operand of the three training GEMMs is an E2M1 payload with UE5M3
block-16 scales under an FP32 tensor scale, gradients rounded
stochastically.

  fprop  Y  = X W^T    X row-wise, W row-wise         (round to nearest even)
  dgrad  dX = dY W     dY row-wise (SR), W column-wise
  wgrad  dW = dY^T X   dY column-wise (SR), X column-wise

X [tokens, in], W [out, in] and dY [tokens, out] are each quantised once on
both axes (one read).  Two tensor-scale policies:
  current  -- an amax pass and a tensor scale before every quantisation (the
              TE recipe's current scaling);
  periodic -- the method's policy: one PeriodicScaler per tensor, T refreshed
              every `period` steps from the amax the quantiser fused into the
              previous step's quantisation, so no amax pass runs after the
              first step.

With `native=True` the operands carry UE4M3 scales and the three GEMMs run
on the tensor cores' block-scaled MMA (fp4q_gemm_nvfp4) -- the native NVFP4
execution the page ablates against; otherwise the GEMMs are the emulated
block-scaled ones (fp4q_gemm) for the chosen scale format.

With `rebias=True` (UE5M3 only) fprop and dgrad compute the same UE5M3 GEMMs
on the block-scaled MMA: the A operand's scale codes are rebiased per row and
B's per tensor to UE4M3 codes times powers of two (fp4q_rebias_scales), the
native kernel applies the factors (fp4q_gemm_nvfp4_rebiased), and the
emulated kernel (fp4q_gemm_if) is launched after it and runs only if some
group spanned more than the 14 binades UE4M3 holds -- decided on the device,
no host read.  wgrad stays emulated by default: its A operand is dY
column-wise, each row running over the batch's tokens, whose gradient
magnitudes can differ by many more binades than that (in the bench's inputs
they span ten decades).  `rebias_wgrad=True` sends it to the block-scaled MMA
as well, with A's codes in two 14-binade windows per row
(fp4q_rebias_scales_two_windows: 28 binades under each row's largest scale)
multiplied into two accumulators (fp4q_gemm_nvfp4_two_windows), and the same
exact fallback when a code lies below both windows.

Every launch goes through libfp4q.so; buffers are allocated once here with
torch and reused by every step.
"""
from __future__ import annotations

import torch

from . import fp4q as _fp4q
from .periodic import PeriodicScaler


class LinearStep:
    def __init__(self, X: torch.Tensor, W: torch.Tensor, dY: torch.Tensor, seed: int = 7,
                 period: int = 16, fmt: int = _fp4q.UE5M3, native: bool = False, rebias: bool = False,
                 rebias_wgrad: bool = False, lib=None):
        q = self.q = lib if lib is not None else _fp4q
        if native and fmt != q.UE4M3:
            raise ValueError("the native block-scaled MMA takes UE4M3 scales (fmt=UE4M3)")
        if rebias and (native or fmt != q.UE5M3):
            raise ValueError("rebias re-expresses UE5M3 scales (fmt=UE5M3, native=False)")
        if rebias_wgrad and not rebias:
            raise ValueError("rebias_wgrad needs rebias=True")
        self.native = native
        tokens, hid = X.shape
        out = W.shape[0]
        if W.shape[1] != hid or tuple(dY.shape) != (tokens, out):
            raise ValueError(f"shapes do not form a linear: X {tuple(X.shape)}, W {tuple(W.shape)}, "
                             f"dY {tuple(dY.shape)}")
        self.dims = (tokens, hid, out)
        self.seed, self.fmt = seed, fmt
        dev = X.device
        u8 = dict(dtype=torch.uint8, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.X, self.W, self.dY = X, W, dY
        self.amax = torch.zeros(3, **f32)
        self.T = torch.zeros(3, **f32)
        self.Xr, self.Xrs = torch.empty((tokens, hid // 2), **u8), torch.empty((tokens, hid // 16), **u8)
        self.Xc, self.Xcs = torch.empty((hid, tokens // 2), **u8), torch.empty((hid, tokens // 16), **u8)
        self.Wr, self.Wrs = torch.empty((out, hid // 2), **u8), torch.empty((out, hid // 16), **u8)
        self.Wc, self.Wcs = torch.empty((hid, out // 2), **u8), torch.empty((hid, out // 16), **u8)
        self.Dr, self.Drs = torch.empty((tokens, out // 2), **u8), torch.empty((tokens, out // 16), **u8)
        self.Dc, self.Dcs = torch.empty((out, tokens // 2), **u8), torch.empty((out, tokens // 16), **u8)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.Y = torch.empty((tokens, out), **bf)
        self.dX = torch.empty((tokens, hid), **bf)
        self.dW = torch.empty((out, hid), **bf)
        # fprop (A = X rows, B = W rows), dgrad (A = dY rows, B = W columns)
        # and, optionally, wgrad (A = dY columns, B = X columns) on the
        # native MMA: rebiased codes, factors and a fallback flag each (wgrad:
        # A's codes and factors in two windows); a GEMM whose K is not a
        # multiple of 256 stays emulated
        ngemms = 3 if rebias_wgrad else 2
        self.rb = [None] * 3
        self.nofit = torch.zeros(ngemms, dtype=torch.int32, device=dev)
        if rebias:
            shapes = ((tokens, out, hid), (tokens, hid, out), (out, hid, tokens))[:ngemms]
            for g, (m, n, k) in enumerate(shapes):
                if k % 256:
                    continue
                a = (torch.empty((m, k // 16), **u8), torch.empty(m, **f32))
                if g == 2:
                    a = (a[0], torch.empty((m, k // 16), **u8), a[1], torch.empty(m, **f32))
                self.rb[g] = a + (torch.empty((n, k // 16), **u8), torch.empty(1, **f32), self.nofit[g:g + 1])
        self.scalers = [PeriodicScaler(period, fmt, device=dev, lib=q) for _ in range(3)]
        self.launches = 0
        # run_overlapped's streams, by priority: X, W and fprop highest, dY
        # and dgrad one step lower, wgrad (the long emulated GEMM, whose CTAs
        # fill what the others leave) and the emulated fallbacks of fprop and
        # dgrad (which return at once unless a group did not fit) lowest --
        # the fallbacks' CTAs then take SMs the step's kernels leave idle
        # instead of queueing between them
        least, greatest = torch.cuda.Stream.priority_range()
        second = min(greatest + 1, least)
        self.main = torch.cuda.Stream(device=dev, priority=greatest)
        self.side = torch.cuda.Stream(device=dev, priority=second)
        self.side2 = torch.cuda.Stream(device=dev, priority=least)
        self.fallback = torch.cuda.Stream(device=dev, priority=least)
        self.ev_start, self.ev_xw, self.ev_side, self.ev_dq, self.ev_side2, self.ev_main = (
            torch.cuda.Event() for _ in range(6))
        self.ev_rb = [torch.cuda.Event(), torch.cuda.Event()]
        self.ev_fb = [torch.cuda.Event(), torch.cuda.Event()]

    # ------------------------------------------------------------ pieces
    def _scale(self, i: int, x: torch.Tensor, periodic: bool):
        """(T, fused-amax output or None) for tensor i, launched on the current stream."""
        q = self.q
        if periodic:
            sc = self.scalers[i]
            before = sc.step % sc.period == 0
            T = sc.scale_for(x)
            self.launches += (2 if sc.step == 0 else 1) if before else 0
            return T, sc.last_amax
        T, A = self.T[i:i + 1], self.amax[i:i + 1]
        q.fp4q_amax(x, A)
        q.fp4q_tensor_scale(A, self.fmt, 1.0, T)
        self.launches += 2
        return T, None

    def _quantize(self, i, x, T, amax, rnd, outs):
        self.q.fp4q_quantize(x, self.q.AXIS_BOTH, self.fmt, T, rnd, self.seed if rnd else 0, *outs,
                             None, amax)
        self.launches += 1
        if amax is not None:
            self.scalers[i].advance()

    def _gemm(self, A, B, M, N, K, out, rb=None, g=None):
        """One GEMM on the current stream.  Through rebiased codes (rb: one
        window per A row, or two), the emulated fallback goes on the
        low-priority stream when g (0 fprop, 1 dgrad) is given -- after the
        rebias launches, joined back before anything later on the current
        stream -- else in line."""
        q = self.q
        if self.native:
            q.fp4q_gemm_nvfp4(*A, *B, M, N, K, out)
        elif rb is not None:
            b4, fb, flag = rb[-3:]
            flag.zero_()
            if len(rb) == 7:   # A's codes in two windows
                ah, al, fh, fl = rb[:4]
                q.fp4q_rebias_scales_two_windows(A[1], M, K // 16, ah, al, fh, fl, flag)
                native = lambda: q.fp4q_gemm_nvfp4_two_windows(A[0], ah, al, fh, A[2], B[0], b4, fb, B[2], M, N,
                                                               K, flag, out)
            else:
                a4, fa = rb[:2]
                q.fp4q_rebias_scales(A[1], M, K // 16, True, a4, fa, flag)
                native = lambda: q.fp4q_gemm_nvfp4_rebiased(A[0], a4, fa, A[2], B[0], b4, fb, B[2], M, N, K, flag,
                                                            out)
            q.fp4q_rebias_scales(B[1], N, K // 16, False, b4, fb, flag)
            if g is None:
                native()
                q.fp4q_gemm_if(*A, *B, M, N, K, self.fmt, flag, out)
            else:
                cur = torch.cuda.current_stream()
                self.ev_rb[g].record(cur)
                native()
                self.fallback.wait_event(self.ev_rb[g])
                with torch.cuda.stream(self.fallback):
                    q.fp4q_gemm_if(*A, *B, M, N, K, self.fmt, flag, out)
                    self.ev_fb[g].record(self.fallback)
                cur.wait_event(self.ev_fb[g])   # exactly one of the two wrote `out`
            self.launches += 3
        else:
            q.fp4q_gemm(*A, *B, M, N, K, self.fmt, out)
        self.launches += 1

    def fallbacks(self):
        """Whether fprop, dgrad (and wgrad, with rebias_wgrad) each fell back
        to the emulated GEMM on the last step (reads the device flags;
        synchronises)."""
        return [bool(v) for v in self.nofit.tolist()]

    def tensor_scales(self, periodic: bool):
        """The device T of X, W and dY that the last step used."""
        if periodic:
            return [sc.T for sc in self.scalers]
        return [self.T[i:i + 1] for i in range(3)]

    # ------------------------------------------------------------ steps
    def run(self, ev=None, periodic: bool = False):
        """The step on the current stream, one kernel after another; with
        `ev` (eight timing events) an event is recorded before the scales,
        before each quantisation and GEMM, and at the end."""
        q = self.q
        tokens, hid, out = self.dims
        rec = (lambda k: ev[k].record()) if ev else (lambda k: None)
        rec(0)
        sc = [self._scale(i, x, periodic) for i, x in enumerate((self.X, self.W, self.dY))]
        (TX, aX), (TW, aW), (TD, aD) = sc
        rec(1)
        self._quantize(0, self.X, TX, aX, q.RNE, (self.Xr, self.Xrs, self.Xc, self.Xcs))
        rec(2)
        self._quantize(1, self.W, TW, aW, q.RNE, (self.Wr, self.Wrs, self.Wc, self.Wcs))
        rec(3)
        self._quantize(2, self.dY, TD, aD, q.SR, (self.Dr, self.Drs, self.Dc, self.Dcs))
        rec(4)
        self._gemm((self.Xr, self.Xrs, TX), (self.Wr, self.Wrs, TW), tokens, out, hid, self.Y, self.rb[0])
        rec(5)
        self._gemm((self.Dr, self.Drs, TD), (self.Wc, self.Wcs, TW), tokens, hid, out, self.dX, self.rb[1])
        rec(6)
        self._gemm((self.Dc, self.Dcs, TD), (self.Xc, self.Xcs, TX), out, hid, tokens, self.dW, self.rb[2])
        rec(7)
        return self

    def run_overlapped(self, periodic: bool = False):
        """The same launches on three streams, in the step's dependency
        order: one takes X and W (scales, dual-axis RNE quantisation) and
        fprop; a side stream takes dY's scale and dual-axis SR quantisation
        at the same time, then dgrad once W is quantised; a second side
        stream runs wgrad once dY and X are quantised, so that the three GEMMs
        fill one another's last waves (priorities and fprop's and dgrad's
        emulated fallbacks: see the constructor).  All start after the
        caller's stream reaches the step, and the caller's stream waits for
        all of them at the end, so a step ends when all of its work is done
        and the next one starts from a clean slate."""
        q, torch_ = self.q, torch
        tokens, hid, out = self.dims
        caller = torch_.cuda.current_stream()
        main = self.main
        self.ev_start.record(caller)
        main.wait_event(self.ev_start)
        with torch_.cuda.stream(main):
            TX, aX = self._scale(0, self.X, periodic)
            TW, aW = self._scale(1, self.W, periodic)
            self._quantize(0, self.X, TX, aX, q.RNE, (self.Xr, self.Xrs, self.Xc, self.Xcs))
            self._quantize(1, self.W, TW, aW, q.RNE, (self.Wr, self.Wrs, self.Wc, self.Wcs))
            self.ev_xw.record(main)
        with torch_.cuda.stream(self.side):
            self.side.wait_event(self.ev_start)
            TD, aD = self._scale(2, self.dY, periodic)
            self._quantize(2, self.dY, TD, aD, q.SR, (self.Dr, self.Drs, self.Dc, self.Dcs))
            self.ev_dq.record(self.side)
            self.side.wait_event(self.ev_xw)
            self._gemm((self.Dr, self.Drs, TD), (self.Wc, self.Wcs, TW), tokens, hid, out, self.dX, self.rb[1], 1)
            self.ev_side.record(self.side)
        with torch_.cuda.stream(self.side2):
            self.side2.wait_event(self.ev_dq)
            self.side2.wait_event(self.ev_xw)
            self._gemm((self.Dc, self.Dcs, TD), (self.Xc, self.Xcs, TX), out, hid, tokens, self.dW, self.rb[2])
            self.ev_side2.record(self.side2)
        with torch_.cuda.stream(main):
            self._gemm((self.Xr, self.Xrs, TX), (self.Wr, self.Wrs, TW), tokens, out, hid, self.Y, self.rb[0], 0)
            self.ev_main.record(main)
        caller.wait_event(self.ev_main)
        caller.wait_event(self.ev_side)
        caller.wait_event(self.ev_side2)
        return self

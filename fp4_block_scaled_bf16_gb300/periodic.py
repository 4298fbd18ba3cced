"""Periodic tensor scaling: the tensor-scale policy of "UE5M3 FP4 Block
Scaling for Stable Language Model Pretraining" (Abstract: UE5M3's wider range
lets the FP32 tensor scale be refreshed periodically instead of from a fresh
amax pass before every quantisation).

Policy (the oracle's `PeriodicScaler` states the same reading): the tensor
scale T is refreshed every `period` quantisations from the amax of the last
quantised tensor -- the quantiser's fused by-product, so no extra pass --
and the first refresh uses an explicit amax pass over the first tensor.  All
of it stays on the device: T and the last amax are device scalars, and a
refresh is one `fp4q_tensor_scale` launch.

The state ({T, last amax, step}) is saved and restored with `state_dict` /
`load_state_dict`, so that a resumed run refreshes on the same steps with the
same scale.

Every launch goes through libfp4q.so (the `fp4q` binding); the `lib`
argument exists only so that tests can drive the schedule through a stand-in
with the same interface.
"""
from __future__ import annotations

import torch

from . import fp4q as _fp4q


class PeriodicScaler:
    def __init__(self, period: int = 16, fmt: int = _fp4q.UE5M3, headroom: float = 1.0,
                 device="cuda", lib=None):
        if period < 1:
            raise ValueError("period must be >= 1")
        self.lib = lib if lib is not None else _fp4q
        self.period, self.fmt, self.headroom = int(period), int(fmt), float(headroom)
        self.T = torch.ones(1, dtype=torch.float32, device=device)
        self.last_amax = torch.zeros(1, dtype=torch.float32, device=device)
        self.have_amax = False
        self.step = 0

    def scale_for(self, x: torch.Tensor) -> torch.Tensor:
        """The device tensor scale for the next quantisation, refreshed first
        when that quantisation is on a period boundary: from an explicit amax
        pass over x on the very first call, otherwise from the amax the
        previous quantisation left in `last_amax`.  The caller quantises with
        the returned T, has the quantiser write its fused amax into
        `last_amax`, then calls `advance()`.  Launches go to the current
        stream."""
        lib = self.lib
        if self.step % self.period == 0:
            if not self.have_amax:
                lib.fp4q_amax(x, self.last_amax)
                self.have_amax = True
            lib.fp4q_tensor_scale(self.last_amax, self.fmt, self.headroom, self.T)
        return self.T

    def advance(self) -> None:
        """Records that a quantisation with the current T has written its amax
        into `last_amax`."""
        self.have_amax = True
        self.step += 1

    def quantize(self, x: torch.Tensor, axis: int = _fp4q.AXIS_ROW, rnd: int = _fp4q.RNE, seed: int = 0,
                 stats: bool = False):
        """Quantises x with the current tensor scale (refreshed first on
        every `period`-th call) and records its amax for the next refresh.
        The returned T is a copy of the scale used, unaffected by later
        refreshes."""
        T = self.scale_for(x).clone()
        q = self.lib.quantize(x, axis, T, self.fmt, rnd, seed, stats=stats, want_amax=True)
        self.last_amax.copy_(q.amax)
        self.advance()
        return q

    def state_dict(self) -> dict:
        return {"period": self.period, "fmt": self.fmt, "headroom": self.headroom,
                "T": float(self.T.item()), "last_amax": float(self.last_amax.item()),
                "have_amax": self.have_amax, "step": self.step}

    def load_state_dict(self, d: dict) -> None:
        if (int(d["period"]), int(d["fmt"]), float(d["headroom"])) != (self.period, self.fmt, self.headroom):
            raise ValueError("state was saved by a scaler with another period, format or headroom")
        self.T.fill_(float(d["T"]))
        self.last_amax.fill_(float(d["last_amax"]))
        self.have_amax = bool(d["have_amax"])
        self.step = int(d["step"])

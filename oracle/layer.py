"""Elementwise steps of the expert FFN and delayed scaling (TEST
INFRASTRUCTURE ONLY).

* SwiGLU between the two grouped GEMMs (Mixtral / Llama4 experts named on
  Megatron-LM issue #1152 and pytorch/ao PR #2275): h = silu(g) * u with
  silu(g) = g / (1 + exp(-g)); its derivative gives
  dG = dH * u * sigma(g) * (1 + g (1 - sigma(g))) and dU = dH * silu(g).
  The gate occupies columns [0, F) of the gate/up GEMM output, the up
  projection columns [F, 2F).
* Delayed scaling ("--fp8-amax-compute-algo max --fp8-amax-history-len 1024",
  Megatron-LM issue #1152, repro steps): each tensor role keeps a ring of the
  last 1024 amax values; a step quantises with the scale derived from the
  ring's maximum over earlier steps, then records its own amax.
"""
from __future__ import annotations

import numpy as np

from .formats import FORMATS, round_to_bf16


def sigmoid(g):
    g = np.asarray(g, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-g))


def silu(g):
    g = np.asarray(g, dtype=np.float64)
    return g * sigmoid(g)


def swiglu(gu, F):
    """gu [R, 2F] -> h [R, F] (float64, not rounded)."""
    gu = np.asarray(gu, dtype=np.float64)
    return silu(gu[:, :F]) * gu[:, F:2 * F]


def dswiglu(dh, gu, F):
    """Returns d(gu) [R, 2F] = [dG | dU] (float64)."""
    gu = np.asarray(gu, dtype=np.float64)
    dh = np.asarray(dh, dtype=np.float64)
    g, u = gu[:, :F], gu[:, F:2 * F]
    s = sigmoid(g)
    dg = dh * u * s * (1.0 + g * (1.0 - s))
    du = dh * g * s
    return np.concatenate([dg, du], axis=1)


class DelayedScaling:
    """Amax history ring of one tensor role and its current scale.

    Starts with a zero ring and scale 1. ``update(amax)`` writes the amax of
    the step into the ring, takes the maximum over the ring and, if that is
    positive and finite, sets scale = float32(max_finite / max) (margin 0);
    otherwise the scale is kept."""

    def __init__(self, fmt="e4m3", length=1024):
        self.fmt = FORMATS[fmt] if isinstance(fmt, str) else fmt
        self.ring = np.zeros(length, dtype=np.float32)
        self.head = 0
        self.scale = np.float32(1.0)

    def update(self, amax):
        self.ring[self.head] = np.float32(amax)
        self.head = (self.head + 1) % len(self.ring)
        m = np.float32(np.max(self.ring))
        if np.isfinite(m) and m > 0:
            self.scale = np.float32(np.float32(self.fmt.max_finite) / m)
        return self.scale


def to_bf16(x):
    return round_to_bf16(x)

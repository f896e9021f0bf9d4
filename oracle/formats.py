"""Bit-level number formats of the oracle (TEST INFRASTRUCTURE ONLY).

Formats named by the pages: e4m3 and e5m2 ("--fp8-format hybrid", Megatron-LM
issue #1152, repro steps), MXFP8 and NVFP4/e2m1 (Megatron-LM PR #5487,
coverage matrix: ``fp8="e4m3" fp8_recipe="mxfp8"``, ``fp4="e2m1"
fp4_recipe="nvfp4"``). The bit layouts are not on the pages; they follow the
OCP OFP8 specification (E4M3: bias 7, no infinity, S.1111.111 is NaN;
E5M2: bias 15, IEEE-style infinities and NaNs) and OCP MX v1.0 (E2M1: bias 1,
no infinity or NaN; E8M0: value 2^(c-127), 0xFF is NaN).

Decoding is the formula of the spec applied to the bit fields. Encoding is the
definition of round-to-nearest-even with saturation ("satfinite"): the nearest
representable finite value, a tie going to the code whose last mantissa bit is
0, anything of magnitude above the largest finite value (infinity included)
giving that value, the sign kept (a negative value that rounds to zero gives
the negative-zero code). It is written as a search over the table of decoded
values, so that it is correct by construction; the tests pin it against the
spec's closed forms and an independent library cast.

All arithmetic is exact: inputs are float32 or bfloat16 values held in float64.
"""
from __future__ import annotations

import numpy as np


class Format:
    """A small float format: sign bit (optional), ``ebits`` exponent bits with
    ``bias``, ``mbits`` mantissa bits, and its special-code rules."""

    def __init__(self, name, ebits, mbits, bias, signed, kind):
        self.name = name
        self.ebits = ebits
        self.mbits = mbits
        self.bias = bias
        self.signed = signed
        self.kind = kind  # "ofp8_e4m3", "ieee", "finite"
        self.nbits = (1 if signed else 0) + ebits + mbits
        self.ncodes = 1 << self.nbits
        self.sign_bit = (1 << (ebits + mbits)) if signed else 0
        vals = np.array([self._decode_one(c) for c in range(self.ncodes)], dtype=np.float64)
        self.values = vals
        pos = [c for c in range(self.ncodes)
               if (c & self.sign_bit) == 0 and np.isfinite(vals[c])]
        # positive finite values are increasing in the code for these formats
        self.pos_codes = np.array(pos, dtype=np.int64)
        self.pos_values = vals[self.pos_codes]
        assert np.all(np.diff(self.pos_values) > 0)
        self.max_finite = float(self.pos_values[-1])
        self.max_code = int(self.pos_codes[-1])
        nan = [c for c in range(self.ncodes) if np.isnan(vals[c]) and (c & self.sign_bit) == 0]
        self.nan_code = nan[-1] if nan else None

    def _decode_one(self, c):
        s = (c >> (self.ebits + self.mbits)) & 1 if self.signed else 0
        e = (c >> self.mbits) & ((1 << self.ebits) - 1)
        m = c & ((1 << self.mbits) - 1)
        emask = (1 << self.ebits) - 1
        if self.kind == "ofp8_e4m3" and e == emask and m == (1 << self.mbits) - 1:
            return float("nan")
        if self.kind == "ieee" and e == emask:
            return float("nan") if m else (-np.inf if s else np.inf)
        if e == 0:
            mag = np.ldexp(m / (1 << self.mbits), 1 - self.bias)
        else:
            mag = np.ldexp(1.0 + m / (1 << self.mbits), e - self.bias)
        return -mag if s else mag

    def __repr__(self):
        return f"Format({self.name})"


E4M3 = Format("e4m3", 4, 3, 7, True, "ofp8_e4m3")
E5M2 = Format("e5m2", 5, 2, 15, True, "ieee")
E2M1 = Format("e2m1", 2, 1, 1, True, "finite")
# NVFP4 block scales: e4m3 restricted to the non-negative codes.
UE4M3 = Format("ue4m3", 4, 3, 7, False, "ofp8_e4m3")

FORMATS = {"e4m3": E4M3, "e5m2": E5M2, "e2m1": E2M1, "ue4m3": UE4M3}

# largest-power-of-two exponent of the largest finite value ("emax_elem" of
# OCP MX v1.0): 448 = 1.75*2^8, 57344 = 1.75*2^15, 6 = 1.5*2^2
EMAX = {"e4m3": 8, "e5m2": 15, "e2m1": 2}


def decode(codes, fmt: Format) -> np.ndarray:
    """Codes (any integer array) -> exact values as float64."""
    codes = np.asarray(codes).astype(np.int64)
    return fmt.values[codes]


def encode(x, fmt: Format) -> np.ndarray:
    """Round-to-nearest-even, saturating cast of float values to ``fmt`` codes.

    ``x`` must hold values exactly representable in float64 (float32 or bf16
    inputs). NaN gives the format's NaN code (E2M1 has none: ValueError).
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    if nan.any() and fmt.nan_code is None:
        raise ValueError(f"{fmt.name} has no NaN code")
    if not fmt.signed and np.any(neg & ~nan & (a > 0)):
        raise ValueError(f"{fmt.name} is unsigned")
    vals, codes = fmt.pos_values, fmt.pos_codes
    a_cl = np.where(nan, 0.0, np.minimum(a, fmt.max_finite))
    # vals[i] <= a < vals[i+1]
    i = np.searchsorted(vals, a_cl, side="right") - 1
    i = np.clip(i, 0, len(vals) - 1)
    j = np.minimum(i + 1, len(vals) - 1)
    lo, hi = vals[i], vals[j]
    mid = (lo + hi) / 2.0  # exact: lo and hi carry at most mbits+1 significant bits
    pick_hi = (a_cl > mid) | ((a_cl == mid) & (codes[i] & 1 == 1))
    pick_hi &= j != i
    out = np.where(pick_hi, codes[j], codes[i])
    if fmt.signed:
        out = np.where(neg, out | fmt.sign_bit, out)
    if fmt.nan_code is not None:
        out = np.where(nan, fmt.nan_code, out)
    return out.astype(np.uint8)


# ---------------------------------------------------------------------------
# E8M0 (OCP MX v1.0 shared scale): value 2^(c-127); code 255 is NaN.

def e8m0_decode(codes) -> np.ndarray:
    c = np.asarray(codes).astype(np.int64)
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, v)


# ---------------------------------------------------------------------------
# bfloat16 and float32 helpers of the oracle.

def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """float64 -> nearest bfloat16 value (ties to even, overflow to inf), as
    float64. Rounds the significand once, straight from float64."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    xf = x[fin]
    _, e = np.frexp(xf)                  # xf = m * 2^e, 0.5 <= |m| < 1
    q = np.maximum(e - 8, -133)          # 8 significant bits; subnormal quantum 2^-133
    n = np.rint(np.ldexp(xf, -q))        # exact scaling, then ties-to-even
    y = np.ldexp(n, q)
    bf16_max = np.ldexp(2.0 - 2.0 ** -7, 127)
    y = np.where(np.abs(y) > bf16_max, np.copysign(np.inf, y), y)
    out[fin] = y
    return out


def f64_to_bf16_bits(x) -> np.ndarray:
    """float64 -> bfloat16 bit patterns (uint16), ties to even."""
    y = round_to_bf16(x).astype(np.float32)   # exact: y is a bf16 value
    return (y.view(np.uint32) >> 16).astype(np.uint16)


def f32(x) -> np.ndarray:
    """Round to float32 (IEEE round-to-nearest-even), returned as float32."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)

"""Pins of the oracle's number formats (CPU only).

Each pin checks the oracle against something other than itself: the constants
the OCP specifications print (tests/golden/ocp_format_constants.txt), the
definition of round-to-nearest-even over every code, and PyTorch's own
float8 casts as an independent implementation.
"""
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ocp_format_constants.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, code, val = line.split()
            rows.append((name, int(code, 16), val))
    return rows


@pytest.mark.parametrize("row", _golden(), ids=lambda r: f"{r[0]}-{r[1]:#x}")
def test_spec_constants(row):
    name, code, val = row
    if name == "e8m0":
        got = float(F.e8m0_decode(code))
    else:
        got = float(F.decode(code, F.FORMATS[name]))
    if val == "nan":
        assert np.isnan(got)
    elif val == "inf":
        assert got == np.inf
    else:
        assert got == float(val)


@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2, F.E2M1, F.UE4M3], ids=str)
def test_roundtrip_every_code(fmt):
    codes = np.arange(fmt.ncodes)
    vals = F.decode(codes, fmt)
    keep = np.isfinite(vals)
    back = F.encode(vals[keep], fmt)
    np.testing.assert_array_equal(back, codes[keep].astype(np.uint8))


@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2, F.E2M1, F.UE4M3], ids=str)
def test_midpoints_go_to_even_code(fmt):
    v, c = fmt.pos_values, fmt.pos_codes
    mid = (v[:-1] + v[1:]) / 2
    got = F.encode(mid, fmt).astype(np.int64)
    want = np.where(c[:-1] % 2 == 0, c[:-1], c[1:])
    np.testing.assert_array_equal(got, want)
    # just below / above a midpoint go to the nearer code
    eps = np.abs(mid) * 2.0 ** -30
    np.testing.assert_array_equal(F.encode(mid - eps, fmt).astype(np.int64), c[:-1])
    np.testing.assert_array_equal(F.encode(mid + eps, fmt).astype(np.int64), c[1:])


@pytest.mark.parametrize("fmt", [F.E4M3, F.E5M2, F.E2M1], ids=str)
def test_saturation_and_sign(fmt):
    m = fmt.max_finite
    big = np.array([m * 1.0001, m * 2, m * 1e6, np.inf])
    assert np.all(F.encode(big, fmt) == fmt.max_code)
    assert np.all(F.encode(-big, fmt) == (fmt.max_code | fmt.sign_bit))
    # a negative value that rounds to zero keeps its sign
    tiny = fmt.pos_values[1] / 4
    assert F.encode(np.array([-tiny]), fmt)[0] == fmt.sign_bit
    assert F.encode(np.array([tiny]), fmt)[0] == 0
    assert F.encode(np.array([-0.0]), fmt)[0] == fmt.sign_bit


def test_e2m1_tie_table():
    # halfway cases of the e2m1 grid {0, .5, 1, 1.5, 2, 3, 4, 6}
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 100.0])
    want = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0])
    np.testing.assert_array_equal(F.decode(F.encode(x, F.E2M1), F.E2M1), want)


def test_nan_codes():
    assert F.encode(np.array([np.nan]), F.E4M3)[0] & 0x7F == 0x7F
    assert np.isnan(F.decode(F.encode(np.array([np.nan]), F.E5M2), F.E5M2)[0])
    with pytest.raises(ValueError):
        F.encode(np.array([np.nan]), F.E2M1)


def _all_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return bits, F.bf16_bits_to_f64(bits)


@pytest.mark.parametrize("name,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_all_bf16_against_torch_cast(name, tdt):
    """Every bf16 bit pattern, clamped to the finite range (PyTorch's casts do
    not saturate), cast by the oracle and by PyTorch's CPU cast."""
    fmt = F.FORMATS[name]
    _, x = _all_bf16()
    x = x[~np.isnan(x)]
    x = np.clip(x, -fmt.max_finite, fmt.max_finite)
    ours = F.encode(x, fmt)
    theirs = torch.from_numpy(x.astype(np.float32)).to(tdt).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, theirs)


def test_random_f32_against_torch_cast():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-20, 12, 200000))).astype(np.float32)
    for fmt, tdt in ((F.E4M3, torch.float8_e4m3fn), (F.E5M2, torch.float8_e5m2)):
        xc = np.clip(x.astype(np.float64), -fmt.max_finite, fmt.max_finite)
        ours = F.encode(xc, fmt)
        theirs = torch.from_numpy(xc.astype(np.float32)).to(tdt).view(torch.uint8).numpy()
        np.testing.assert_array_equal(ours, theirs)


def test_bf16_rounding_against_torch():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(100000) * np.exp2(rng.integers(-140, 120, 100000))).astype(np.float32)
    x = np.concatenate([x, np.array([0.0, -0.0, 3.3895314e38, -3.4e38], dtype=np.float32)])
    ours = F.f64_to_bf16_bits(x.astype(np.float64))
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, theirs)


def test_e8m0_all_codes():
    c = np.arange(255)
    np.testing.assert_array_equal(F.e8m0_decode(c), np.exp2(c.astype(np.float64) - 127))
    assert np.isnan(F.e8m0_decode(255))

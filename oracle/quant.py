"""Block quantisation of the oracle (TEST INFRASTRUCTURE ONLY).

Each function takes its steps in the order the pages and the specs give:
amax over a block, a scale derived from it, a round-to-nearest-even saturating
cast of the scaled values. Inputs are float64 arrays that hold bfloat16 or
float32 values exactly. Scales come back in their natural layout
(``[rows, K / block]``), codes as uint8 (e2m1: packed two per byte).

Sources:
* MXFP8 (32-element blocks, E8M0 power-of-two scales): the "mxfp8" recipe of
  Megatron-LM PR #5487 (coverage matrix); block size and scale format from
  OCP MX v1.0. Two readings of the scale exponent are provided: "rceil" (the
  smallest power of two that keeps the block's amax at or below the format's
  largest value, so no element saturates) and "floor" (OCP MX v1.0:
  floor(log2 amax) - emax_elem).
* Blockwise FP8 with float32 scales, 1x128 for activations and 128x128 for
  weights ("Deepseek FP8 block scaling recipe"; 1x128 forward / 128x1
  backward): TransformerEngine issue #2393, maintainer replies. Missing
  elements of a partial block count as zero (same replies).
* Per-tensor scaling with a caller-given scale (delayed scaling of Megatron-LM
  issue #1152, repro steps).
* NVFP4: e2m1 codes packed two per byte (Megatron-LM PR #5487, review
  comments), 16-element e4m3 block scales and one float32 scale per tensor.
* NVFP4 weights with 16x16 blocks (the NVFP4 primary-weight path of the same
  PR's coverage matrix, where one grouped weight carries row-wise and
  column-wise data): the pages fix no weight block shape. Reading taken here:
  one ue4m3 scale per 16x16 block of each expert's weight, from the block's
  amax by the 1x16 rule, shared by the row-wise and the column-wise copy, so
  the two copies hold the same element codes, transposed.
"""
from __future__ import annotations

import numpy as np

from .formats import (E2M1, E4M3, E5M2, EMAX, FORMATS, UE4M3, decode, encode,
                      e8m0_decode, f32)

FLT_MAX = float(np.finfo(np.float32).max)


def _fmt(fmt):
    return FORMATS[fmt] if isinstance(fmt, str) else fmt


def _pad_cols(x, block):
    """Zero-fill a partial trailing block (TransformerEngine issue #2393:
    missing elements of a block are zero-filled by the quantiser)."""
    M, K = x.shape
    Kp = -(-K // block) * block
    if Kp == K:
        return x
    out = np.zeros((M, Kp), dtype=np.float64)
    out[:, :K] = x
    return out


def block_amax(x, block):
    """max |x| over consecutive blocks of ``block`` elements of each row.
    A NaN anywhere in the block makes the amax NaN."""
    x = _pad_cols(np.asarray(x, dtype=np.float64), block)
    M, K = x.shape
    return np.max(np.abs(x.reshape(M, K // block, block)), axis=2)


# ---------------------------------------------------------------------------
# MXFP8

def mx_scale_exponent(amax, fmt, mode="rceil"):
    """Shared-scale exponent e of a block (the block is stored as x * 2^-e).

    rceil: the smallest integer e with amax <= max_finite * 2^e.
    floor: floor(log2 amax) - emax_elem (OCP MX v1.0).
    amax == 0 gives -127. The result is clamped to [-127, 127]. Returns
    (e as int64, E8M0 code as uint8); a NaN or infinite amax gives code 255.
    """
    fmt = _fmt(fmt)
    emax = EMAX[fmt.name]
    amax = np.asarray(amax, dtype=np.float64)
    fin = np.isfinite(amax)
    pos = fin & (amax > 0)
    safe = np.where(pos, amax, 1.0)
    _, ex = np.frexp(safe)               # safe = m * 2^ex, 0.5 <= m < 1
    e = (ex - 1) - emax                  # floor(log2 amax) - emax
    if mode == "rceil":
        e = np.where(safe > np.ldexp(fmt.max_finite, e), e + 1, e)
    elif mode != "floor":
        raise ValueError(mode)
    e = np.where(pos, e, -127)
    e = np.clip(e, -127, 127).astype(np.int64)
    code = np.where(fin, e + 127, 255).astype(np.uint8)
    return e, code


def quantize_mx(x, fmt="e4m3", mode="rceil", block=32):
    """Row-wise MX quantisation of ``x`` [M, K]: blocks of ``block`` along K.

    Returns codes [M, K] uint8 and E8M0 scale codes [M, ceil(K/block)] uint8.
    Element code = cast(float32(x * 2^-e)); for a NaN/inf block the codes are
    cast(x * NaN).
    """
    fmt = _fmt(fmt)
    x = np.asarray(x, dtype=np.float64)
    M, K = x.shape
    xp = _pad_cols(x, block)
    nb = xp.shape[1] // block
    amax = block_amax(xp, block)
    e, sc = mx_scale_exponent(amax, fmt, mode)
    mult = np.where(sc == 255, np.nan, np.ldexp(1.0, -e))
    y = xp.reshape(M, nb, block) * mult[:, :, None]   # exact in float64
    y = f32(y).astype(np.float64)                      # the float32 product
    codes = encode(y, fmt).reshape(M, nb * block)[:, :K]
    return codes, sc


def dequantize_mx(codes, scales, fmt="e4m3", block=32):
    fmt = _fmt(fmt)
    codes = np.asarray(codes)
    M, K = codes.shape
    v = decode(codes, fmt)
    s = np.repeat(e8m0_decode(scales), block, axis=1)[:, :K]
    return v * s


# ---------------------------------------------------------------------------
# Blockwise FP8 with float32 scales

def blockwise_scale(amax, fmt):
    """s = float32(max_finite / amax) (IEEE division); amax == 0 -> 1;
    an overflowing quotient -> the largest float32."""
    fmt = _fmt(fmt)
    amax = np.asarray(amax, dtype=np.float64)
    a32 = f32(amax)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = np.float32(fmt.max_finite) / np.where(a32 == 0, np.float32(1), a32)
    s = np.where(a32 == 0, np.float32(1.0), s)
    s = np.where(np.isinf(s), np.float32(FLT_MAX), s).astype(np.float32)
    return s


def quantize_block_1x128(x, fmt="e4m3", block=128):
    """1 x block quantisation along K of ``x`` [M, K].

    Returns codes [M, K] uint8 and scale_inv = float32(1 / s) [M, ceil(K/block)].
    Element code = cast(float32(x * s))."""
    fmt = _fmt(fmt)
    x = np.asarray(x, dtype=np.float64)
    M, K = x.shape
    xp = _pad_cols(x, block)
    nb = xp.shape[1] // block
    s = blockwise_scale(block_amax(xp, block), fmt)
    y = f32(xp).reshape(M, nb, block) * s[:, :, None]   # float32 multiply, RN
    codes = encode(y.astype(np.float64), fmt).reshape(M, nb * block)[:, :K]
    scale_inv = (np.float32(1.0) / s).astype(np.float32)
    return codes, scale_inv


def quantize_block_128x128(w, fmt="e4m3", block=128):
    """block x block tile quantisation of a weight ``w`` [N, K].

    Returns codes [N, K] uint8 and scale_inv [ceil(N/block), ceil(K/block)]."""
    fmt = _fmt(fmt)
    w = np.asarray(w, dtype=np.float64)
    N, K = w.shape
    wp = _pad_cols(_pad_cols(w, block).T, block).T      # zero-fill both dims
    nbn, nbk = wp.shape[0] // block, wp.shape[1] // block
    tiles = wp.reshape(nbn, block, nbk, block)
    amax = np.max(np.abs(tiles), axis=(1, 3))
    s = blockwise_scale(amax, fmt)
    y = f32(tiles) * s[:, None, :, None]
    codes = encode(y.astype(np.float64), fmt).reshape(nbn * block, nbk * block)[:N, :K]
    scale_inv = (np.float32(1.0) / s).astype(np.float32)
    return codes, scale_inv


def dequantize_block_1x128(codes, scale_inv, fmt="e4m3", block=128):
    """value = decode(code) * scale_inv of the code's 1 x block block."""
    fmt = _fmt(fmt)
    M, K = codes.shape
    return decode(codes, fmt) * np.repeat(scale_inv.astype(np.float64), block, axis=1)[:, :K]


def dequantize_block_128x128(codes, scale_inv, fmt="e4m3", block=128):
    """value = decode(code) * scale_inv of the code's block x block tile."""
    fmt = _fmt(fmt)
    N, K = codes.shape
    s = np.repeat(np.repeat(scale_inv.astype(np.float64), block, axis=0), block, axis=1)
    return decode(codes, fmt) * s[:N, :K]


# ---------------------------------------------------------------------------
# Per-tensor scaling

def quantize_tensor(x, scale, fmt="e4m3"):
    """code = cast(float32(x * scale)); returns (codes, amax of x)."""
    fmt = _fmt(fmt)
    x = np.asarray(x, dtype=np.float64)
    y = f32(x) * np.float32(scale)
    codes = encode(y.astype(np.float64), fmt)
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    return codes, amax


def dequantize_tensor(codes, scale, fmt="e4m3"):
    """value = decode(code) / s, with s the float32 scale the codes were cast
    with (float64 division)."""
    return decode(codes, _fmt(fmt)) / np.float64(np.float32(scale))


# ---------------------------------------------------------------------------
# NVFP4

NVFP4_BLOCK = 16


def nvfp4_global_scale(amax_tensor):
    """s_g = float32(6 * 448 / amax_tensor); amax 0 -> 1; overflow -> FLT_MAX."""
    a = np.float32(amax_tensor)
    if a == 0:
        return np.float32(1.0)
    s = np.float32(6.0 * 448.0) / a
    return np.float32(FLT_MAX) if np.isinf(s) else np.float32(s)


def quantize_nvfp4(x, s_g):
    """NVFP4 quantisation of ``x`` [M, K] with global scale ``s_g``.

    Block scale code = ue4m3 cast of float32(float32(amax_b / 6) * s_g); with
    sc its value, r = float32(s_g / sc) (0 when sc == 0) and the element code is
    the e2m1 cast of float32(x * r). Returns packed codes [M, K/2] uint8
    (element 2i in the low nibble) and ue4m3 scale codes [M, K/16]."""
    x = np.asarray(x, dtype=np.float64)
    M, K = x.shape
    xp = _pad_cols(x, NVFP4_BLOCK)
    nb = xp.shape[1] // NVFP4_BLOCK
    amax_b = f32(block_amax(xp, NVFP4_BLOCK))
    s_g = np.float32(s_g)
    t = (amax_b / np.float32(6.0)).astype(np.float32) * s_g
    sc_code = encode(t.astype(np.float32).astype(np.float64), UE4M3)
    sc = decode(sc_code, UE4M3).astype(np.float32)
    with np.errstate(divide="ignore"):
        r = np.where(sc == 0, np.float32(0), s_g / np.where(sc == 0, np.float32(1), sc))
    r = r.astype(np.float32)
    y = f32(xp).reshape(M, nb, NVFP4_BLOCK) * r[:, :, None]
    q = encode(y.astype(np.float64), E2M1).reshape(M, nb * NVFP4_BLOCK)[:, :K]
    if K % 2:
        raise ValueError("K must be even to pack e2m1 pairs")
    packed = (q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)
    return packed.astype(np.uint8), sc_code


def unpack_e2m1(packed, K):
    packed = np.asarray(packed).astype(np.uint8)
    M = packed.shape[0]
    q = np.empty((M, packed.shape[1] * 2), dtype=np.uint8)
    q[:, 0::2] = packed & 0xF
    q[:, 1::2] = packed >> 4
    return q[:, :K]


def dequantize_nvfp4(packed, sc_code, s_g, K):
    """value = e2m1 * sc / s_g (float64)."""
    q = unpack_e2m1(packed, K)
    v = decode(q, E2M1)
    sc = np.repeat(decode(sc_code, UE4M3), NVFP4_BLOCK, axis=1)[:, :K]
    return v * sc / np.float64(np.float32(s_g))


def quantize_nvfp4_2d(w, s_g):
    """NVFP4 quantisation of one weight ``w`` [M, K] (M, K multiples of 16)
    with 16x16 blocks and global scale ``s_g``.

    Block scale code = ue4m3 cast of float32(float32(amax_b / 6) * s_g) over
    the 16x16 block; with sc its value, r = float32(s_g / sc) (0 when sc == 0)
    and each element code is the e2m1 cast of float32(x * r). Returns
    (row codes [M, K/2], row scale codes [M, K/16], column codes [K, M/2],
    column scale codes [K, M/16]): each 1x16 block of either copy carries the
    scale of its 16x16 block; element 2i in the low nibble."""
    x = np.asarray(w, dtype=np.float64)
    M, K = x.shape
    B = NVFP4_BLOCK
    if M % B or K % B:
        raise ValueError("M and K must be multiples of 16")
    blocks = np.abs(x).reshape(M // B, B, K // B, B)
    amax_b = f32(blocks.max(axis=(1, 3)))                       # [M/16, K/16]
    s_g = np.float32(s_g)
    t = (amax_b / np.float32(6.0)).astype(np.float32) * s_g
    sc_code = encode(t.astype(np.float32).astype(np.float64), UE4M3)
    sc = decode(sc_code, UE4M3).astype(np.float32)
    with np.errstate(divide="ignore"):
        r = np.where(sc == 0, np.float32(0), s_g / np.where(sc == 0, np.float32(1), sc))
    r = r.astype(np.float32)
    r_full = np.repeat(np.repeat(r, B, axis=0), B, axis=1)      # [M, K]
    y = f32(x) * r_full
    q = encode(f32(y).astype(np.float64), E2M1)                 # [M, K] element codes

    def pack(c):
        return ((c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)).astype(np.uint8)

    row_sc = np.repeat(sc_code, B, axis=0)                      # [M, K/16]
    col_sc = np.repeat(sc_code.T, B, axis=0)                    # [K, M/16]
    return pack(q), row_sc.astype(np.uint8), pack(np.ascontiguousarray(q.T)), col_sc.astype(np.uint8)

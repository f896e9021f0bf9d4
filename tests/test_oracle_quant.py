"""Pins of the oracle's block quantisers (CPU only).

Pins used: brute force over every bf16 amax, closed forms at the edges of the
scale rule, exact round trips of values built to be representable, element
error bounds of round-to-nearest, zero fill of partial blocks, and the
transpose identity of TransformerEngine issue #2393 (maintainer replies).
"""
import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q


def _all_pos_bf16():
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32).astype(np.uint16)
    return F.bf16_bits_to_f64(bits)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_mx_rceil_every_bf16_amax(fmt):
    f = F.FORMATS[fmt]
    a = _all_pos_bf16()
    e, code = Q.mx_scale_exponent(a, fmt, "rceil")
    assert np.all(code == e + 127)
    unclamped = e > -127
    # no element of the block saturates ...
    assert np.all(a * np.exp2(-e.astype(np.float64)) <= f.max_finite)
    # ... and one power of two less would saturate the amax
    assert np.all(a[unclamped] * np.exp2(-(e[unclamped] - 1.0)) > f.max_finite)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_mx_floor_every_bf16_amax(fmt):
    a = _all_pos_bf16()
    e, _ = Q.mx_scale_exponent(a, fmt, "floor")
    emax = F.EMAX[fmt]
    s = a * np.exp2(-e.astype(np.float64))
    ok = e > -127
    assert np.all((s[ok] >= 2.0 ** emax) & (s[ok] < 2.0 ** (emax + 1)))


def test_mx_closed_forms():
    for j in (-20, -3, 0, 5, 40):
        amax = 448.0 * 2.0 ** j
        e, _ = Q.mx_scale_exponent(np.array([amax]), "e4m3", "rceil")
        assert e[0] == j
        nxt = amax * (1 + 2.0 ** -7)       # next bf16 above 448 * 2^j
        e2, _ = Q.mx_scale_exponent(np.array([nxt]), "e4m3", "rceil")
        assert e2[0] == j + 1
        ef, _ = Q.mx_scale_exponent(np.array([nxt]), "e4m3", "floor")
        assert ef[0] == j                  # floor keeps j and saturates
    x = np.zeros((1, 32))
    x[0, 3] = 448.0 * 2.0 ** 5
    codes, sc = Q.quantize_mx(x, "e4m3")
    assert sc[0, 0] == 127 + 5 and codes[0, 3] == 0x7E
    # amax 0 -> scale code 0, all codes +0 / -0
    z = np.zeros((1, 32))
    z[0, 1] = -0.0
    codes, sc = Q.quantize_mx(z)
    assert sc[0, 0] == 0 and np.all(codes & 0x7F == 0)
    # non-finite amax -> NaN scale, NaN codes
    n = np.ones((1, 32))
    n[0, 0] = np.inf
    codes, sc = Q.quantize_mx(n)
    assert sc[0, 0] == 255 and np.all(codes & 0x7F == 0x7F)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_mx_exact_roundtrip(fmt):
    f = F.FORMATS[fmt]
    rng = np.random.default_rng(3)
    M, K = 16, 256
    finite = f.pos_codes[f.pos_values <= f.max_finite]
    codes = rng.choice(finite, size=(M, K)) | (rng.integers(0, 2, (M, K)) * f.sign_bit)
    # put the largest code in every block so the block's scale is known
    for b in range(K // 32):
        codes[:, b * 32 + rng.integers(0, 32)] = f.max_code
    ex = rng.integers(-30, 30, size=(M, K // 32))
    x = F.decode(codes, f) * np.repeat(np.exp2(ex.astype(np.float64)), 32, axis=1)
    got_codes, got_sc = Q.quantize_mx(x, fmt, "rceil")
    np.testing.assert_array_equal(got_sc, (ex + 127).astype(np.uint8))
    np.testing.assert_array_equal(got_codes, codes.astype(np.uint8))
    np.testing.assert_array_equal(Q.dequantize_mx(got_codes, got_sc, fmt), x)


def test_mx_error_bound_and_sqnr():
    rng = np.random.default_rng(4)
    x = F.round_to_bf16(rng.standard_normal((64, 1024)))
    codes, sc = Q.quantize_mx(x, "e4m3")
    d = Q.dequantize_mx(codes, sc, "e4m3")
    scale = np.repeat(F.e8m0_decode(sc), 32, axis=1)
    y = np.abs(x) / scale
    # half a code step: 2^(floor(log2 y) - 3) / 2 in the normal range,
    # 2^-9 / 2 below 2^-6 (subnormal codes)
    step = np.where(y >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(y, 1e-300))) - 3), 2.0 ** -9)
    assert np.all(np.abs(d - x) <= step / 2 * scale + 1e-300)
    sq = 10 * np.log10(np.sum(x ** 2) / np.sum((x - d) ** 2))
    assert 29.0 < sq < 33.0


def test_mx_partial_block_zero_fill():
    rng = np.random.default_rng(5)
    x = F.round_to_bf16(rng.standard_normal((8, 40)))
    xp = np.zeros((8, 64))
    xp[:, :40] = x
    c1, s1 = Q.quantize_mx(x)
    c2, s2 = Q.quantize_mx(xp)
    np.testing.assert_array_equal(c1, c2[:, :40])
    np.testing.assert_array_equal(s1, s2)


def test_blockwise_closed_form_and_roundtrip():
    rng = np.random.default_rng(6)
    # single block: the element equal to amax maps to the largest code
    for a in (1.0, 3.140625, 1e-3, 250.0):
        x = np.zeros((1, 128))
        x[0, 7] = a
        x[0, 9] = -a
        c, si = Q.quantize_block_1x128(x, "e4m3")
        assert c[0, 7] == 0x7E and c[0, 9] == 0xFE
        assert si[0, 0] == np.float32(1.0) / (np.float32(448.0) / np.float32(a))
    # power-of-two scales make the round trip exact
    f = F.E4M3
    codes = rng.choice(f.pos_codes[:-1], size=(4, 256)) | (rng.integers(0, 2, (4, 256)) * 0x80)
    codes[:, 5] = 0x7E
    codes[:, 200] = 0xFE
    k = rng.integers(-10, 10, size=(4, 2))
    x = F.decode(codes, f) * np.repeat(np.exp2(-k.astype(np.float64)), 128, axis=1)
    c, si = Q.quantize_block_1x128(x, "e4m3")
    np.testing.assert_array_equal(c, codes.astype(np.uint8))
    np.testing.assert_array_equal(si, np.exp2(-k).astype(np.float32))
    # amax 0: scale 1
    c, si = Q.quantize_block_1x128(np.zeros((2, 128)))
    assert np.all(si == 1.0) and np.all(c == 0)


def test_blockwise_128x128_tile_amax():
    w = np.zeros((256, 256))
    w[3, 5] = 10.0       # tile (0,0) amax 10 in row 3
    w[100, 17] = 1.0     # same tile, another row: scaled by the tile's amax
    w[130, 140] = 2.0    # tile (1,1)
    c, si = Q.quantize_block_128x128(w, "e4m3")
    assert si.shape == (2, 2)
    assert si[0, 0] == np.float32(1) / (np.float32(448) / np.float32(10))
    assert c[3, 5] == 0x7E and c[130, 140] == 0x7E
    assert F.decode(c[100, 17], F.E4M3) == float(F.decode(F.encode(np.float32(np.float32(1.0) * (np.float32(448) / np.float32(10))), F.E4M3), F.E4M3))
    assert si[0, 1] == 1.0 and si[1, 0] == 1.0


def test_transpose_identity_definition():
    """128x1 blocks of x equal 1x128 blocks of x^T, transposed back
    (TransformerEngine issue #2393): the column quantiser is the row
    quantiser applied to the transpose."""
    rng = np.random.default_rng(7)
    x = F.round_to_bf16(rng.standard_normal((256, 128)))
    c_row, s_row = Q.quantize_block_1x128(x.T)
    # column blocks computed directly along axis 0
    amax = np.max(np.abs(x.reshape(2, 128, 128)), axis=1)       # [2 blocks, 128 cols]
    s = Q.blockwise_scale(amax, "e4m3")
    direct = F.encode((F.f32(x).reshape(2, 128, 128) * s[:, None, :]).astype(np.float64), F.E4M3)
    np.testing.assert_array_equal(c_row.T, direct.reshape(256, 128))


def test_tensor_scale_roundtrip():
    rng = np.random.default_rng(8)
    codes = rng.choice(F.E5M2.pos_codes[:-1], size=(8, 64)).astype(np.uint8)
    x = F.decode(codes, F.E5M2) * 2.0 ** -6
    c, amax = Q.quantize_tensor(x, np.float32(64.0), "e5m2")
    np.testing.assert_array_equal(c, codes)
    assert amax == np.max(np.abs(x))


def test_nvfp4_exhaustive_roundtrip():
    """Every finite nonzero ue4m3 block scale times every e2m1 code comes back
    exactly (global scale 1, i.e. tensor amax 6*448)."""
    s_g = Q.nvfp4_global_scale(6.0 * 448.0)
    assert s_g == np.float32(1.0)
    sc_codes = [c for c in F.UE4M3.pos_codes if F.UE4M3.pos_values[list(F.UE4M3.pos_codes).index(c)] > 0]
    q_codes = np.arange(16)
    rows = []
    want_q, want_sc = [], []
    for sc in sc_codes:
        scv = float(F.decode(sc, F.UE4M3))
        q = q_codes.copy()
        q[0] = 0x7                                   # a 6 in the block: amax = 6 * sc
        rows.append(F.decode(q, F.E2M1) * scv)
        want_q.append(q)
        want_sc.append(sc)
    x = np.array(rows)
    packed, scc = Q.quantize_nvfp4(x, s_g)
    np.testing.assert_array_equal(scc[:, 0], np.array(want_sc, dtype=np.uint8))
    np.testing.assert_array_equal(Q.unpack_e2m1(packed, 16), np.array(want_q, dtype=np.uint8))
    np.testing.assert_array_equal(Q.dequantize_nvfp4(packed, scc, s_g, 16), x)


def test_nvfp4_packing_order():
    x = np.zeros((1, 16))
    x[0, 0], x[0, 1] = 6.0, 1.0     # e2m1 codes 7 and 2
    packed, _ = Q.quantize_nvfp4(x, np.float32(1.0))
    assert packed[0, 0] == 0x27


# ---- NVFP4 weights with 16x16 blocks -------------------------------------------

def _diag_block_weight(rng, nbm, nbk):
    """Each 16x16 block holds its largest magnitude A_b once in every row and
    every column (on its diagonal, random signs), the rest smaller."""
    B = 16
    w = rng.uniform(-1.0, 1.0, (nbm * B, nbk * B)) * 0.5
    for i in range(nbm):
        for j in range(nbk):
            A = rng.uniform(1.0, 4.0)
            for d in range(B):
                w[i * B + d, j * B + d] = A * rng.choice([-1.0, 1.0])
    return F.round_to_bf16(w)


def test_nvfp4_2d_equals_1d_when_every_row_and_column_holds_the_block_max():
    """With the block maximum in every row and every column of each 16x16
    block, the 2D block scale equals each 1x16 row block's and each 16x1
    column block's own scale: the row copy is the 1x16 quantisation of w and
    the column copy the 1x16 quantisation of w^T."""
    rng = np.random.default_rng(41)
    w = _diag_block_weight(rng, 3, 4)
    s_g = Q.nvfp4_global_scale(float(np.max(np.abs(w))))
    rc, rs, cc, cs = Q.quantize_nvfp4_2d(w, s_g)
    rc1, rs1 = Q.quantize_nvfp4(w, s_g)
    cc1, cs1 = Q.quantize_nvfp4(w.T, s_g)
    np.testing.assert_array_equal(rc, rc1)
    np.testing.assert_array_equal(rs, rs1)
    np.testing.assert_array_equal(cc, cc1)
    np.testing.assert_array_equal(cs, cs1)


def test_nvfp4_2d_block_scale_is_shared_across_rows():
    """One large element sets the scale of its whole 16x16 block: with s_g = 1
    and amax 6 the scale is 1.0 (ue4m3 0x38), so 0.4 in another row of the
    block is cast as e2m1(0.4) = 0.5 (code 1), where its own 1x16 row block
    would have scaled it to 6 (code 7)."""
    w = np.zeros((16, 16))
    w[0, 3] = 6.0
    w[5, 9] = 0.4
    w = F.round_to_bf16(w)
    rc, rs, cc, cs = Q.quantize_nvfp4_2d(w, np.float32(1.0))
    assert np.all(rs == 0x38) and np.all(cs == 0x38)
    q = Q.unpack_e2m1(rc, 16)
    assert q[0, 3] == 0x7 and q[5, 9] == 0x1
    assert int(np.count_nonzero(q)) == 2
    # the column copy holds the same element codes, transposed
    np.testing.assert_array_equal(Q.unpack_e2m1(cc, 16), q.T)
    rc1, _ = Q.quantize_nvfp4(w[5:6], np.float32(1.0))
    assert Q.unpack_e2m1(rc1, 16)[0, 9] == 0x7


def test_nvfp4_2d_dequantised_error_bound():
    """|dequant(q) - w| is at most half the e2m1 spacing at y = |w| s_g / sc,
    plus the saturated excess max(0, y - 6) (the ue4m3 scale may round below
    amax_b s_g / 6), times sc / s_g, up to the float32 rounding of r."""
    rng = np.random.default_rng(43)
    w = F.round_to_bf16(rng.standard_normal((64, 96)) * 0.02)
    s_g = Q.nvfp4_global_scale(float(np.max(np.abs(w))))
    rc, rs, cc, cs = Q.quantize_nvfp4_2d(w, s_g)
    deq = Q.dequantize_nvfp4(rc, rs, s_g, 96)
    sc = np.repeat(F.decode(rs, F.UE4M3), 16, axis=1)
    y = np.abs(w) * np.float64(s_g) / np.where(sc == 0, 1, sc)
    spacing = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
    bound = (0.5 * spacing + np.maximum(0.0, y - 6.0)) * sc / np.float64(s_g) * (1 + 2.0 ** -20)
    assert np.all(np.abs(deq - w) <= bound + 1e-30)
    assert np.max(y) > 6.0                      # the case the excess term covers occurs here
    np.testing.assert_array_equal(Q.dequantize_nvfp4(cc, cs, s_g, 64), deq.T)


def test_tensor_dequantise_divides_by_the_float32_scale():
    """Per-tensor dequantisation (delayed scaling, Megatron-LM issue #1152):
    the value of a code is decode(code) / s with s the float32 scale. Checked
    against exact rational arithmetic for a scale that is not a power of two
    (so float64(448 / 3) and float32(448 / 3) give different values), and by
    the round trip x -> codes -> values staying within e4m3's half step."""
    from fractions import Fraction
    s32 = np.float32(448.0) / np.float32(3.0)
    assert float(s32) != 448.0 / 3.0
    codes = np.array([[0x7E, 0x38, 0x01, 0xFE, 0x00, 0x80]], dtype=np.uint8)
    got = Q.dequantize_tensor(codes, s32)
    for c, v in zip(codes[0], got[0]):
        want = Fraction(float(F.decode(np.uint8(c), F.E4M3))) / Fraction(float(s32))
        assert v == float(want), (c, v, float(want))
    assert abs(got[0, 0] - 3.0) < 1e-6                  # 448 / (448 / 3)
    # a scale handed in as a float64 is the float32 the codes were cast with
    np.testing.assert_array_equal(Q.dequantize_tensor(codes, 448.0 / 3.0), got)
    rng = np.random.default_rng(9)
    x = F.round_to_bf16(rng.standard_normal((16, 64)) * 0.7)
    s = np.float32(448.0) / np.float32(np.max(np.abs(x)))
    c, _ = Q.quantize_tensor(x, s)
    back = Q.dequantize_tensor(c, s)
    big = np.abs(x) >= 2.0 ** -6 / float(s)             # normal range of e4m3 after scaling
    assert np.all(np.abs(back - x)[big] <= 2.0 ** -4 * np.abs(x)[big] + 1e-12)


def test_blockwise_1x128_dequantise_roundtrip():
    """1x128 blocks (TransformerEngine issue #2393): with power-of-two block
    scales the round trip codes -> values -> codes -> values is exact, and
    each 128-element block of each row carries its own scale (four rows times
    two blocks, all different)."""
    rng = np.random.default_rng(10)
    f = F.E4M3
    codes = (rng.choice(f.pos_codes[:-1], size=(4, 256)) | (rng.integers(0, 2, (4, 256)) * 0x80)).astype(np.uint8)
    codes[:, 3] = 0x7E
    codes[:, 131] = 0xFE
    k = np.arange(8).reshape(4, 2) - 3                   # eight different exponents
    x = F.decode(codes, f) * np.repeat(np.exp2(-k.astype(np.float64)), 128, axis=1)
    c, si = Q.quantize_block_1x128(x)
    np.testing.assert_array_equal(c, codes)
    np.testing.assert_array_equal(Q.dequantize_block_1x128(c, si), x)
    # the block of element (r, j) is (r, j // 128): a wrong axis would mix rows
    assert Q.dequantize_block_1x128(c, si)[1, 200] == F.decode(codes[1, 200], f) * 2.0 ** -k[1, 1]


def test_blockwise_128x128_dequantise_roundtrip():
    """128x128 weight tiles (TransformerEngine issue #2393): a 256x384 weight
    whose six tiles have six different power-of-two scales comes back
    exactly, so the scale of element (n, k) is tile (n // 128, k // 128) and
    not its transpose."""
    rng = np.random.default_rng(11)
    f = F.E4M3
    N, K = 256, 384
    codes = (rng.choice(f.pos_codes[:-1], size=(N, K)) | (rng.integers(0, 2, (N, K)) * 0x80)).astype(np.uint8)
    for bn in range(2):
        for bk in range(3):
            codes[bn * 128 + 5, bk * 128 + 7] = 0x7E     # each tile reaches the largest code
    k = np.array([[0, 2, 5], [-3, 1, 4]])
    scale = np.repeat(np.repeat(np.exp2(-k.astype(np.float64)), 128, axis=0), 128, axis=1)
    x = F.decode(codes, f) * scale
    c, si = Q.quantize_block_128x128(x)
    np.testing.assert_array_equal(c, codes)
    np.testing.assert_array_equal(si, np.exp2(-k).astype(np.float32))
    np.testing.assert_array_equal(Q.dequantize_block_128x128(c, si), x)


def test_tile_128x128_transpose_identity():
    """The column-wise copy of a 128x128-tile weight (TransformerEngine issue
    #2393: 128x128 weight blocks, transpose identity): quantising W^T gives
    the transposed codes and the transposed tile scales, because a tile's
    amax does not depend on its orientation. Tiles with different scales and
    an all-zero tile."""
    rng = np.random.default_rng(12)
    w = F.round_to_bf16(rng.standard_normal((256, 384)) * 0.02)
    w[:128, 128:256] *= 1000.0
    w[128:, :128] = 0.0
    for fmt in ("e4m3", "e5m2"):
        c, si = Q.quantize_block_128x128(w, fmt)
        ct, sit = Q.quantize_block_128x128(np.ascontiguousarray(w.T), fmt)
        np.testing.assert_array_equal(ct, c.T)
        np.testing.assert_array_equal(sit, si.T)
        assert si[1, 0] == 1.0 and np.all(c[128:, :128] == 0)

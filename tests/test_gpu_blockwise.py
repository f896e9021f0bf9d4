"""Blockwise FP8 backward path against the oracle, through the C ABI.

TransformerEngine issue #2393 (maintainer replies) fixes the recipe: 1x128
blocks in the forward, 128x1 blocks for the backward, the column-wise copy
being the 1x128 quantisation of the transpose (transpose identity), with
128x128 tiles for weights. Checked here:
* column-wise copies (128x1 blocks inside each 128-aligned group) from every
  quantiser that writes one: grouped quantise, permute, SwiGLU, dSwiGLU,
  unpermute backward, and plain matrices; codes and float32 scale_inv
  bit-exact;
* 128x128 weights with both copies from one pass (the column-wise copy is the
  transposed codes with the transposed tile scales);
* the blockwise dgrad (dY row-wise x the column-wise weight copy) and wgrad
  (both operands column-wise, contraction over each group's rows, empty
  group, beta 1) within the GEMM tolerances, on operands the oracle
  quantised.
"""
import numpy as np
import pytest
import torch

from oracle import formats as OF
from oracle import gemm as OG
from oracle import layer as OL
from oracle import quant as OQ
from oracle import routing as OR
from tests.layer_check import GEMM_TOL_BF16, GEMM_TOL_F32, bf16_np, check_elementwise, rel_fro, u8_np

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def mgq():
    from fp8_grouped_gemm_gb300 import mgq as m
    m.load()
    return m


def _dt(mgq, fmt):
    return mgq.E5M2 if fmt == "e5m2" else mgq.E4M3


def _bf16(rng, shape, std=1.0):
    return torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16)


def _col_oracle(x_rows, off, fmt):
    """Column-wise copy per group: 1x128 quantisation of each group's
    transpose. Returns {e: (codes [C, n], scale_inv [C, n/128])}."""
    out = {}
    for e in range(len(off) - 1):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            out[e] = OQ.quantize_block_1x128(np.ascontiguousarray(x_rows[lo:hi].T), fmt)
    return out


def _check_cols(col, csc, x_rows, off, fmt, what):
    """col: device [C, R_cap] codes; csc: device float32 [R_cap/128][C]."""
    cg, sg = u8_np(col), csc.cpu().numpy()
    for e, (cc, cs) in _col_oracle(x_rows, off, fmt).items():
        lo, hi = int(off[e]), int(off[e + 1])
        assert np.array_equal(cg[:, lo:hi], cc), (what, e, "codes")
        assert np.array_equal(sg[lo // 128:hi // 128].T, cs), (what, e, "scales")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_grouped_quantize_blockwise_rows_and_columns(mgq, fmt):
    rng = np.random.default_rng(91)
    C, R_cap = 384, 1024
    sizes = [256, 0, 128, 384]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    E, Rp = len(sizes), int(off[-1])
    x = _bf16(rng, (R_cap, C), 3.0)
    x[5, 7] = 0.0
    x[130:140] = 0.0                      # part of a block all zero; an all-zero column block follows
    x[256:384, 0] = 0.0
    x[Rp:] = 1e4                          # rows past the groups: never read
    xf = bf16_np(x)[:Rp]
    dt = _dt(mgq, fmt)
    codes = torch.full((R_cap, C), 0xAB, dtype=torch.uint8, device=DEV)
    sc = torch.full((C // 128, R_cap), -1.0, dtype=torch.float32, device=DEV)
    col = torch.full((C, R_cap), 0xAB, dtype=torch.uint8, device=DEV)
    csc = torch.full((R_cap // 128, C), -1.0, dtype=torch.float32, device=DEV)
    q = mgq.qdesc(dt, mgq.BLK_1x128_F32, codes, sc, col, csc)
    offd = torch.from_numpy(off).to(DEV)
    mgq.grouped_quantize(x.to(DEV), offd, E, q)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    c, si = OQ.quantize_block_1x128(xf, fmt)
    assert np.array_equal(u8_np(codes)[:Rp], c)
    assert np.array_equal(sc.cpu().numpy().T[:Rp], si)
    _check_cols(col, csc, xf, off, fmt, "grouped")
    assert torch.all(codes[Rp:] == 0xAB).item()
    # the all-zero column block: codes 0, scale_inv 1 (scale 1)
    assert float(csc[2, 0].item()) == 1.0 and torch.all(col[0, 256:384] == 0).item()
    # a group start off the 128-row block boundary is reported
    bad = torch.from_numpy(np.array([0, 64, Rp], dtype=np.int32)).to(DEV)
    mgq.grouped_quantize(x.to(DEV), bad, 2, q)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.ERR_INVALID_ARG


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_block_quantize_blockwise_columns(mgq, fmt):
    """Plain matrices [G, M, K]: 128x128 weight tiles with both copies from
    one pass, and 1x128 rows with 128x1 columns."""
    rng = np.random.default_rng(92)
    G, M, K = 3, 256, 384
    w = _bf16(rng, (G, M, K), 0.02)
    w[1, :128, 128:256] *= 1000.0           # one tile far larger than its neighbours
    w[2, 128:, :128] = 0.0                  # an all-zero tile
    wf = bf16_np(w)
    dt = _dt(mgq, fmt)
    wd = w.to(DEV)
    # 128x128 tiles
    rq = torch.full((G, M, K), 0xAB, dtype=torch.uint8, device=DEV)
    rs = torch.full((G, M // 128, K // 128), -1.0, dtype=torch.float32, device=DEV)
    cq = torch.full((G, K, M), 0xAB, dtype=torch.uint8, device=DEV)
    cs = torch.full((G, K // 128, M // 128), -1.0, dtype=torch.float32, device=DEV)
    mgq.block_quantize(wd, mgq.qdesc(dt, mgq.BLK_128x128_F32, rq, rs, cq, cs))
    # the row-only call (its own kernel) gives the same row copy
    rq2 = torch.full((G, M, K), 0xAB, dtype=torch.uint8, device=DEV)
    rs2 = torch.full((G, M // 128, K // 128), -1.0, dtype=torch.float32, device=DEV)
    mgq.block_quantize(wd, mgq.qdesc(dt, mgq.BLK_128x128_F32, rq2, rs2))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    for g in range(G):
        c, si = OQ.quantize_block_128x128(wf[g], fmt)
        ct, sit = OQ.quantize_block_128x128(np.ascontiguousarray(wf[g].T), fmt)
        assert np.array_equal(u8_np(rq[g]), c) and np.array_equal(rs[g].cpu().numpy(), si), g
        assert np.array_equal(u8_np(cq[g]), ct) and np.array_equal(cs[g].cpu().numpy(), sit), g
    assert torch.equal(rq, rq2) and torch.equal(rs, rs2)
    # 1x128 rows and 128x1 columns of each group
    rq = torch.full((G, M, K), 0xAB, dtype=torch.uint8, device=DEV)
    rs = torch.full((K // 128, G * M), -1.0, dtype=torch.float32, device=DEV)
    cq = torch.full((G, K, M), 0xAB, dtype=torch.uint8, device=DEV)
    cs = torch.full((M // 128, G * K), -1.0, dtype=torch.float32, device=DEV)
    mgq.block_quantize(wd, mgq.qdesc(dt, mgq.BLK_1x128_F32, rq, rs, cq, cs))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    for g in range(G):
        c, si = OQ.quantize_block_1x128(wf[g], fmt)
        ct, sit = OQ.quantize_block_1x128(np.ascontiguousarray(wf[g].T), fmt)
        assert np.array_equal(u8_np(rq[g]), c), g
        assert np.array_equal(rs.cpu().numpy()[:, g * M:(g + 1) * M].T, si), g
        assert np.array_equal(u8_np(cq[g]), ct), g
        assert np.array_equal(cs.cpu().numpy()[:, g * K:(g + 1) * K].T, sit), g


@pytest.mark.parametrize("case", [(1000, 6, 2, 384, (2,)), (300, 8, 1, 5120, (0, 5)), (2500, 16, 8, 256, ())],
                         ids=lambda c: f"T{c[0]}E{c[1]}k{c[2]}H{c[3]}")
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_permute_blockwise_columns(mgq, case, fmt):
    T, E, k, H, empty = case
    rng = np.random.default_rng(T + 93)
    allowed = np.array([e for e in range(E) if e not in empty])
    idx = np.stack([rng.choice(allowed, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    x = _bf16(rng, (T, H))
    xf = bf16_np(x)
    R = mgq.r_cap(T, k, E, 128)
    dt = _dt(mgq, fmt)
    rim = torch.empty((T, k), dtype=torch.int32, device=DEV)
    src = torch.empty((R,), dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    cnt = torch.empty(E, dtype=torch.int32, device=DEV)
    ws = torch.empty(mgq.permute_workspace_size(T, k, E), dtype=torch.uint8, device=DEV)
    codes = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    sc = torch.full((H // 128, R), -1.0, dtype=torch.float32, device=DEV)
    col = torch.full((H, R), 0xAB, dtype=torch.uint8, device=DEV)
    csc = torch.full((R // 128, H), -1.0, dtype=torch.float32, device=DEV)
    q = mgq.qdesc(dt, mgq.BLK_1x128_F32, codes, sc, col, csc)
    mgq.moe_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), E, 128, q, R, rim, src, off, cnt, ws)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    w_rim, w_src, w_off, w_cnt = OR.permute_indices(idx, E, 128)
    Rp = int(w_off[-1])
    assert np.array_equal(off.cpu().numpy(), w_off) and np.array_equal(rim.cpu().numpy(), w_rim)
    assert np.array_equal(src.cpu().numpy()[:Rp], w_src)
    c, si = OQ.quantize_block_1x128(xf, fmt)
    assert np.array_equal(u8_np(codes)[:Rp], OR.permute_rows(c, w_rim, Rp))
    assert np.array_equal(sc.cpu().numpy().T[:Rp], OR.permute_rows(si, w_rim, Rp, fill=0.0))
    _check_cols(col, csc, OR.permute_rows(xf, w_rim, Rp, fill=0.0), w_off, fmt, "permute")


def _layout(rng, E, R_cap, empty=(1,)):
    sizes = [0 if e in empty else int(rng.integers(1, 4)) * 128 for e in range(E)]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    assert off[-1] <= R_cap
    return off


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_swiglu_and_dswiglu_blockwise_columns(mgq, fmt):
    rng = np.random.default_rng(94)
    E, F, R_cap = 4, 768, 1280
    off = _layout(rng, E, R_cap)
    Rp = int(off[-1])
    offd = torch.from_numpy(off).to(DEV)
    dt = _dt(mgq, fmt)
    gu = _bf16(rng, (R_cap, 2 * F), 2.0).to(DEV)
    dh = _bf16(rng, (R_cap, F), 0.5).to(DEV)
    # SwiGLU: h [R_cap, F], rows 1x128 and columns 128x1
    h = torch.empty((R_cap, F), dtype=torch.bfloat16, device=DEV)
    codes = torch.full((R_cap, F), 0xAB, dtype=torch.uint8, device=DEV)
    sc = torch.full((F // 128, R_cap), -1.0, dtype=torch.float32, device=DEV)
    col = torch.full((F, R_cap), 0xAB, dtype=torch.uint8, device=DEV)
    csc = torch.full((R_cap // 128, F), -1.0, dtype=torch.float32, device=DEV)
    mgq.swiglu_quantize(gu, R_cap, F, offd, E, mgq.qdesc(dt, mgq.BLK_1x128_F32, codes, sc, col, csc), h)
    # dSwiGLU: [dG | dU] [R_cap, 2F]
    dgu = torch.empty((R_cap, 2 * F), dtype=torch.bfloat16, device=DEV)
    dcodes = torch.full((R_cap, 2 * F), 0xAB, dtype=torch.uint8, device=DEV)
    dsc = torch.full((2 * F // 128, R_cap), -1.0, dtype=torch.float32, device=DEV)
    dcol = torch.full((2 * F, R_cap), 0xAB, dtype=torch.uint8, device=DEV)
    dcsc = torch.full((R_cap // 128, 2 * F), -1.0, dtype=torch.float32, device=DEV)
    mgq.dswiglu_quantize(dh, gu, R_cap, F, offd, E, mgq.qdesc(dt, mgq.BLK_1x128_F32, dcodes, dsc, dcol, dcsc), dgu)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    guf = bf16_np(gu)[:Rp]
    hg = bf16_np(h)[:Rp]
    check_elementwise(OL.swiglu(guf, F), hg, "swiglu")
    c, si = OQ.quantize_block_1x128(hg, fmt)
    assert np.array_equal(u8_np(codes)[:Rp], c) and np.array_equal(sc.cpu().numpy().T[:Rp], si)
    _check_cols(col, csc, hg, off, fmt, "swiglu")
    dg = bf16_np(dgu)[:Rp]
    check_elementwise(OL.dswiglu(bf16_np(dh)[:Rp], guf, F), dg, "dswiglu")
    c, si = OQ.quantize_block_1x128(dg, fmt)
    assert np.array_equal(u8_np(dcodes)[:Rp], c) and np.array_equal(dsc.cpu().numpy().T[:Rp], si)
    _check_cols(dcol, dcsc, dg, off, fmt, "dswiglu")


@pytest.mark.parametrize("fmt", ["e5m2", "e4m3"])
def test_unpermute_bwd_blockwise_columns(mgq, fmt):
    rng = np.random.default_rng(95)
    T, E, k, H = 900, 6, 2, 512
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    probs = rng.random((T, k)).astype(np.float32)
    rim, src, off, cnt = OR.permute_indices(idx, E, 128)
    Rp = int(off[-1])
    R = mgq.r_cap(T, k, E, 128)
    y = _bf16(rng, (R, H))
    dout = _bf16(rng, (T, H), 1e-3)
    dt = _dt(mgq, fmt)
    codes = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    sc = torch.full((H // 128, R), -1.0, dtype=torch.float32, device=DEV)
    col = torch.full((H, R), 0xAB, dtype=torch.uint8, device=DEV)
    csc = torch.full((R // 128, H), -1.0, dtype=torch.float32, device=DEV)
    dprobs = torch.empty((T, k), dtype=torch.float32, device=DEV)
    q = mgq.qdesc(dt, mgq.BLK_1x128_F32, codes, sc, col, csc)
    mgq.moe_unpermute_bwd(dout.to(DEV), y.to(DEV), torch.from_numpy(rim).to(DEV), torch.from_numpy(
        np.concatenate([src, np.full(R - Rp, -1, np.int32)])).to(DEV), torch.from_numpy(probs).to(DEV), R,
        torch.from_numpy(off).to(DEV), E, q, dprobs)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    dy32, dp = OR.unpermute_bwd(bf16_np(dout), bf16_np(y)[:Rp], rim, probs, Rp)
    c, si = OQ.quantize_block_1x128(dy32.astype(np.float64), fmt)
    si[src < 0] = 0.0                    # filler rows: zero codes and zero scales
    assert np.array_equal(u8_np(codes)[:Rp], c)
    assert np.array_equal(sc.cpu().numpy().T[:Rp], si)
    _check_cols(col, csc, dy32.astype(np.float64), off, fmt, "unpermute_bwd")
    assert rel_fro(dp, dprobs.cpu().numpy()) <= 1e-5


def _rows_blk(a, fmt):
    """Oracle 1x128 codes and scale_inv laid out as the GEMM reads them
    ([rows, K] codes, [K/128][rows] scale_inv), plus the dequantised values."""
    c, si = OQ.quantize_block_1x128(a, fmt)
    return c, np.ascontiguousarray(si.T), OQ.dequantize_block_1x128(c, si, fmt)


def _cols_blk(a, off, R_cap, fmt):
    """Column-wise copy of a [R, C] matrix, 128x1 blocks inside each group:
    codes [C, R_cap], scale_inv [R_cap/128][C], dequantised [R, C]."""
    R, C = a.shape
    codes = np.zeros((C, R_cap), np.uint8)
    si = np.zeros((R_cap // 128, C), np.float32)
    deq = np.zeros((R, C))
    for e in range(len(off) - 1):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        cc, cs = OQ.quantize_block_1x128(np.ascontiguousarray(a[lo:hi].T), fmt)
        codes[:, lo:hi] = cc
        si[lo // 128:hi // 128] = cs.T
        deq[lo:hi] = OQ.dequantize_block_1x128(cc, cs, fmt).T
    return codes, si, deq


@pytest.mark.parametrize("fmts", [("e5m2", "e4m3"), ("e4m3", "e4m3")], ids=["hybrid", "e4m3"])
def test_gemm_dgrad_and_wgrad_blockwise(mgq, fmts):
    """dgrad: dA = dY W_e with dY row-wise (1x128 along N) and the weight's
    column-wise copy (128x128 tiles of W_e^T); wgrad: dW_e = beta dW_e +
    dY_e^T A_e from the column-wise copies (128x1 blocks along the group's
    rows), an empty group giving zeros (beta 0) or dW_e unchanged (beta 1)."""
    fg, fa = fmts
    rng = np.random.default_rng(96)
    E, N, K, R_cap = 3, 384, 512, 1024       # wgrad output columns: a multiple of 256
    off = np.array([0, 256, 256, 640], dtype=np.int32)        # group 1 empty
    Rp = int(off[-1])
    dy = bf16_np(_bf16(rng, (R_cap, N), 1e-2))
    dy[Rp:] = 0.0
    a = bf16_np(_bf16(rng, (R_cap, K)))
    a[Rp:] = 0.0
    w = bf16_np(_bf16(rng, (E, N, K), 0.02))
    dga, dwa = _dt(mgq, fg), _dt(mgq, fa)
    offd = torch.from_numpy(off).to(DEV)
    # dgrad
    dyc, dys, dyd = _rows_blk(dy, fg)
    wcol = np.zeros((E, K, N), np.uint8)
    wcs = np.zeros((E, K // 128, N // 128), np.float32)
    wcd = np.zeros((E, K, N))
    for e in range(E):
        c, si = OQ.quantize_block_128x128(np.ascontiguousarray(w[e].T), fa)
        wcol[e], wcs[e], wcd[e] = c, si, OQ.dequantize_block_128x128(c, si, fa)
    # device copies, kept alive while the GEMMs run (operands hold raw pointers)
    keep = {}

    def T_(name, x):
        keep[name] = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
        return keep[name]

    dA = torch.full((R_cap, K), 7.0, dtype=torch.bfloat16, device=DEV)
    mgq.grouped_gemm_dgrad(mgq.operand(T_("dyc", dyc), T_("dys", dys), N, dga),
                           mgq.operand(T_("wcol", wcol), T_("wcs", wcs), N, dwa),
                           mgq.BLK_1x128_F32, offd, E, R_cap, N, K, dA)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    ref = OG.grouped_gemm_fwd(dyd, wcd, off)                    # dY_e (Wcol_e)^T = dY_e W_e
    assert rel_fro(OF.round_to_bf16(ref[:Rp]), bf16_np(dA)[:Rp]) <= GEMM_TOL_BF16
    # wgrad, beta 0 then beta 1
    gcc, gcs, gcd = _cols_blk(dy[:Rp], off, R_cap, fg)
    acc, acs, acd = _cols_blk(a[:Rp], off, R_cap, fa)
    dW = torch.full((E, N, K), 3.0, dtype=torch.float32, device=DEV)
    A_ = mgq.operand(T_("gcc", gcc), T_("gcs", gcs), R_cap, dga)
    B_ = mgq.operand(T_("acc", acc), T_("acs", acs), R_cap, dwa)
    mgq.grouped_gemm_wgrad(A_, B_, mgq.BLK_1x128_F32, offd, E, R_cap, N, K, dW, 0.0, mgq.OUT_F32)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    ref = OG.grouped_gemm_wgrad(gcd, acd, off, E)
    got = dW.cpu().numpy()
    assert np.all(got[1] == 0.0)
    for e in (0, 2):
        assert rel_fro(ref[e], got[e]) <= GEMM_TOL_F32, e
    mgq.grouped_gemm_wgrad(A_, B_, mgq.BLK_1x128_F32, offd, E, R_cap, N, K, dW, 1.0, mgq.OUT_F32)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    got2 = dW.cpu().numpy()
    assert np.all(got2[1] == 0.0)
    for e in (0, 2):
        assert rel_fro(2.0 * ref[e], got2[e]) <= GEMM_TOL_F32, e
    # bf16 dW (beta 0): the same products, rounded once
    dWb = torch.full((E, N, K), 3.0, dtype=torch.bfloat16, device=DEV)
    mgq.grouped_gemm_wgrad(A_, B_, mgq.BLK_1x128_F32, offd, E, R_cap, N, K, dWb, 0.0, mgq.OUT_BF16)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    gotb = bf16_np(dWb)
    assert np.all(gotb[1] == 0.0)
    for e in (0, 2):
        assert rel_fro(OF.round_to_bf16(ref[e]), gotb[e]) <= GEMM_TOL_BF16, e

"""Parity of each CUDA kernel with the CPU oracle, through the C ABI.

Sizes span several 128x256 GEMM tiles, ragged token counts (tails of the
per-warp and per-chunk loops), empty expert groups, k = 1 and k = 8, and
multi-slice rows. Tolerances are those of tests/layer_check.py.
"""
import numpy as np
import pytest
import torch

from oracle import formats as OF
from oracle import gemm as OG
from oracle import layer as OL
from oracle import quant as OQ
from oracle import routing as OR
from tests.layer_check import (GEMM_TOL_BF16, GEMM_TOL_F32, bf16_np, check_elementwise, rel_fro,
                               tile_mx_scales, u8_np, untile_mx_scales)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def mgq():
    from fp8_grouped_gemm_gb300 import mgq as m
    m.load()
    return m


def _routing(rng, T, E, k, empty=()):
    allowed = np.array([e for e in range(E) if e not in empty])
    idx = np.stack([rng.choice(allowed, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    return idx.reshape(T, k)


def _bf16(rng, shape, std=1.0):
    x = torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16)
    return x


# ---------------------------------------------------------------------------- permute

PERMUTE_CASES = [
    # T, E, k, H, align, empty experts
    (1024, 4, 2, 256, 128, ()),
    (1001, 6, 2, 384, 128, (2,)),
    (300, 8, 1, 5120, 128, (0, 5)),
    (777, 16, 8, 128, 32, (3,)),
    (5, 4, 4, 1024, 128, ()),
    (2500, 128, 8, 256, 128, ()),
    (3000, 1024, 2, 128, 32, ()),      # the largest expert count: most groups empty or tiny
]


@pytest.mark.parametrize("case", PERMUTE_CASES, ids=lambda c: f"T{c[0]}E{c[1]}k{c[2]}H{c[3]}a{c[4]}")
@pytest.mark.parametrize("mode", ["mx_e4m3", "mx_e5m2", "mx_col_e4m3", "mx_col_e5m2", "tensor_e4m3", "blk_e4m3",
                                  "nvfp4", "nvfp4_col"])
def test_permute_quantize(mgq, case, mode):
    T, E, k, H, align, empty = case
    rng = np.random.default_rng(T * 7 + E)
    idx = _routing(rng, T, E, k, empty)
    x = _bf16(rng, (T, H))
    if mode.startswith("tensor"):
        x[:, 3] *= 50                                      # an outlier channel
    R = mgq.r_cap(T, k, E, align)
    dev = torch.device(DEV)
    xd, idxd = x.to(dev), torch.from_numpy(idx).to(dev)
    rim = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    src = torch.full((R,), -7, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    cnt = torch.empty(E, dtype=torch.int32, device=dev)
    ws = torch.empty(mgq.permute_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    nv = mode.startswith("nvfp4")
    codes = torch.full((R, H // 2 if nv else H), 0xAB, dtype=torch.uint8, device=dev)
    fmt = "e5m2" if "e5m2" in mode else "e4m3"
    dt = mgq.E5M2 if fmt == "e5m2" else mgq.E4M3
    xf = bf16_np(x)
    if nv:
        sc = torch.full((mgq.nv_scale_bytes(R, H),), 0xCD, dtype=torch.uint8, device=dev)
        amax = torch.full((1,), 7.0, dtype=torch.float32, device=dev)     # overwritten by the call
        sg = torch.zeros(1, dtype=torch.float32, device=dev)
        col = csc = None
        if mode == "nvfp4_col":
            # column-wise copy: 16-row blocks along the permuted rows, packed along them
            col = torch.full((H, R // 2), 0xAB, dtype=torch.uint8, device=dev)
            csc = torch.full((mgq.nv_scale_bytes(H, R),), 0xCD, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, codes, sc, col, csc, tensor_scale=sg, amax_out=amax)
    elif mode.startswith("mx_col"):
        # row-wise and column-wise (blocks of 32 along the permuted rows) copies
        sc = torch.full((mgq.mx_scale_bytes(R, H),), 0xCD, dtype=torch.uint8, device=dev)
        col = torch.full((H, R), 0xAB, dtype=torch.uint8, device=dev)
        csc = torch.full((mgq.mx_scale_bytes(H, R),), 0xCD, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(dt, mgq.MX32_E8M0, codes, sc, col, csc)
    elif mode.startswith("mx"):
        sc = torch.full((mgq.mx_scale_bytes(R, H),), 0xCD, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(dt, mgq.MX32_E8M0, codes, sc)
    elif mode.startswith("blk"):
        sc = torch.full((H // 128, R), -1.0, dtype=torch.float32, device=dev)
        q = mgq.qdesc(dt, mgq.BLK_1x128_F32, codes, sc)
    else:
        s = torch.tensor([0.37], dtype=torch.float32, device=dev)
        amax = torch.zeros(1, dtype=torch.float32, device=dev)
        col = torch.full((H, R), 0xAB, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(dt, mgq.TENSOR_F32, codes, None, col, None, s, amax)
    mgq.moe_permute(xd, idxd, E, align, q, R, rim, src, off, cnt, ws)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    w_rim, w_src, w_off, w_cnt = OR.permute_indices(idx, E, align)
    Rp = int(w_off[-1])
    assert np.array_equal(off.cpu().numpy(), w_off)
    assert np.array_equal(cnt.cpu().numpy(), w_cnt)
    assert np.array_equal(rim.cpu().numpy(), w_rim)
    assert np.array_equal(src.cpu().numpy()[:Rp], w_src)
    if nv:
        am = float(np.max(np.abs(xf)))
        s_g = OQ.nvfp4_global_scale(am)
        assert float(amax.item()) == am and float(sg.item()) == float(s_g)
        c, s = OQ.quantize_nvfp4(xf, s_g)
        assert np.array_equal(u8_np(codes)[:Rp], OR.permute_rows(c, w_rim, Rp))
        assert np.array_equal(untile_mx_scales(u8_np(sc), R, H, 16)[:Rp], OR.permute_rows(s, w_rim, Rp))
        if mode == "nvfp4_col":
            xp = OR.permute_rows(xf, w_rim, Rp, fill=0.0)
            cc, cs = OQ.quantize_nvfp4(xp.T, s_g)
            assert np.array_equal(u8_np(col)[:, :Rp // 2], cc)
            assert np.array_equal(untile_mx_scales(u8_np(csc), H, R, 16)[:, :Rp // 16], cs)
    elif mode.startswith("mx"):
        c, s = OQ.quantize_mx(xf, fmt)
        assert np.array_equal(u8_np(codes)[:Rp], OR.permute_rows(c, w_rim, Rp))
        assert np.array_equal(untile_mx_scales(u8_np(sc), R, H)[:Rp], OR.permute_rows(s, w_rim, Rp))
        if mode.startswith("mx_col"):
            # groups are padded to multiples of 32 rows: no block straddles two
            xp = OR.permute_rows(xf, w_rim, Rp, fill=0.0)
            cc, cs = OQ.quantize_mx(xp.T, fmt)
            assert np.array_equal(u8_np(col)[:, :Rp], cc)
            assert np.array_equal(untile_mx_scales(u8_np(csc), H, R)[:, :Rp // 32], cs)
    elif mode.startswith("blk"):
        c, si = OQ.quantize_block_1x128(xf, fmt)
        assert np.array_equal(u8_np(codes)[:Rp], OR.permute_rows(c, w_rim, Rp))
        got = sc.cpu().numpy().T[:Rp]
        assert np.array_equal(got, OR.permute_rows(si, w_rim, Rp, fill=0.0))
    else:
        c, am = OQ.quantize_tensor(xf, np.float32(0.37), fmt)
        want = OR.permute_rows(c, w_rim, Rp)
        assert np.array_equal(u8_np(codes)[:Rp], want)
        assert np.array_equal(u8_np(col)[:, :Rp], want.T)
        assert float(amax.item()) == am


def test_permute_bad_expert_index_is_reported(mgq):
    dev = torch.device(DEV)
    T, E, k, H = 64, 4, 2, 128
    idx = np.tile(np.array([[0, 1]], dtype=np.int32), (T, 1))
    idx[5, 1] = 9                       # out of range: skipped and reported
    R = mgq.r_cap(T, k, E, 128)
    bufs = dict(rim=torch.empty(T, k, dtype=torch.int32, device=dev),
                src=torch.empty(R, dtype=torch.int32, device=dev),
                off=torch.empty(E + 1, dtype=torch.int32, device=dev),
                cnt=torch.empty(E, dtype=torch.int32, device=dev))
    codes = torch.empty(R, H, dtype=torch.uint8, device=dev)
    sc = torch.empty(mgq.mx_scale_bytes(R, H), dtype=torch.uint8, device=dev)
    ws = torch.empty(mgq.permute_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    mgq.moe_permute(_bf16(np.random.default_rng(0), (T, H)).to(dev), torch.from_numpy(idx).to(dev), E, 128,
                    mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, codes, sc), R, bufs["rim"], bufs["src"], bufs["off"],
                    bufs["cnt"], ws)
    assert mgq.get_error() == mgq.ERR_DEVICE_INDEX
    assert mgq.get_error() == mgq.OK                 # read and cleared
    assert bufs["rim"][5, 1].item() == -1
    assert bufs["cnt"].cpu().tolist() == [64, 63, 0, 0]


# ---------------------------------------------------------------------------- GEMM

def _mx_operand(rng, rows, K, fmt="e4m3", small=False, sc_lo=120, sc_hi=134):
    f = OF.FORMATS[fmt]
    if small:
        sc_lo, sc_hi = 125, 129          # keeps every partial sum exact in float32
        codes = rng.choice(np.array([0x00, 0x38, 0xB8] if fmt == "e4m3" else [0x00, 0x3C, 0xBC]),
                           size=(rows, K)).astype(np.uint8)
    else:
        codes = rng.choice(f.pos_codes[:-1], size=(rows, K)).astype(np.uint8)
        codes |= (rng.integers(0, 2, (rows, K)) * f.sign_bit).astype(np.uint8)
    sc = rng.integers(sc_lo, sc_hi, size=(rows, K // 32)).astype(np.uint8)
    return codes, sc


def _to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


_KEEP = []   # device buffers referenced by raw pointers in Operand structs


def _op(mgq, codes, scale, ld, dtype, dev):
    """Operand over fresh device copies; the copies stay alive (the struct
    only holds their addresses)."""
    c, s = _to_dev(codes, dev), _to_dev(scale, dev)
    _KEEP.append((c, s))
    if len(_KEEP) > 64:
        del _KEEP[:32]
    return mgq.operand(c, s, ld, dtype)


GEMM_GROUPS = [
    [0, 128, 128, 384, 512],          # E=4, one empty group
    [0, 256],                         # one expert
    [0, 128, 256, 384, 512, 640, 768, 896, 1024, 1152],
]


@pytest.mark.parametrize("offs", GEMM_GROUPS, ids=lambda o: f"E{len(o) - 1}")
@pytest.mark.parametrize("small", [True, False], ids=["exact", "random"])
def test_gemm_fwd_mx(mgq, offs, small):
    rng = np.random.default_rng(len(offs) + small)
    dev = torch.device(DEV)
    E = len(offs) - 1
    N, K = 512, 384
    Rp = offs[-1]
    R_cap = Rp + 256                   # spare rows stay untouched
    ac, asc = _mx_operand(rng, R_cap, K, small=small)
    wc, wsc = _mx_operand(rng, E * N, K, small=small)
    off = np.array(offs, dtype=np.int32)
    out_dtype = mgq.OUT_F32 if small else mgq.OUT_BF16
    Y = torch.full((R_cap, N), float("nan"), dtype=torch.float32 if small else torch.bfloat16, device=dev)
    A = _op(mgq, ac, tile_mx_scales(asc), K, mgq.E4M3, dev)
    Wo = _op(mgq, wc, tile_mx_scales(wsc), K, mgq.E4M3, dev)
    tens = [torch.from_numpy(off).to(dev)]
    mgq.grouped_gemm_fwd(A, Wo, mgq.MX32_E8M0, tens[0], E, R_cap, N, K, Y, out_dtype)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    ref = OG.grouped_gemm_fwd(OQ.dequantize_mx(ac, asc)[:Rp], OQ.dequantize_mx(wc, wsc).reshape(E, N, K), off)
    got = Y.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isnan(got[Rp:]))                 # rows beyond the groups untouched
    if small:
        np.testing.assert_array_equal(got[:Rp], ref)  # every sum exact in float32
    else:
        assert rel_fro(OF.round_to_bf16(ref), got[:Rp]) <= GEMM_TOL_BF16


@pytest.mark.parametrize("fmts", [("e4m3", "e4m3"), ("e5m2", "e4m3")])
def test_gemm_fwd_tensor_scale(mgq, fmts):
    rng = np.random.default_rng(11)
    dev = torch.device(DEV)
    offs = [0, 256, 256, 640]
    E, N, K = 3, 768, 256
    Rp = offs[-1]
    fa, fw = OF.FORMATS[fmts[0]], OF.FORMATS[fmts[1]]
    ac = (rng.choice(fa.pos_codes[:-1], size=(Rp, K)) | (rng.integers(0, 2, (Rp, K)) * fa.sign_bit)).astype(np.uint8)
    wc = (rng.choice(fw.pos_codes[:-1], size=(E * N, K)) | (rng.integers(0, 2, (E * N, K)) * fw.sign_bit)).astype(np.uint8)
    sa = np.array([3.5], dtype=np.float32)
    sw = np.array([0.75, 12.0, 0.01], dtype=np.float32)
    Y = torch.empty(Rp, N, dtype=torch.bfloat16, device=dev)
    da = mgq.E5M2 if fmts[0] == "e5m2" else mgq.E4M3
    A = _op(mgq, ac, sa, K, da, dev)
    Wo = _op(mgq, wc, sw, K, mgq.E4M3, dev)
    offd = torch.tensor(offs, dtype=torch.int32, device=dev)
    mgq.grouped_gemm_fwd(A, Wo, mgq.TENSOR_F32, offd, E, Rp, N, K, Y)
    torch.cuda.synchronize()
    ref = OG.grouped_gemm_fwd(OQ.dequantize_tensor(ac, sa[0], fmts[0]),
                              np.stack([OQ.dequantize_tensor(wc[e * N:(e + 1) * N], sw[e], fmts[1])
                                        for e in range(E)]), np.array(offs))
    assert rel_fro(OF.round_to_bf16(ref), bf16_np(Y)) <= GEMM_TOL_BF16


@pytest.mark.parametrize("scaling", ["tensor", "mx"])
def test_gemm_dgrad_and_wgrad(mgq, scaling):
    """dgrad on the column-wise weight copy and wgrad on the column-wise
    copies of dY and A, with an empty group (wgrad writes zeros, or keeps the
    accumulator with beta = 1)."""
    rng = np.random.default_rng(21)
    dev = torch.device(DEV)
    offs = np.array([0, 128, 128, 512, 640], dtype=np.int32)
    E, N, K = 4, 512, 256            # forward W_e is [N, K]
    Rp = int(offs[-1])
    offd = torch.from_numpy(offs).to(dev)
    if scaling == "tensor":
        f5, f4 = OF.E5M2, OF.E4M3
        dyc = (rng.choice(f5.pos_codes[:-1], size=(Rp, N)) | (rng.integers(0, 2, (Rp, N)) * 0x80)).astype(np.uint8)
        wc = (rng.choice(f4.pos_codes[:-1], size=(E, N, K)) | (rng.integers(0, 2, (E, N, K)) * 0x80)).astype(np.uint8)
        ac = (rng.choice(f4.pos_codes[:-1], size=(Rp, K)) | (rng.integers(0, 2, (Rp, K)) * 0x80)).astype(np.uint8)
        s_dy = np.array([1000.0], dtype=np.float32)
        s_w = np.array([2.0, 0.5, 8.0, 1.0], dtype=np.float32)
        s_a = np.array([4.0], dtype=np.float32)
        dy_deq = OQ.dequantize_tensor(dyc, s_dy[0], "e5m2")
        w_deq = np.stack([OQ.dequantize_tensor(wc[e], s_w[e]) for e in range(E)])
        a_deq = OQ.dequantize_tensor(ac, s_a[0])
        wcol = np.ascontiguousarray(wc.transpose(0, 2, 1))            # [E, K, N]
        dgrad_B = _op(mgq, wcol, s_w, N, mgq.E4M3, dev)
        dgrad_A = _op(mgq, dyc, s_dy, N, mgq.E5M2, dev)
        wg_A = _op(mgq, np.ascontiguousarray(dyc.T), s_dy, Rp, mgq.E5M2, dev)
        wg_B = _op(mgq, np.ascontiguousarray(ac.T), s_a, Rp, mgq.E4M3, dev)
        sc = mgq.TENSOR_F32
    else:
        # dgrad: dY row-wise (blocks along N), W column-wise (blocks along N)
        dyc, dys = _mx_operand(rng, Rp, N, "e5m2")
        wcol, wcols = _mx_operand(rng, E * K, N)                       # [E*K, N]
        dy_deq = OQ.dequantize_mx(dyc, dys, "e5m2")
        w_deq = OQ.dequantize_mx(wcol, wcols).reshape(E, K, N).transpose(0, 2, 1)
        dgrad_A = _op(mgq, dyc, tile_mx_scales(dys), N, mgq.E5M2, dev)
        dgrad_B = _op(mgq, wcol, tile_mx_scales(wcols), N, mgq.E4M3, dev)
        # wgrad: column-wise copies [N, Rp] / [K, Rp] with blocks along the tokens
        dyt, dyts = _mx_operand(rng, N, Rp, "e5m2")
        at, ats = _mx_operand(rng, K, Rp)
        wg_A = _op(mgq, dyt, tile_mx_scales(dyts), Rp, mgq.E5M2, dev)
        wg_B = _op(mgq, at, tile_mx_scales(ats), Rp, mgq.E4M3, dev)
        wg_dy = OQ.dequantize_mx(dyt, dyts, "e5m2").T
        wg_a = OQ.dequantize_mx(at, ats).T
        sc = mgq.MX32_E8M0
    dA = torch.empty(Rp, K, dtype=torch.bfloat16, device=dev)
    mgq.grouped_gemm_dgrad(dgrad_A, dgrad_B, sc, offd, E, Rp, N, K, dA)
    dW = torch.full((E, N, K), 5.0, dtype=torch.float32, device=dev)
    mgq.grouped_gemm_wgrad(wg_A, wg_B, sc, offd, E, Rp, N, K, dW, 0.0)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    ref = OG.grouped_gemm_dgrad(dy_deq, w_deq, offs)
    assert rel_fro(OF.round_to_bf16(ref), bf16_np(dA)) <= GEMM_TOL_BF16
    if scaling == "tensor":
        wg_dy, wg_a = dy_deq, a_deq
    ref_w = OG.grouped_gemm_wgrad(wg_dy, wg_a, offs, E)
    got = dW.cpu().numpy().astype(np.float64)
    assert np.all(got[1] == 0.0)
    assert rel_fro(ref_w, got) <= GEMM_TOL_F32
    # beta = 1: accumulate; the empty group keeps its previous value
    prev = torch.from_numpy(rng.standard_normal((E, N, K)).astype(np.float32)).to(dev)
    dW2 = prev.clone()
    mgq.grouped_gemm_wgrad(wg_A, wg_B, sc, offd, E, Rp, N, K, dW2, 1.0)
    torch.cuda.synchronize()
    got2 = dW2.cpu().numpy().astype(np.float64)
    assert np.array_equal(got2[1], prev[1].cpu().numpy().astype(np.float64))
    assert rel_fro(ref_w + prev.cpu().numpy(), got2) <= GEMM_TOL_F32


@pytest.mark.parametrize("scaling", ["tensor", "mx"])
def test_gemm_largest_expert_count(mgq, scaling):
    """The largest expert count the library takes (1024 groups), most of them
    empty and the rest one or two 128-row tiles: forward over the groups'
    rows (rows past them untouched) and wgrad (empty groups written as
    zeros), against the oracle."""
    rng = np.random.default_rng(1024 + (scaling == "mx"))
    dev = torch.device(DEV)
    E, N, K = 1024, 256, 256
    sizes = rng.choice([0, 128, 256], size=E, p=[0.7, 0.25, 0.05])
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    Rp = int(offs[-1])
    R_cap = Rp + 256
    offd = torch.from_numpy(offs).to(dev)
    if scaling == "tensor":
        f4 = OF.E4M3
        ac = (rng.choice(f4.pos_codes[:-1], size=(R_cap, K)) | (rng.integers(0, 2, (R_cap, K)) * 0x80)).astype(np.uint8)
        wc = (rng.choice(f4.pos_codes[:-1], size=(E * N, K)) | (rng.integers(0, 2, (E * N, K)) * 0x80)).astype(np.uint8)
        dyt = (rng.choice(f4.pos_codes[:-1], size=(N, Rp)) | (rng.integers(0, 2, (N, Rp)) * 0x80)).astype(np.uint8)
        s_a = np.array([2.5], dtype=np.float32)
        s_w = rng.uniform(0.25, 8.0, size=E).astype(np.float32)
        s_dy = np.array([300.0], dtype=np.float32)
        A = _op(mgq, ac, s_a, K, mgq.E4M3, dev)
        Wo = _op(mgq, wc, s_w, K, mgq.E4M3, dev)
        wg_A = _op(mgq, dyt, s_dy, Rp, mgq.E4M3, dev)
        wg_B = _op(mgq, np.ascontiguousarray(ac[:Rp].T), s_a, Rp, mgq.E4M3, dev)
        a_deq = OQ.dequantize_tensor(ac[:Rp], s_a[0])
        w_deq = np.stack([OQ.dequantize_tensor(wc[e * N:(e + 1) * N], s_w[e]) for e in range(E)])
        dy_deq = OQ.dequantize_tensor(dyt, s_dy[0]).T
        wa_deq = a_deq
        sc = mgq.TENSOR_F32
    else:
        ac, asc = _mx_operand(rng, R_cap, K)
        wc, wsc = _mx_operand(rng, E * N, K)
        dyt, dyts = _mx_operand(rng, N, Rp)
        at, ats = _mx_operand(rng, K, Rp)
        A = _op(mgq, ac, tile_mx_scales(asc), K, mgq.E4M3, dev)
        Wo = _op(mgq, wc, tile_mx_scales(wsc), K, mgq.E4M3, dev)
        wg_A = _op(mgq, dyt, tile_mx_scales(dyts), Rp, mgq.E4M3, dev)
        wg_B = _op(mgq, at, tile_mx_scales(ats), Rp, mgq.E4M3, dev)
        a_deq = OQ.dequantize_mx(ac, asc)[:Rp]
        w_deq = OQ.dequantize_mx(wc, wsc).reshape(E, N, K)
        dy_deq = OQ.dequantize_mx(dyt, dyts).T
        wa_deq = OQ.dequantize_mx(at, ats).T
        sc = mgq.MX32_E8M0
    Y = torch.full((R_cap, N), float("nan"), dtype=torch.bfloat16, device=dev)
    mgq.grouped_gemm_fwd(A, Wo, sc, offd, E, R_cap, N, K, Y)
    dW = torch.full((E, N, K), 5.0, dtype=torch.float32, device=dev)
    mgq.grouped_gemm_wgrad(wg_A, wg_B, sc, offd, E, Rp, N, K, dW, 0.0)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    got = bf16_np(Y)
    assert np.all(np.isnan(got[Rp:]))
    ref = OG.grouped_gemm_fwd(a_deq, w_deq, offs)
    assert rel_fro(OF.round_to_bf16(ref), got[:Rp]) <= GEMM_TOL_BF16
    got_w = dW.cpu().numpy().astype(np.float64)
    assert np.all(got_w[sizes == 0] == 0.0)
    ref_w = OG.grouped_gemm_wgrad(dy_deq, wa_deq, offs, E)
    assert rel_fro(ref_w, got_w) <= GEMM_TOL_F32


@pytest.mark.parametrize("exact", [True, False], ids=["exact", "random"])
def test_gemm_mn_major_operands(mgq, exact):
    """Per-tensor dgrad and wgrad reading the row-wise codes transposed
    (MGQ_LAYOUT_MN): dgrad on the forward weight W [E, N, K], wgrad on dY
    [R, N] and A [R, K] themselves, against the oracle and against the same
    GEMMs on explicit column-wise copies."""
    rng = np.random.default_rng(23 + exact)
    dev = torch.device(DEV)
    offs = np.array([0, 128, 128, 512, 640, 1024], dtype=np.int32)
    E, N, K = 5, 768, 512
    Rp = int(offs[-1])
    offd = torch.from_numpy(offs).to(dev)
    f5, f4 = OF.E5M2, OF.E4M3

    def codes(fmt, shape):
        if exact:    # +-1, +-2 and 0: every float32 partial sum is exact
            pool = np.array([0x00, 0x3C, 0xBC, 0x40, 0xC0] if fmt is f5 else [0x00, 0x38, 0xB8, 0x40, 0xC0])
            return rng.choice(pool, size=shape).astype(np.uint8)
        return (rng.choice(fmt.pos_codes[:-1], size=shape) | (rng.integers(0, 2, shape) * 0x80)).astype(np.uint8)

    dyc, wc, ac = codes(f5, (Rp, N)), codes(f4, (E, N, K)), codes(f4, (Rp, K))
    s_dy = np.array([0.5 if exact else 1000.0], dtype=np.float32)
    s_w = np.array([2.0, 0.5, 8.0, 1.0, 4.0], dtype=np.float32)
    s_a = np.array([4.0], dtype=np.float32)
    dy_deq = OQ.dequantize_tensor(dyc, s_dy[0], "e5m2")
    w_deq = np.stack([OQ.dequantize_tensor(wc[e], s_w[e]) for e in range(E)])
    a_deq = OQ.dequantize_tensor(ac, s_a[0])
    MN, sc = mgq.LAYOUT_MN, mgq.TENSOR_F32
    dY = _op(mgq, dyc, s_dy, N, mgq.E5M2, dev)
    W_mn = _op(mgq, wc, s_w, K, mgq.E4M3, dev)
    W_mn.layout = MN
    W_col = _op(mgq, np.ascontiguousarray(wc.transpose(0, 2, 1)), s_w, N, mgq.E4M3, dev)
    dY_mn = _op(mgq, dyc, s_dy, N, mgq.E5M2, dev)
    dY_mn.layout = MN
    A_mn = _op(mgq, ac, s_a, K, mgq.E4M3, dev)
    A_mn.layout = MN
    dY_col = _op(mgq, np.ascontiguousarray(dyc.T), s_dy, Rp, mgq.E5M2, dev)
    A_col = _op(mgq, np.ascontiguousarray(ac.T), s_a, Rp, mgq.E4M3, dev)
    od = mgq.OUT_F32 if exact else mgq.OUT_BF16
    ddt = torch.float32 if exact else torch.bfloat16
    dA_mn = torch.full((Rp, K), float("nan"), dtype=ddt, device=dev)
    dA_k = torch.full((Rp, K), float("nan"), dtype=ddt, device=dev)
    mgq.grouped_gemm_dgrad(dY, W_mn, sc, offd, E, Rp, N, K, dA_mn, od)
    mgq.grouped_gemm_dgrad(dY, W_col, sc, offd, E, Rp, N, K, dA_k, od)
    dW_mn = torch.full((E, N, K), 5.0, dtype=torch.float32, device=dev)
    dW_k = torch.full((E, N, K), 5.0, dtype=torch.float32, device=dev)
    mgq.grouped_gemm_wgrad(dY_mn, A_mn, sc, offd, E, Rp, N, K, dW_mn, 0.0)
    mgq.grouped_gemm_wgrad(dY_col, A_col, sc, offd, E, Rp, N, K, dW_k, 0.0)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    ref = OG.grouped_gemm_dgrad(dy_deq, w_deq, offs)
    ref_w = OG.grouped_gemm_wgrad(dy_deq, a_deq, offs, E)
    got = dA_mn.float().cpu().numpy().astype(np.float64)
    got_w = dW_mn.cpu().numpy().astype(np.float64)
    assert np.all(got_w[1] == 0.0)                            # the empty group
    if exact:
        np.testing.assert_array_equal(got, ref)
        np.testing.assert_array_equal(got_w, ref_w)
    else:
        assert rel_fro(OF.round_to_bf16(ref), got) <= GEMM_TOL_BF16
        assert rel_fro(ref_w, got_w) <= GEMM_TOL_F32
    # the explicit column-wise copies give the same products
    if exact:
        assert torch.equal(dA_mn, dA_k) and torch.equal(dW_mn, dW_k)
    else:
        assert rel_fro(dA_k.float().cpu().numpy(), got) <= 1e-4
        assert rel_fro(dW_k.cpu().numpy(), got_w) <= 1e-4


def _many_groups(seed, E=1024):
    """Offsets of E groups, most of them empty, the rest one or two 128-row tiles."""
    sizes = np.random.default_rng(seed).choice([0, 128, 256], size=E, p=[0.7, 0.25, 0.05])
    return [0] + np.cumsum(sizes).tolist()


@pytest.mark.parametrize("offs", [[0, 128, 128, 512], [0, 384], _many_groups(41)], ids=["E3", "E1", "E1024"])
def test_gemm_fwd_blockwise(mgq, offs):
    """1x128 activation x 128x128 weight float32 block scales (promotion of
    every 128-deep partial product)."""
    rng = np.random.default_rng(41)
    dev = torch.device(DEV)
    E = len(offs) - 1
    N, K = (512, 640) if E < 1024 else (256, 256)
    Rp = offs[-1]
    R_cap = Rp + 128
    f = OF.E4M3
    ac = (rng.choice(f.pos_codes[:-1], size=(R_cap, K)) | (rng.integers(0, 2, (R_cap, K)) * 0x80)).astype(np.uint8)
    wc = (rng.choice(f.pos_codes[:-1], size=(E * N, K)) | (rng.integers(0, 2, (E * N, K)) * 0x80)).astype(np.uint8)
    sa = np.exp2(rng.uniform(-12, 4, size=(R_cap, K // 128))).astype(np.float32)      # scale_inv per 1x128
    sw = np.exp2(rng.uniform(-12, 0, size=(E, N // 128, K // 128))).astype(np.float32)
    Y = torch.full((R_cap, N), float("nan"), dtype=torch.bfloat16, device=dev)
    A = _op(mgq, ac, np.ascontiguousarray(sa.T), K, mgq.E4M3, dev)                   # [K/128][R_cap]
    Wo = _op(mgq, wc, sw, K, mgq.E4M3, dev)
    offd = torch.tensor(offs, dtype=torch.int32, device=dev)
    mgq.grouped_gemm_fwd(A, Wo, mgq.BLK_1x128_F32, offd, E, R_cap, N, K, Y)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    a_deq = OQ.dequantize_block_1x128(ac[:Rp], sa[:Rp])
    w_deq = np.stack([OQ.dequantize_block_128x128(wc[e * N:(e + 1) * N], sw[e]) for e in range(E)])
    ref = OG.grouped_gemm_fwd(a_deq, w_deq, np.array(offs))
    got = bf16_np(Y)
    assert np.all(np.isnan(got[Rp:]))
    assert rel_fro(OF.round_to_bf16(ref), got[:Rp]) <= GEMM_TOL_BF16


@pytest.mark.parametrize("offs", [[0, 128, 128, 512], [0, 256], _many_groups(51)], ids=["E3", "E1", "E1024"])
def test_gemm_fwd_nvfp4(mgq, offs):
    """e2m1 x e2m1 with 16-element ue4m3 block scales (kind::mxf4nvf4,
    scale_vec::4X) and a float32 global scale per tensor / per expert."""
    rng = np.random.default_rng(51)
    dev = torch.device(DEV)
    E = len(offs) - 1
    N, K = (512, 768) if E < 1024 else (256, 256)
    Rp = offs[-1]
    R_cap = Rp + 128
    qa = rng.integers(0, 16, size=(R_cap, K)).astype(np.uint8)
    qw = rng.integers(0, 16, size=(E * N, K)).astype(np.uint8)
    pack = lambda q: ((q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    sca = rng.integers(0x20, 0x58, size=(R_cap, K // 16)).astype(np.uint8)       # ue4m3 codes
    scw = rng.integers(0x20, 0x58, size=(E * N, K // 16)).astype(np.uint8)
    sga = np.array([2.5], dtype=np.float32)
    sgw = np.exp2(rng.uniform(-3, 3, size=E)).astype(np.float32)
    Y = torch.full((R_cap, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ga, gw = _to_dev(sga, dev), _to_dev(sgw, dev)
    A = _op(mgq, pack(qa), tile_mx_scales(sca), K, mgq.E2M1, dev)
    A.global_scale = ga.data_ptr()
    Wo = _op(mgq, pack(qw), tile_mx_scales(scw), K, mgq.E2M1, dev)
    Wo.global_scale = gw.data_ptr()
    offd = torch.tensor(offs, dtype=torch.int32, device=dev)
    mgq.grouped_gemm_fwd(A, Wo, mgq.NV16_UE4M3, offd, E, R_cap, N, K, Y)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    a_deq = OQ.dequantize_nvfp4(pack(qa)[:Rp], sca[:Rp], sga[0], K)
    # all experts in one call with s_g = 1, then each expert's 1 / s_g (the same
    # float64 values as one call per expert: v * sc / 1 is exact)
    w_deq = (OQ.dequantize_nvfp4(pack(qw), scw, 1.0, K).reshape(E, N, K)
             / sgw.astype(np.float64)[:, None, None])
    ref = OG.grouped_gemm_fwd(a_deq, w_deq, np.array(offs))
    got = bf16_np(Y)
    assert np.all(np.isnan(got[Rp:]))
    assert rel_fro(OF.round_to_bf16(ref), got[:Rp]) <= GEMM_TOL_BF16


def test_nvfp4_2d_weights_fwd_and_dgrad(mgq):
    """NVFP4 weights with 16x16 blocks in one pass (row-wise and column-wise
    copies, one amax pre-pass, s_g per expert) equal the oracle's; the forward
    GEMM on the row-wise copy and the dgrad on the column-wise copy (both read
    as ordinary 1x16 NVFP4 operands) equal the oracle's GEMMs of the
    dequantised operands."""
    rng = np.random.default_rng(71)
    dev = torch.device(DEV)
    E, N, K = 3, 256, 512
    offs = np.array([0, 128, 384, 512], dtype=np.int32)
    Rp = int(offs[-1])
    R_cap = Rp + 128
    w = _bf16(rng, (E, N, K), 0.02)
    w[1, 7, 100] = 0.5                                    # an outlier block in expert 1
    wf = bf16_np(w)
    rowc = torch.full((E, N, K // 2), 0xAB, dtype=torch.uint8, device=dev)
    rows = torch.full((mgq.nv_scale_bytes(E * N, K),), 0xCD, dtype=torch.uint8, device=dev)
    colc = torch.full((E, K, N // 2), 0xAB, dtype=torch.uint8, device=dev)
    cols = torch.full((mgq.nv_scale_bytes(E * K, N),), 0xCD, dtype=torch.uint8, device=dev)
    amax = torch.full((E,), -1.0, dtype=torch.float32, device=dev)
    sg = torch.zeros(E, dtype=torch.float32, device=dev)
    mgq.block_quantize(w.to(dev), mgq.qdesc(mgq.E2M1, mgq.NV16x16_UE4M3, rowc, rows, colc, cols,
                                            tensor_scale=sg, amax_out=amax))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    rs_all = untile_mx_scales(u8_np(rows), E * N, K, 16).reshape(E, N, K // 16)
    cs_all = untile_mx_scales(u8_np(cols), E * K, N, 16).reshape(E, K, N // 16)
    w_deq, wt_deq = [], []
    for e in range(E):
        am = float(np.max(np.abs(wf[e])))
        s_g = OQ.nvfp4_global_scale(am)
        assert float(amax[e].item()) == am and float(sg[e].item()) == float(s_g)
        rc, rs, cc, cs = OQ.quantize_nvfp4_2d(wf[e], s_g)
        assert np.array_equal(u8_np(rowc)[e], rc)
        assert np.array_equal(rs_all[e], rs)
        assert np.array_equal(u8_np(colc)[e], cc)
        assert np.array_equal(cs_all[e], cs)
        w_deq.append(OQ.dequantize_nvfp4(rc, rs, s_g, K))
        wt_deq.append(OQ.dequantize_nvfp4(cc, cs, s_g, N))
    w_deq, wt_deq = np.stack(w_deq), np.stack(wt_deq)
    assert np.array_equal(wt_deq, w_deq.transpose(0, 2, 1))

    def act(rows_, cols_, std):
        x = _bf16(rng, (rows_, cols_), std)
        x[Rp:] = 0
        c = torch.empty(rows_, cols_ // 2, dtype=torch.uint8, device=dev)
        sc = torch.empty(mgq.nv_scale_bytes(rows_, cols_), dtype=torch.uint8, device=dev)
        am, g = torch.empty(1, device=dev), torch.empty(1, device=dev)
        mgq.block_quantize(x.to(dev), mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, c, sc, tensor_scale=g, amax_out=am))
        torch.cuda.synchronize()
        op = _op(mgq, u8_np(c), u8_np(sc), cols_, mgq.E2M1, dev)
        op.global_scale = g.data_ptr()
        deq = OQ.dequantize_nvfp4(u8_np(c)[:Rp], untile_mx_scales(u8_np(sc), rows_, cols_, 16)[:Rp],
                                  np.float32(g.item()), cols_)
        return op, deq, (c, sc, g)

    offd = torch.from_numpy(offs).to(dev)
    A, a_deq, keep_a = act(R_cap, K, 1.0)
    W_row = _op(mgq, u8_np(rowc).reshape(E * N, K // 2), u8_np(rows), K, mgq.E2M1, dev)
    W_row.global_scale = sg.data_ptr()
    Y = torch.full((R_cap, N), float("nan"), dtype=torch.bfloat16, device=dev)
    mgq.grouped_gemm_fwd(A, W_row, mgq.NV16_UE4M3, offd, E, R_cap, N, K, Y)
    dY, dy_deq, keep_dy = act(R_cap, N, 1e-3)
    W_col = _op(mgq, u8_np(colc).reshape(E * K, N // 2), u8_np(cols), N, mgq.E2M1, dev)
    W_col.global_scale = sg.data_ptr()
    dA = torch.full((R_cap, K), float("nan"), dtype=torch.bfloat16, device=dev)
    mgq.grouped_gemm_dgrad(dY, W_col, mgq.NV16_UE4M3, offd, E, R_cap, N, K, dA)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    ref = OG.grouped_gemm_fwd(a_deq, w_deq, offs)
    assert rel_fro(OF.round_to_bf16(ref), bf16_np(Y)[:Rp]) <= GEMM_TOL_BF16
    ref_d = OG.grouped_gemm_dgrad(dy_deq, w_deq, offs)
    assert rel_fro(OF.round_to_bf16(ref_d), bf16_np(dA)[:Rp]) <= GEMM_TOL_BF16


def _nv_operand(rng, rows, cols):
    """Random e2m1 codes [rows, cols] packed along cols, random ue4m3 block
    scales [rows, cols/16]."""
    q = rng.integers(0, 16, size=(rows, cols)).astype(np.uint8)
    packed = ((q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    sc = rng.integers(0x20, 0x58, size=(rows, cols // 16)).astype(np.uint8)
    return packed, sc


def test_gemm_wgrad_nvfp4(mgq):
    """NVFP4 wgrad: dW_e = sum over the rows of group e of dY^T A, from the
    column-wise copies dYcol [N, R_cap] and Acol [K, R_cap] (e2m1 packed along
    the rows, 16-row ue4m3 blocks, one global scale each); groups of whole
    256-row stages, one empty (zeros with beta 0, kept with beta 1)."""
    rng = np.random.default_rng(73)
    dev = torch.device(DEV)
    offs = np.array([0, 256, 256, 768], dtype=np.int32)
    E, N, K = 3, 256, 512
    Rp = int(offs[-1])
    R_cap = Rp + 256
    dyt, dyts = _nv_operand(rng, N, R_cap)
    at, ats = _nv_operand(rng, K, R_cap)
    sg_dy = np.array([1.5e4], dtype=np.float32)
    sg_a = np.array([3.0], dtype=np.float32)
    A_op = _op(mgq, dyt, tile_mx_scales(dyts), R_cap, mgq.E2M1, dev)
    B_op = _op(mgq, at, tile_mx_scales(ats), R_cap, mgq.E2M1, dev)
    gdy, ga = _to_dev(sg_dy, dev), _to_dev(sg_a, dev)
    A_op.global_scale = gdy.data_ptr()
    B_op.global_scale = ga.data_ptr()
    offd = torch.from_numpy(offs).to(dev)
    dW = torch.full((E, N, K), 5.0, dtype=torch.float32, device=dev)
    mgq.grouped_gemm_wgrad(A_op, B_op, mgq.NV16_UE4M3, offd, E, R_cap, N, K, dW, 0.0)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    dy_deq = OQ.dequantize_nvfp4(dyt, dyts, sg_dy[0], R_cap).T[:Rp]
    a_deq = OQ.dequantize_nvfp4(at, ats, sg_a[0], R_cap).T[:Rp]
    ref = OG.grouped_gemm_wgrad(dy_deq, a_deq, offs, E)
    got = dW.cpu().numpy().astype(np.float64)
    assert np.all(got[1] == 0.0)
    assert rel_fro(ref, got) <= GEMM_TOL_F32
    prev = torch.from_numpy(rng.standard_normal((E, N, K)).astype(np.float32)).to(dev)
    dW2 = prev.clone()
    mgq.grouped_gemm_wgrad(A_op, B_op, mgq.NV16_UE4M3, offd, E, R_cap, N, K, dW2, 1.0)
    torch.cuda.synchronize()
    got2 = dW2.cpu().numpy().astype(np.float64)
    assert np.array_equal(got2[1], prev[1].cpu().numpy().astype(np.float64))
    assert rel_fro(ref + prev.cpu().numpy(), got2) <= GEMM_TOL_F32


def test_nv_scale_image_gemms_identical(mgq):
    """The scale image of an NVFP4 operand holds each 512-byte scale chunk four
    times in order; the grouped GEMMs fed the image (fwd and dgrad in rows mode,
    wgrad in contract mode) give the same bits as those fed the scales alone."""
    rng = np.random.default_rng(75)
    dev = torch.device(DEV)
    offs = np.array([0, 256, 256, 768], dtype=np.int32)
    E, N, K = 3, 512, 768
    Rp = int(offs[-1])
    R_cap = Rp + 256
    offd = torch.from_numpy(offs).to(dev)

    def nv_op(rows, cols, g):
        c, s = _nv_operand(rng, rows, cols)
        st = tile_mx_scales(s)
        op = _op(mgq, c, st, cols, mgq.E2M1, dev)
        op.global_scale = g.data_ptr()
        img = torch.full((mgq.nv_scale_image_bytes(rows, cols),), 0xEE, dtype=torch.uint8, device=dev)
        mgq.nv_scale_image(op.scale, rows, cols, img)
        torch.cuda.synchronize()
        assert mgq.get_error() == mgq.OK
        assert np.array_equal(u8_np(img), np.repeat(st.reshape(-1, 512), 4, axis=0).reshape(-1))
        return op, img

    ga = _to_dev(np.array([2.5], dtype=np.float32), dev)
    gw = _to_dev(np.exp2(rng.uniform(-3, 3, size=E)).astype(np.float32), dev)
    # forward: A [R_cap, K], W [E * N, K]
    A, _ = nv_op(R_cap, K, ga)
    W, w_img = nv_op(E * N, K, gw)
    outs = []
    for img in (None, w_img):
        W.scale_image = 0 if img is None else img.data_ptr()
        Y = torch.full((R_cap, N), float("nan"), dtype=torch.bfloat16, device=dev)
        mgq.grouped_gemm_fwd(A, W, mgq.NV16_UE4M3, offd, E, R_cap, N, K, Y)
        torch.cuda.synchronize()
        assert mgq.get_error() == mgq.OK
        outs.append(bf16_np(Y)[:Rp])
    assert np.array_equal(outs[0], outs[1])
    # dgrad: dY [R_cap, N], Wcol [E * K, N]
    dY, _ = nv_op(R_cap, N, ga)
    Wc, wc_img = nv_op(E * K, N, gw)
    outs = []
    for img in (None, wc_img):
        Wc.scale_image = 0 if img is None else img.data_ptr()
        dA = torch.full((R_cap, K), float("nan"), dtype=torch.bfloat16, device=dev)
        mgq.grouped_gemm_dgrad(dY, Wc, mgq.NV16_UE4M3, offd, E, R_cap, N, K, dA)
        torch.cuda.synchronize()
        assert mgq.get_error() == mgq.OK
        outs.append(bf16_np(dA)[:Rp])
    assert np.array_equal(outs[0], outs[1])
    # wgrad: dYcol [N, R_cap], Acol [K, R_cap]
    dYc, _ = nv_op(N, R_cap, ga)
    Ac, ac_img = nv_op(K, R_cap, ga)
    outs = []
    for img in (None, ac_img):
        Ac.scale_image = 0 if img is None else img.data_ptr()
        dW = torch.full((E, N, K), 5.0, dtype=torch.float32, device=dev)
        mgq.grouped_gemm_wgrad(dYc, Ac, mgq.NV16_UE4M3, offd, E, R_cap, N, K, dW, 0.0)
        torch.cuda.synchronize()
        assert mgq.get_error() == mgq.OK
        outs.append(dW.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


def test_gemm_wgrad_nvfp4_needs_256_row_groups(mgq):
    """A group boundary inside a 256-row e2m1 stage is reported by the kernel
    (MGQ_ERR_INVALID_ARG through the error word) and nothing is written."""
    rng = np.random.default_rng(74)
    dev = torch.device(DEV)
    offs = np.array([0, 128, 512], dtype=np.int32)
    E, N, K = 2, 256, 256
    R_cap = 512
    dyt, dyts = _nv_operand(rng, N, R_cap)
    at, ats = _nv_operand(rng, K, R_cap)
    A_op = _op(mgq, dyt, tile_mx_scales(dyts), R_cap, mgq.E2M1, dev)
    B_op = _op(mgq, at, tile_mx_scales(ats), R_cap, mgq.E2M1, dev)
    g1 = torch.ones(1, device=dev)
    A_op.global_scale = g1.data_ptr()
    B_op.global_scale = g1.data_ptr()
    dW = torch.full((E, N, K), 5.0, dtype=torch.float32, device=dev)
    mgq.grouped_gemm_wgrad(A_op, B_op, mgq.NV16_UE4M3, torch.from_numpy(offs).to(dev), E, R_cap, N, K, dW, 0.0)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.ERR_INVALID_ARG
    assert torch.all(dW == 5.0).item()


def test_gemm_grouped_equals_per_group(mgq):
    """The grouped call equals single-group calls on each expert's rows
    (grouped vs discrete comparison of Megatron-LM PR #5487's test matrix),
    bit for bit."""
    rng = np.random.default_rng(31)
    dev = torch.device(DEV)
    offs = np.array([0, 256, 384, 768], dtype=np.int32)
    E, N, K = 3, 256, 512
    Rp = int(offs[-1])
    ac, asc = _mx_operand(rng, Rp, K)
    wc, wsc = _mx_operand(rng, E * N, K)
    Y = torch.empty(Rp, N, dtype=torch.bfloat16, device=dev)
    A = _op(mgq, ac, tile_mx_scales(asc), K, mgq.E4M3, dev)
    Wo = _op(mgq, wc, tile_mx_scales(wsc), K, mgq.E4M3, dev)
    offd = torch.from_numpy(offs).to(dev)
    mgq.grouped_gemm_fwd(A, Wo, mgq.MX32_E8M0, offd, E, Rp, N, K, Y)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        Ye = torch.empty(hi - lo, N, dtype=torch.bfloat16, device=dev)
        Ae = _op(mgq, ac[lo:hi], tile_mx_scales(asc[lo:hi]), K, mgq.E4M3, dev)
        We = _op(mgq, wc[e * N:(e + 1) * N], tile_mx_scales(wsc[e * N:(e + 1) * N]), K, mgq.E4M3, dev)
        mgq.grouped_gemm_fwd(Ae, We, mgq.MX32_E8M0, torch.tensor([0, hi - lo], dtype=torch.int32, device=dev), 1,
                             hi - lo, N, K, Ye)
        torch.cuda.synchronize()
        assert torch.equal(Ye, Y[lo:hi])


def test_gemm_misaligned_offsets_reported(mgq):
    dev = torch.device(DEV)
    rng = np.random.default_rng(3)
    ac, asc = _mx_operand(rng, 256, 128)
    wc, wsc = _mx_operand(rng, 2 * 256, 128)
    Y = torch.zeros(256, 256, dtype=torch.bfloat16, device=dev)
    A = _op(mgq, ac, tile_mx_scales(asc), 128, mgq.E4M3, dev)
    Wo = _op(mgq, wc, tile_mx_scales(wsc), 128, mgq.E4M3, dev)
    mgq.grouped_gemm_fwd(A, Wo, mgq.MX32_E8M0, torch.tensor([0, 100, 256], dtype=torch.int32, device=dev), 2,
                         256, 256, 128, Y)
    assert mgq.get_error() == mgq.ERR_INVALID_ARG
    assert torch.count_nonzero(Y).item() == 0          # nothing written


# ---------------------------------------------------------------------------- elementwise

def _layout(rng, T, E, k, dev, align=128):
    idx = _routing(rng, T, E, k, ())
    rim, src, off, cnt = OR.permute_indices(idx, E, align)
    return idx, rim, src, off, cnt


@pytest.mark.parametrize("mode", ["mx", "tensor", "mx_col", "nvfp4_col"])
@pytest.mark.parametrize("F", [512, 768, 1536])
def test_swiglu_quantize(mgq, mode, F):
    rng = np.random.default_rng(F)
    dev = torch.device(DEV)
    off = np.array([0, 128, 384], dtype=np.int32)
    R = 512
    gu = _bf16(rng, (R, 2 * F), 2.0)
    gu[off[-1]:] = 0
    offd = torch.from_numpy(off).to(dev)
    codes = torch.empty(R, F // 2 if mode.startswith("nvfp4") else F, dtype=torch.uint8, device=dev)
    h = torch.empty(R, F, dtype=torch.bfloat16, device=dev)
    if mode == "nvfp4_col":
        sc = torch.empty(mgq.nv_scale_bytes(R, F), dtype=torch.uint8, device=dev)
        col = torch.full((F, R // 2), 0xAB, dtype=torch.uint8, device=dev)
        csc = torch.full((mgq.nv_scale_bytes(F, R),), 0xCD, dtype=torch.uint8, device=dev)
        amax, sg = torch.full((1,), 7.0, device=dev), torch.zeros(1, device=dev)
        q = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, codes, sc, col, csc, tensor_scale=sg, amax_out=amax)
    elif mode == "mx":
        sc = torch.empty(mgq.mx_scale_bytes(R, F), dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, codes, sc)
    elif mode == "mx_col":
        sc = torch.empty(mgq.mx_scale_bytes(R, F), dtype=torch.uint8, device=dev)
        col = torch.full((F, R), 0xAB, dtype=torch.uint8, device=dev)
        csc = torch.full((mgq.mx_scale_bytes(F, R),), 0xCD, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, codes, sc, col, csc)
    else:
        s = torch.tensor([20.0], device=dev)
        amax = torch.zeros(1, device=dev)
        col = torch.empty(F, R, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E4M3, mgq.TENSOR_F32, codes, None, col, None, s, amax)
    mgq.swiglu_quantize(gu.to(dev), R, F, offd, 2, q, h)
    torch.cuda.synchronize()
    n = int(off[-1])
    hg = bf16_np(h)[:n]
    check_elementwise(OL.swiglu(bf16_np(gu)[:n], F), hg, "swiglu")
    if mode == "nvfp4_col":
        am = float(np.max(np.abs(hg)))
        s_g = OQ.nvfp4_global_scale(am)
        assert float(amax.item()) == am and float(sg.item()) == float(s_g)
        c, s_ = OQ.quantize_nvfp4(hg, s_g)
        assert np.array_equal(u8_np(codes)[:n], c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), R, F, 16)[:n], s_)
        cc, cs = OQ.quantize_nvfp4(hg.T, s_g)
        assert np.array_equal(u8_np(col)[:, :n // 2], cc)
        assert np.array_equal(untile_mx_scales(u8_np(csc), F, R, 16)[:, :n // 16], cs)
    elif mode in ("mx", "mx_col"):
        c, s_ = OQ.quantize_mx(hg)
        assert np.array_equal(u8_np(codes)[:n], c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), R, F)[:n], s_)
        if mode == "mx_col":
            # column-wise: blocks of 32 along the rows (row groups are 128-aligned)
            cc, cs = OQ.quantize_mx(hg.T)
            assert np.array_equal(u8_np(col)[:, :n], cc)
            assert np.array_equal(untile_mx_scales(u8_np(csc), F, R)[:, :n // 32], cs)
    else:
        c, am = OQ.quantize_tensor(hg, np.float32(20.0))
        assert np.array_equal(u8_np(codes)[:n], c)
        assert np.array_equal(u8_np(col)[:, :n], c.T)
        assert float(amax.item()) == am


@pytest.mark.parametrize("mode", ["tensor", "mx_col", "nvfp4", "nvfp4_col"])
def test_dswiglu_quantize(mgq, mode):
    rng = np.random.default_rng(5)
    dev = torch.device(DEV)
    F, R = 768, 384
    off = np.array([0, 256, 384], dtype=np.int32)
    gu = _bf16(rng, (R, 2 * F), 2.0)
    dh = _bf16(rng, (R, F), 1e-3)
    nv = mode.startswith("nvfp4")
    codes = torch.empty(R, F if nv else 2 * F, dtype=torch.uint8, device=dev)
    col = torch.empty(2 * F, R // 2 if nv else R, dtype=torch.uint8, device=dev)
    dgu = torch.empty(R, 2 * F, dtype=torch.bfloat16, device=dev)
    s = torch.tensor([20000.0], device=dev)
    amax = torch.zeros(1, device=dev)
    if nv:
        sc = torch.empty(mgq.nv_scale_bytes(R, 2 * F), dtype=torch.uint8, device=dev)
        csc = torch.empty(mgq.nv_scale_bytes(2 * F, R), dtype=torch.uint8, device=dev)
        sg = torch.zeros(1, device=dev)
        q = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, codes, sc, col if mode == "nvfp4_col" else None,
                      csc if mode == "nvfp4_col" else None, tensor_scale=sg, amax_out=amax)
    elif mode == "tensor":
        q = mgq.qdesc(mgq.E5M2, mgq.TENSOR_F32, codes, None, col, None, s, amax)
    else:
        sc = torch.empty(mgq.mx_scale_bytes(R, 2 * F), dtype=torch.uint8, device=dev)
        csc = torch.empty(mgq.mx_scale_bytes(2 * F, R), dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E5M2, mgq.MX32_E8M0, codes, sc, col, csc)
    mgq.dswiglu_quantize(dh.to(dev), gu.to(dev), R, F, torch.from_numpy(off).to(dev), 2, q, dgu)
    torch.cuda.synchronize()
    g = bf16_np(dgu)
    check_elementwise(OL.dswiglu(bf16_np(dh), bf16_np(gu), F), g, "dswiglu")
    if nv:
        n = int(off[-1])
        gn = g[:n]
        am = float(np.max(np.abs(gn)))
        s_g = OQ.nvfp4_global_scale(am)
        assert float(amax.item()) == am and float(sg.item()) == float(s_g)
        c, s_ = OQ.quantize_nvfp4(gn, s_g)
        assert np.array_equal(u8_np(codes)[:n], c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), R, 2 * F, 16)[:n], s_)
        if mode == "nvfp4_col":
            cc, cs = OQ.quantize_nvfp4(gn.T, s_g)
            assert np.array_equal(u8_np(col)[:, :n // 2], cc)
            assert np.array_equal(untile_mx_scales(u8_np(csc), 2 * F, R, 16)[:, :n // 16], cs)
    elif mode == "tensor":
        c, am = OQ.quantize_tensor(g, np.float32(20000.0), "e5m2")
        assert np.array_equal(u8_np(codes), c)
        assert np.array_equal(u8_np(col), c.T)
        assert float(amax.item()) == am
    else:
        c, s_ = OQ.quantize_mx(g, "e5m2")
        assert np.array_equal(u8_np(codes), c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), R, 2 * F), s_)
        cc, cs = OQ.quantize_mx(g.T, "e5m2")
        assert np.array_equal(u8_np(col), cc)
        assert np.array_equal(untile_mx_scales(u8_np(csc), 2 * F, R), cs)


@pytest.mark.parametrize("mode", ["tensor", "mx_col"])
def test_dswiglu_quantize_partial_tile(mgq, mode):
    """Rows in use end inside a 128-row tile (320 of R_cap = 512) and the
    buffers hold NaN past them: the row-wise codes and dG | dU cover the rows
    in use, and the column-wise copy treats the rest of the last tile as zeros
    (zero codes and scales), as the oracle's blocks of the zero-filled tile."""
    rng = np.random.default_rng(9)
    dev = torch.device(DEV)
    F, R, n = 768, 512, 320
    off = np.array([0, 256, n], dtype=np.int32)
    gu = _bf16(rng, (R, 2 * F), 2.0)
    dh = _bf16(rng, (R, F), 1e-3)
    gu[n:] = float("nan")
    dh[n:] = float("nan")
    codes = torch.full((R, 2 * F), 0xAB, dtype=torch.uint8, device=dev)
    col = torch.full((2 * F, R), 0xAB, dtype=torch.uint8, device=dev)
    dgu = torch.zeros(R, 2 * F, dtype=torch.bfloat16, device=dev)
    amax = torch.zeros(1, device=dev)
    s = torch.tensor([20000.0], device=dev)              # (kept alive: the descriptor holds its address)
    if mode == "tensor":
        q = mgq.qdesc(mgq.E5M2, mgq.TENSOR_F32, codes, None, col, None, s, amax)
    else:
        sc = torch.full((mgq.mx_scale_bytes(R, 2 * F),), 0xAB, dtype=torch.uint8, device=dev)
        csc = torch.full((mgq.mx_scale_bytes(2 * F, R),), 0xAB, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E5M2, mgq.MX32_E8M0, codes, sc, col, csc)
    mgq.dswiglu_quantize(dh.to(dev), gu.to(dev), R, F, torch.from_numpy(off).to(dev), 2, q, dgu)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    g = bf16_np(dgu)[:n]
    check_elementwise(OL.dswiglu(bf16_np(dh)[:n], bf16_np(gu)[:n], F), g, "dswiglu")
    gz = np.zeros((384, 2 * F), dtype=g.dtype)          # the three tiles in use, zero past n
    gz[:n] = g
    if mode == "tensor":
        c, am = OQ.quantize_tensor(gz, np.float32(20000.0), "e5m2")
        assert np.array_equal(u8_np(codes)[:n], c[:n])
        assert np.array_equal(u8_np(col)[:, :384], c.T)
        assert float(amax.item()) == am
    else:
        c, s_ = OQ.quantize_mx(gz, "e5m2")
        assert np.array_equal(u8_np(codes)[:n], c[:n])
        assert np.array_equal(untile_mx_scales(u8_np(sc), R, 2 * F)[:n], s_[:n])
        cc, cs = OQ.quantize_mx(gz.T, "e5m2")
        assert np.array_equal(u8_np(col)[:, :384], cc)
        assert np.array_equal(untile_mx_scales(u8_np(csc), 2 * F, R)[:, :384 // 32], cs)


@pytest.mark.parametrize("T,E,k,H", [(1000, 8, 2, 512), (333, 16, 8, 256), (64, 4, 1, 5120)])
def test_unpermute_and_permute_bwd(mgq, T, E, k, H):
    rng = np.random.default_rng(T)
    dev = torch.device(DEV)
    idx, rim, src, off, cnt = _layout(rng, T, E, k, dev)
    Rp = int(off[-1])
    y = _bf16(rng, (Rp, H))
    probs = rng.random((T, k)).astype(np.float32)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    rimd = torch.from_numpy(rim).to(dev)
    mgq.moe_unpermute(y.to(dev), rimd, torch.from_numpy(probs).to(dev), out)
    dx = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    mgq.moe_permute_bwd(y.to(dev), rimd, dx)
    torch.cuda.synchronize()
    check_elementwise(OR.unpermute(bf16_np(y), rim, probs), bf16_np(out), "unpermute")
    check_elementwise(OR.permute_bwd(bf16_np(y), rim), bf16_np(dx), "permute_bwd")


@pytest.mark.parametrize("H", [1024, 384])      # (384: a partial 1024-element chunk per row)
@pytest.mark.parametrize("mode", ["tensor", "mx", "mx_col", "nvfp4", "nvfp4_col"])
def test_unpermute_bwd_quantize(mgq, mode, H):
    rng = np.random.default_rng(9)
    dev = torch.device(DEV)
    T, E, k = 700, 8, 2
    idx, rim, src, off, cnt = _layout(rng, T, E, k, dev)
    Rp = int(off[-1])
    R = Rp + 128
    dout = _bf16(rng, (T, H), 1e-3)
    y = _bf16(rng, (R, H))
    probs = rng.random((T, k)).astype(np.float32)
    nv = mode.startswith("nvfp4")
    codes = torch.full((R, H // 2 if nv else H), 0xAB, dtype=torch.uint8, device=dev)
    dprobs = torch.empty(T, k, dtype=torch.float32, device=dev)
    if nv:
        sc = torch.full((mgq.nv_scale_bytes(R, H),), 0xCD, dtype=torch.uint8, device=dev)
        amax = torch.full((1,), 7.0, device=dev)
        sg = torch.zeros(1, device=dev)
        col = csc = None
        if mode == "nvfp4_col":
            col = torch.full((H, R // 2), 0xAB, dtype=torch.uint8, device=dev)
            csc = torch.full((mgq.nv_scale_bytes(H, R),), 0xCD, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, codes, sc, col, csc, tensor_scale=sg, amax_out=amax)
    elif mode == "tensor":
        col = torch.empty(H, R, dtype=torch.uint8, device=dev)
        s = torch.tensor([30000.0], device=dev)
        amax = torch.zeros(1, device=dev)
        q = mgq.qdesc(mgq.E5M2, mgq.TENSOR_F32, codes, None, col, None, s, amax)
    elif mode == "mx_col":
        sc = torch.full((mgq.mx_scale_bytes(R, H),), 0xCD, dtype=torch.uint8, device=dev)
        col = torch.full((H, R), 0xAB, dtype=torch.uint8, device=dev)
        csc = torch.full((mgq.mx_scale_bytes(H, R),), 0xCD, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E5M2, mgq.MX32_E8M0, codes, sc, col, csc)
    else:
        sc = torch.full((mgq.mx_scale_bytes(R, H),), 0xCD, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E5M2, mgq.MX32_E8M0, codes, sc)
    mgq.moe_unpermute_bwd(dout.to(dev), y.to(dev), torch.from_numpy(rim).to(dev), torch.from_numpy(src).to(dev),
                          torch.from_numpy(probs).to(dev), R, torch.from_numpy(off).to(dev), E, q, dprobs)
    torch.cuda.synchronize()
    dy32, dp = OR.unpermute_bwd(bf16_np(dout), bf16_np(y), rim, probs, Rp)
    assert rel_fro(dp, dprobs.cpu().numpy()) <= 1e-5
    if nv:
        am = float(np.max(np.abs(dy32)))
        s_g = OQ.nvfp4_global_scale(am)
        assert float(amax.item()) == am and float(sg.item()) == float(s_g)
        c, s_ = OQ.quantize_nvfp4(dy32.astype(np.float64), s_g)
        assert np.array_equal(u8_np(codes)[:Rp], c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), R, H, 16)[:Rp], s_)
        if mode == "nvfp4_col":
            cc, cs = OQ.quantize_nvfp4(dy32.astype(np.float64).T, s_g)
            assert np.array_equal(u8_np(col)[:, :Rp // 2], cc)
            assert np.array_equal(untile_mx_scales(u8_np(csc), H, R, 16)[:, :Rp // 16], cs)
    elif mode == "tensor":
        c, am = OQ.quantize_tensor(dy32.astype(np.float64), np.float32(30000.0), "e5m2")
        assert np.array_equal(u8_np(codes)[:Rp], c)
        assert np.array_equal(u8_np(col)[:, :Rp], c.T)
        assert float(amax.item()) == am
    else:
        c, s_ = OQ.quantize_mx(dy32.astype(np.float64), "e5m2")
        assert np.array_equal(u8_np(codes)[:Rp], c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), R, H)[:Rp], s_)
        if mode == "mx_col":
            cc, cs = OQ.quantize_mx(dy32.astype(np.float64).T, "e5m2")
            assert np.array_equal(u8_np(col)[:, :Rp], cc)
            assert np.array_equal(untile_mx_scales(u8_np(csc), H, R)[:, :Rp // 32], cs)


@pytest.mark.parametrize("fmt,e8m0", [("e4m3", "rceil"), ("e5m2", "rceil"), ("e4m3", "floor"), ("e5m2", "floor")])
def test_block_quantize_mx_special_values(mgq, fmt, e8m0):
    """Row- and column-wise MX codes of a tile pass over NaN, +-inf, signed
    zeros, bf16 subnormals, an all-subnormal block and the largest bf16 values
    equal the oracle's (a NaN / inf block: scale 0xFF and NaN codes)."""
    rng = np.random.default_rng(29)
    dev = torch.device(DEV)
    G, M, K = 2, 256, 256
    w = rng.standard_normal((G, M, K)).astype(np.float32) * 0.02
    w[0, 0, 5] = np.nan                       # NaN: row block (0, 0) and column block (5, 0)
    w[0, 40, 1] = np.inf
    w[0, 70, 140] = -np.inf
    w[1, 3, 200] = -0.0
    w[1, 10, 0:32] = rng.standard_normal(32) * 1e-39          # an all-subnormal row block
    w[1, 64:96, 9] = rng.standard_normal(32) * 2e-39          # an all-subnormal column block
    w[1, 20, :] = 0.0
    w[1, 30, 64:96] = 3.38e38 * np.sign(rng.standard_normal(32))   # near the largest bf16
    w[0, 100, 7] = 1e-39                                      # subnormals among normal values
    w[0, 101, 7] = -4e-40
    wt = torch.from_numpy(w).to(torch.bfloat16)
    wf = bf16_np(wt)
    dt = mgq.E4M3 if fmt == "e4m3" else mgq.E5M2
    mode = mgq.RCEIL if e8m0 == "rceil" else mgq.FLOOR
    codes = torch.empty(G, M, K, dtype=torch.uint8, device=dev)
    sc = torch.empty(mgq.mx_scale_bytes(G * M, K), dtype=torch.uint8, device=dev)
    col = torch.empty(G, K, M, dtype=torch.uint8, device=dev)
    csc = torch.empty(mgq.mx_scale_bytes(G * K, M), dtype=torch.uint8, device=dev)
    mgq.block_quantize(wt.to(dev), mgq.qdesc(dt, mgq.MX32_E8M0, codes, sc, col, csc, e8m0_mode=mode))
    torch.cuda.synchronize()
    c, s_ = OQ.quantize_mx(wf.reshape(G * M, K), fmt, e8m0)
    assert np.array_equal(u8_np(codes).reshape(G * M, K), c)
    assert np.array_equal(untile_mx_scales(u8_np(sc), G * M, K), s_)
    cs_all = untile_mx_scales(u8_np(csc), G * K, M).reshape(G, K, M // 32)
    for g in range(G):
        cc, cs = OQ.quantize_mx(wf[g].T, fmt, e8m0)
        assert np.array_equal(u8_np(col)[g], cc)
        assert np.array_equal(cs_all[g], cs)
    assert s_[0, 0] == 255 and s_[40, 0] == 255                 # the NaN and inf blocks


@pytest.mark.parametrize("mode", ["mx", "tensor", "blk128", "nvfp4", "mx_col", "nvfp4_col"])
def test_block_quantize_weights(mgq, mode):
    rng = np.random.default_rng(13)
    dev = torch.device(DEV)
    G, M, K = 3, 256, 640
    w = _bf16(rng, (G, M, K), 0.02)
    codes = torch.empty(G, M, K, dtype=torch.uint8, device=dev)
    wf = bf16_np(w)
    if mode == "mx_col":
        # row-wise MX (blocks along K) and column-wise MX (blocks of 32 along
        # each expert's rows, stored transposed [G, K, M]) in one pass
        wf = bf16_np(w)
        sc = torch.empty(mgq.mx_scale_bytes(G * M, K), dtype=torch.uint8, device=dev)
        col = torch.empty(G, K, M, dtype=torch.uint8, device=dev)
        csc = torch.empty(mgq.mx_scale_bytes(G * K, M), dtype=torch.uint8, device=dev)
        mgq.block_quantize(w.to(dev), mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, codes, sc, col, csc))
        torch.cuda.synchronize()
        c, s_ = OQ.quantize_mx(wf.reshape(G * M, K))
        assert np.array_equal(u8_np(codes).reshape(G * M, K), c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), G * M, K), s_)
        cs_all = untile_mx_scales(u8_np(csc), G * K, M).reshape(G, K, M // 32)
        for g in range(G):
            cc, cs = OQ.quantize_mx(wf[g].T)
            assert np.array_equal(u8_np(col)[g], cc)
            assert np.array_equal(cs_all[g], cs)
        return
    if mode == "nvfp4_col":
        # 1x16 blocks along K (rows) and along each group's M rows (columns)
        w[2, 100, 9] = -0.75
        wf = bf16_np(w)
        cnv = torch.empty(G, M, K // 2, dtype=torch.uint8, device=dev)
        sc = torch.empty(mgq.nv_scale_bytes(G * M, K), dtype=torch.uint8, device=dev)
        col = torch.full((G, K, M // 2), 0xAB, dtype=torch.uint8, device=dev)
        csc = torch.full((mgq.nv_scale_bytes(G * K, M),), 0xCD, dtype=torch.uint8, device=dev)
        amax = torch.empty(G, dtype=torch.float32, device=dev)
        sg = torch.empty(G, dtype=torch.float32, device=dev)
        mgq.block_quantize(w.to(dev), mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, cnv, sc, col, csc, tensor_scale=sg,
                                                amax_out=amax))
        torch.cuda.synchronize()
        s_all = untile_mx_scales(u8_np(sc), G * M, K, 16).reshape(G, M, K // 16)
        cs_all = untile_mx_scales(u8_np(csc), G * K, M, 16).reshape(G, K, M // 16)
        for g in range(G):
            am = float(np.max(np.abs(wf[g])))
            s_g = OQ.nvfp4_global_scale(am)
            assert float(amax[g].item()) == am and float(sg[g].item()) == float(s_g)
            c, s_ = OQ.quantize_nvfp4(wf[g], s_g)
            assert np.array_equal(u8_np(cnv)[g], c)
            assert np.array_equal(s_all[g], s_)
            cc, cs = OQ.quantize_nvfp4(wf[g].T, s_g)
            assert np.array_equal(u8_np(col)[g], cc)
            assert np.array_equal(cs_all[g], cs)
        return
    if mode == "nvfp4":
        w[0, 3, 4] = 0.5
        wf = bf16_np(w)
        cnv = torch.empty(G, M, K // 2, dtype=torch.uint8, device=dev)
        sc = torch.empty(mgq.nv_scale_bytes(G * M, K), dtype=torch.uint8, device=dev)
        amax = torch.empty(G, dtype=torch.float32, device=dev)
        sg = torch.empty(G, dtype=torch.float32, device=dev)
        mgq.block_quantize(w.to(dev), mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, cnv, sc, tensor_scale=sg, amax_out=amax))
        torch.cuda.synchronize()
        s_all = untile_mx_scales(u8_np(sc), G * M, K, 16).reshape(G, M, K // 16)
        for g in range(G):
            am = float(np.max(np.abs(wf[g])))
            s_g = OQ.nvfp4_global_scale(am)
            assert float(amax[g].item()) == am and float(sg[g].item()) == float(s_g)
            c, s_ = OQ.quantize_nvfp4(wf[g], s_g)
            assert np.array_equal(u8_np(cnv)[g], c)
            assert np.array_equal(s_all[g], s_)
        return
    if mode == "blk128":
        w[1, 5, 7] = 3.0                                   # one large element in one tile
        w[2] = 0                                           # all-zero tiles: scale 1
        wf = bf16_np(w)
        sc = torch.empty(G, M // 128, K // 128, dtype=torch.float32, device=dev)
        mgq.block_quantize(w.to(dev), mgq.qdesc(mgq.E4M3, mgq.BLK_128x128_F32, codes, sc))
        torch.cuda.synchronize()
        for g in range(G):
            c, si = OQ.quantize_block_128x128(wf[g])
            assert np.array_equal(u8_np(codes)[g], c)
            assert np.array_equal(sc[g].cpu().numpy(), si)
    elif mode == "mx":
        sc = torch.empty(mgq.mx_scale_bytes(G * M, K), dtype=torch.uint8, device=dev)
        mgq.block_quantize(w.to(dev), mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, codes, sc))
        torch.cuda.synchronize()
        c, s_ = OQ.quantize_mx(wf.reshape(G * M, K))
        assert np.array_equal(u8_np(codes).reshape(G * M, K), c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), G * M, K), s_)
    else:
        s = torch.tensor([1000.0, 2000.0, 7.5], device=dev)
        amax = torch.zeros(G, device=dev)
        col = torch.empty(G, K, M, dtype=torch.uint8, device=dev)
        mgq.block_quantize(w.to(dev), mgq.qdesc(mgq.E4M3, mgq.TENSOR_F32, codes, None, col, None, s, amax))
        torch.cuda.synchronize()
        for g in range(G):
            c, am = OQ.quantize_tensor(wf[g], np.float32(s[g].item()))
            assert np.array_equal(u8_np(codes)[g], c)
            assert np.array_equal(u8_np(col)[g], c.T)
            assert float(amax[g].item()) == am


def test_amax_history_update(mgq):
    dev = torch.device(DEV)
    L, n = 4, 3
    hist = torch.zeros(n, L, device=dev)
    head = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = torch.ones(n, device=dev)
    ref = [OL.DelayedScaling("e4m3", L) for _ in range(n)]
    rng = np.random.default_rng(0)
    for step in range(9):
        a = rng.random(n).astype(np.float32) * (10 if step != 3 else 100)
        if step == 0:
            a[1] = 0.0
        amax = torch.from_numpy(a).to(dev)
        mgq.amax_history_update(hist, head, amax, scale, 448.0)
        torch.cuda.synchronize()
        for i in range(n):
            ref[i].update(a[i])
        assert np.array_equal(scale.cpu().numpy(), np.array([r.scale for r in ref], dtype=np.float32))
        assert torch.count_nonzero(amax).item() == 0


@pytest.mark.parametrize("scaling", ["tensor", "mx", "mx_col", "mx_col_e5m2_floor", "nvfp4"])
def test_gemm_fwd_swiglu_equals_separate_steps(mgq, scaling):
    """The gate/up GEMM with SwiGLU + quantisation in its epilogue writes the
    same bytes as grouped_gemm_fwd followed by swiglu_quantize: g | u, h, the
    h codes and scales, the per-tensor amax and (mx_col) the MX column-wise
    copy of h, also with e5m2 codes and the OCP floor exponent (groups of 128
    and 384 rows, an empty group, pair tiles reaching past a group)."""
    col = scaling.startswith("mx_col")
    hfmt, hmode = ("e5m2", "floor") if scaling.endswith("floor") else ("e4m3", "rceil")
    scaling = "mx" if col else scaling
    rng = np.random.default_rng(31)
    dev = torch.device(DEV)
    offs = np.array([0, 128, 128, 512, 640], dtype=np.int32)
    E, F, K = 4, 384, 256
    Rp = int(offs[-1])
    R_cap = Rp + 128
    offd = torch.from_numpy(offs).to(dev)
    if scaling == "mx":
        ac, asc = _mx_operand(rng, R_cap, K, sc_lo=118, sc_hi=124)
        wc, wsc = _mx_operand(rng, E * 2 * F, K, sc_lo=118, sc_hi=124)
        A = _op(mgq, ac, tile_mx_scales(asc), K, mgq.E4M3, dev)
        W1 = _op(mgq, wc, tile_mx_scales(wsc), K, mgq.E4M3, dev)
        sc = mgq.MX32_E8M0
    elif scaling == "nvfp4":
        pack = lambda q: ((q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)).astype(np.uint8)
        sca = rng.integers(0x20, 0x50, size=(R_cap, K // 16)).astype(np.uint8)
        scw = rng.integers(0x20, 0x50, size=(E * 2 * F, K // 16)).astype(np.uint8)
        A = _op(mgq, pack(rng.integers(0, 16, size=(R_cap, K)).astype(np.uint8)), tile_mx_scales(sca), K,
                mgq.E2M1, dev)
        W1 = _op(mgq, pack(rng.integers(0, 16, size=(E * 2 * F, K)).astype(np.uint8)), tile_mx_scales(scw), K,
                 mgq.E2M1, dev)
        ga = _to_dev(np.array([2.5], dtype=np.float32), dev)
        gw = _to_dev(np.exp2(rng.uniform(-2, 2, size=E)).astype(np.float32), dev)
        _KEEP.append((ga, gw))
        A.global_scale, W1.global_scale = ga.data_ptr(), gw.data_ptr()
        sc = mgq.NV16_UE4M3
    else:
        f4 = OF.E4M3
        ac = (rng.choice(f4.pos_codes[:-1], size=(R_cap, K)) | (rng.integers(0, 2, (R_cap, K)) * 0x80)).astype(np.uint8)
        wc = (rng.choice(f4.pos_codes[:-1], size=(E * 2 * F, K)) |
              (rng.integers(0, 2, (E * 2 * F, K)) * 0x80)).astype(np.uint8)
        A = _op(mgq, ac, np.array([64.0], dtype=np.float32), K, mgq.E4M3, dev)
        W1 = _op(mgq, wc, np.array([40.0, 16.0, 8.0, 30.0], dtype=np.float32), K, mgq.E4M3, dev)
        sc = mgq.TENSOR_F32

    def outputs():
        nv = sc == mgq.NV16_UE4M3
        o = dict(gu=torch.full((R_cap, 2 * F), 3.0, dtype=torch.bfloat16, device=dev),
                 h=torch.full((R_cap, F), 3.0, dtype=torch.bfloat16, device=dev),
                 hq=torch.full((R_cap, F // 2 if nv else F), 0xAB, dtype=torch.uint8, device=dev),
                 hs=torch.full(((mgq.nv_scale_bytes if nv else mgq.mx_scale_bytes)(R_cap, F),), 0xCD,
                               dtype=torch.uint8, device=dev),
                 ts=torch.tensor([2.5], device=dev), am=torch.full((1,), 7.0, device=dev))
        o["c"] = torch.full((F, R_cap), 0xAB, dtype=torch.uint8, device=dev)
        o["cs"] = torch.full((mgq.mx_scale_bytes(F, R_cap),), 0xCD, dtype=torch.uint8, device=dev)
        if sc == mgq.MX32_E8M0:
            o["q"] = mgq.qdesc(mgq.E5M2 if hfmt == "e5m2" else mgq.E4M3, sc, o["hq"], o["hs"],
                               *((o["c"], o["cs"]) if col else (None, None)),
                               e8m0_mode=mgq.FLOOR if hmode == "floor" else mgq.RCEIL)
        elif nv:   # s_g is written to ts, the amax (zeroed by the call) to am
            o["q"] = mgq.qdesc(mgq.E2M1, sc, o["hq"], o["hs"], tensor_scale=o["ts"], amax_out=o["am"])
        else:
            o["am"].zero_()
            o["q"] = mgq.qdesc(mgq.E4M3, sc, o["hq"], None, None, None, o["ts"], o["am"])
        return o

    sep, fus = outputs(), outputs()
    mgq.grouped_gemm_fwd(A, W1, sc, offd, E, R_cap, 2 * F, K, sep["gu"])
    mgq.swiglu_quantize(sep["gu"], R_cap, F, offd, E, sep["q"], sep["h"])
    mgq.grouped_gemm_fwd_swiglu(A, W1, sc, offd, E, R_cap, F, K, fus["q"], fus["gu"], fus["h"])
    # without the optional outputs the codes are the same (NVFP4 needs h itself)
    bare = outputs()
    mgq.grouped_gemm_fwd_swiglu(A, W1, sc, offd, E, R_cap, F, K, bare["q"],
                                h=bare["h"] if sc == mgq.NV16_UE4M3 else None)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    for key in ("gu", "h", "hq", "hs", "am", "ts", "c", "cs"):
        assert torch.equal(sep[key], fus[key]), key
    assert torch.equal(sep["hq"], bare["hq"]) and torch.equal(sep["am"], bare["am"])
    assert torch.equal(sep["c"], bare["c"]) and torch.equal(sep["cs"], bare["cs"])
    assert torch.all(bare["gu"] == 3.0)
    assert torch.all(fus["hq"][Rp:] == 0xAB)          # rows past the groups untouched
    # and h against the oracle's SwiGLU of the GEMM output
    gu = bf16_np(sep["gu"])[:Rp]
    hf = bf16_np(fus["h"])[:Rp]
    check_elementwise(OL.swiglu(gu, F), hf, "swiglu")
    if col:   # both copies against the oracle (the columns: 32-row blocks inside the groups)
        c_, s_ = OQ.quantize_mx(hf, hfmt, hmode)
        assert np.array_equal(u8_np(fus["hq"])[:Rp], c_)
        assert np.array_equal(untile_mx_scales(u8_np(fus["hs"]), R_cap, F)[:Rp], s_)
        assert torch.all(fus["c"][:, Rp:] == 0xAB)
        ct, st = OQ.quantize_mx(hf.T, hfmt, hmode)
        assert np.array_equal(u8_np(fus["c"])[:, :Rp], ct)
        assert np.array_equal(untile_mx_scales(u8_np(fus["cs"]), F, R_cap)[:, :Rp // 32], st)


@pytest.mark.parametrize("w_layout", ["mn_major", "k_major", "mx", "mx_col", "mx_col_floor"])
def test_gemm_dgrad_dswiglu_equals_separate_steps(mgq, w_layout):
    """The down-projection dgrad with dSwiGLU + quantisation in its epilogue
    writes the same bytes as grouped_gemm_dgrad followed by dswiglu_quantize
    (per-tensor e5m2 gradients with W2 read MN-major or as its column-wise
    copy; MX e5m2 gradients, rows only or with the column-wise copy; an empty
    group, pair tiles reaching past a group)."""
    mx = w_layout.startswith("mx")
    col = w_layout.startswith("mx_col")
    mode = "floor" if w_layout.endswith("floor") else "rceil"
    rng = np.random.default_rng(37)
    dev = torch.device(DEV)
    offs = np.array([0, 128, 128, 512, 640], dtype=np.int32)
    E, H, F = 4, 256, 512
    Rp = int(offs[-1])
    R_cap = Rp + 128
    offd = torch.from_numpy(offs).to(dev)
    f5, f4 = OF.E5M2, OF.E4M3
    dyc = (rng.choice(f5.pos_codes[:-1], size=(R_cap, H)) | (rng.integers(0, 2, (R_cap, H)) * 0x80)).astype(np.uint8)
    wc = (rng.choice(f4.pos_codes[:-1], size=(E, H, F)) | (rng.integers(0, 2, (E, H, F)) * 0x80)).astype(np.uint8)
    dY = _op(mgq, dyc, np.array([2048.0], dtype=np.float32), H, mgq.E5M2, dev)
    s_w = np.array([40.0, 16.0, 8.0, 30.0], dtype=np.float32)
    if mx:
        dyc, dys = _mx_operand(rng, R_cap, H, fmt="e5m2", sc_lo=110, sc_hi=116)
        dY = _op(mgq, dyc, tile_mx_scales(dys), H, mgq.E5M2, dev)
        wc2, ws2 = _mx_operand(rng, E * F, H, sc_lo=118, sc_hi=124)          # W2col [E, F, H]
        W2 = _op(mgq, wc2, tile_mx_scales(ws2), H, mgq.E4M3, dev)
    elif w_layout == "mn_major":
        W2 = _op(mgq, wc, s_w, F, mgq.E4M3, dev)
        W2.layout = mgq.LAYOUT_MN
    else:
        W2 = _op(mgq, np.ascontiguousarray(wc.transpose(0, 2, 1)), s_w, H, mgq.E4M3, dev)   # [E, F, H]
    gu = (torch.randn(R_cap, 2 * F, device=dev) * 2).to(torch.bfloat16)

    def outputs():
        o = dict(dh=torch.full((R_cap, F), 3.0, dtype=torch.bfloat16, device=dev),
                 dgu=torch.full((R_cap, 2 * F), 3.0, dtype=torch.bfloat16, device=dev),
                 q=torch.full((R_cap, 2 * F), 0xAB, dtype=torch.uint8, device=dev),
                 s=torch.full((mgq.mx_scale_bytes(R_cap, 2 * F),), 0xCD, dtype=torch.uint8, device=dev),
                 c=torch.full((2 * F, R_cap), 0xAB, dtype=torch.uint8, device=dev),
                 cs=torch.full((mgq.mx_scale_bytes(2 * F, R_cap),), 0xCD, dtype=torch.uint8, device=dev),
                 ts=torch.tensor([5000.0], device=dev), am=torch.zeros(1, device=dev))
        if mx:
            o["qd"] = mgq.qdesc(mgq.E5M2, mgq.MX32_E8M0, o["q"], o["s"],
                                *((o["c"], o["cs"]) if col else (None, None)),
                                e8m0_mode=mgq.FLOOR if mode == "floor" else mgq.RCEIL)
        else:
            o["qd"] = mgq.qdesc(mgq.E5M2, mgq.TENSOR_F32, o["q"], None, None, None, o["ts"], o["am"])
        return o

    sep, fus, bare = outputs(), outputs(), outputs()
    sc = mgq.MX32_E8M0 if mx else mgq.TENSOR_F32
    mgq.grouped_gemm_dgrad(dY, W2, sc, offd, E, R_cap, H, F, sep["dh"])
    mgq.dswiglu_quantize(sep["dh"], gu, R_cap, F, offd, E, sep["qd"], sep["dgu"])
    mgq.grouped_gemm_dgrad_dswiglu(dY, W2, sc, offd, E, R_cap, H, F, gu, fus["qd"], fus["dh"], fus["dgu"])
    mgq.grouped_gemm_dgrad_dswiglu(dY, W2, sc, offd, E, R_cap, H, F, gu, bare["qd"])
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    for key in ("dh", "dgu", "q"):
        assert torch.equal(sep[key][:Rp], fus[key][:Rp]), key
    for key in ("am", "s", "c", "cs"):      # (untouched alike outside the groups)
        assert torch.equal(sep[key], fus[key]), key
    for key in ("q", "s", "c", "cs"):
        assert torch.equal(sep[key][:Rp] if key == "q" else sep[key], bare[key][:Rp] if key == "q" else bare[key])
    assert torch.equal(sep["am"], bare["am"])
    assert torch.all(bare["dh"] == 3.0)
    assert torch.all(fus["q"][Rp:] == 0xAB)
    # and dSwiGLU against the oracle
    dgu = bf16_np(fus["dgu"])[:Rp]
    check_elementwise(OL.dswiglu(bf16_np(sep["dh"])[:Rp], bf16_np(gu)[:Rp], F), dgu, "dswiglu")
    if mx:    # the codes against the oracle's MX blocks (columns: 32 rows inside the groups)
        c, s_ = OQ.quantize_mx(dgu, "e5m2", mode)
        assert np.array_equal(u8_np(fus["q"])[:Rp], c)
        assert np.array_equal(untile_mx_scales(u8_np(fus["s"]), R_cap, 2 * F)[:Rp], s_)
        if col:
            ct, st = OQ.quantize_mx(dgu.T, "e5m2", mode)
            assert np.array_equal(u8_np(fus["c"])[:, :Rp], ct)
            assert np.array_equal(untile_mx_scales(u8_np(fus["cs"]), 2 * F, R_cap)[:, :Rp // 32], st)
        else:
            assert torch.all(fus["c"] == 0xAB)


@pytest.mark.parametrize("mode", ["mx", "mx_col", "tensor", "nvfp4"])
def test_route_then_permute_routed_equals_permute(mgq, mode):
    """mgq_moe_route followed by mgq_moe_permute_routed writes what one
    mgq_moe_permute call writes (routing arrays, codes, scales, amax)."""
    rng = np.random.default_rng(61)
    dev = torch.device(DEV)
    T, E, k, H = 1000, 6, 2, 512
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = torch.from_numpy((rng.standard_normal((T, H)) * 3).astype(np.float32)).to(torch.bfloat16).to(dev)
    idxd = torch.from_numpy(idx).to(dev)
    R_cap = mgq.r_cap(T, k, E, 128)
    ws = torch.empty(max(16, mgq.permute_workspace_size(T, k, E)), dtype=torch.uint8, device=dev)

    def bufs():
        nv = mode == "nvfp4"
        b = dict(rim=torch.full((T, k), -7, dtype=torch.int32, device=dev),
                 src=torch.full((R_cap,), -7, dtype=torch.int32, device=dev),
                 off=torch.zeros(E + 1, dtype=torch.int32, device=dev),
                 cnt=torch.zeros(E, dtype=torch.int32, device=dev),
                 q=torch.full((R_cap, H // 2 if nv else H), 0xAB, dtype=torch.uint8, device=dev),
                 s=torch.full(((mgq.nv_scale_bytes if nv else mgq.mx_scale_bytes)(R_cap, H),), 0xCD,
                              dtype=torch.uint8, device=dev),
                 ts=torch.tensor([3.0], device=dev), am=torch.zeros(1, device=dev),
                 c=torch.full((H, R_cap), 0xAB, dtype=torch.uint8, device=dev),
                 cs=torch.full((mgq.mx_scale_bytes(H, R_cap),), 0xCD, dtype=torch.uint8, device=dev))
        if mode == "mx":
            b["qd"] = mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, b["q"], b["s"])
        elif mode == "mx_col":
            b["qd"] = mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, b["q"], b["s"], b["c"], b["cs"])
        elif mode == "nvfp4":
            b["qd"] = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, b["q"], b["s"], tensor_scale=b["ts"], amax_out=b["am"])
        else:
            b["qd"] = mgq.qdesc(mgq.E4M3, mgq.TENSOR_F32, b["q"], None, None, None, b["ts"], b["am"])
        return b

    one, two = bufs(), bufs()
    mgq.moe_permute(x, idxd, E, 128, one["qd"], R_cap, one["rim"], one["src"], one["off"], one["cnt"], ws)
    mgq.moe_route(idxd, E, 128, R_cap, two["rim"], two["src"], two["off"], two["cnt"], ws)
    mgq.moe_permute_routed(x, k, E, two["qd"], R_cap, two["rim"], two["src"], two["off"], two["cnt"])
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    Rp = int(one["off"][-1].item())
    for key in ("rim", "off", "cnt", "q", "s", "am", "ts", "c", "cs"):
        assert torch.equal(one[key], two[key]), key
    assert torch.equal(one["src"][:Rp], two["src"][:Rp])
    rim, src, off, cnt = OR.permute_indices(idx, E, 128)
    assert np.array_equal(two["rim"].cpu().numpy(), rim)
    assert np.array_equal(two["src"].cpu().numpy()[:Rp], src)


@pytest.mark.parametrize("mode", ["mx_col", "nvfp4", "nvfp4_col"])
def test_empty_batch_block_scaled_paths(mgq, mode):
    """T = 0 through the block-scaled permute (routed), unpermute backward and
    (NVFP4) SwiGLU / dSwiGLU quantisers: no error, no code written, the NVFP4
    amax set to 0."""
    dev = torch.device(DEV)
    E, k, H, F = 4, 2, 256, 256
    T = 0
    nv = mode.startswith("nvfp4")
    align = 256 if nv else 128
    R_cap = max(256, mgq.r_cap(T, k, E, align))
    idx = torch.empty(0, k, dtype=torch.int32, device=dev)
    rim = torch.empty(0, k, dtype=torch.int32, device=dev)
    src = torch.full((R_cap,), -9, dtype=torch.int32, device=dev)
    off = torch.full((E + 1,), -9, dtype=torch.int32, device=dev)
    cnt = torch.full((E,), -9, dtype=torch.int32, device=dev)
    ws = torch.empty(max(16, mgq.permute_workspace_size(T, k, E)), dtype=torch.uint8, device=dev)
    mgq.moe_route(idx, E, align, R_cap, rim, src, off, cnt, ws)

    def qd(C):
        cb = C // 2 if nv else C
        codes = torch.full((R_cap, cb), 0xAB, dtype=torch.uint8, device=dev)
        sc = torch.full(((mgq.nv_scale_bytes if nv else mgq.mx_scale_bytes)(R_cap, C),), 0xCD, dtype=torch.uint8,
                        device=dev)
        col = csc = None
        if mode.endswith("col"):
            col = torch.full((C, R_cap // 2 if nv else R_cap), 0xAB, dtype=torch.uint8, device=dev)
            csc = torch.full(((mgq.nv_scale_bytes if nv else mgq.mx_scale_bytes)(C, R_cap),), 0xCD,
                             dtype=torch.uint8, device=dev)
        if nv:
            am, sg = torch.full((1,), 7.0, device=dev), torch.full((1,), 9.0, device=dev)
            q = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, codes, sc, col, csc, tensor_scale=sg, amax_out=am)
        else:
            am = sg = None
            q = mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, codes, sc, col, csc)
        return q, [codes, sc] + ([col, csc] if col is not None else []), am

    x = torch.empty(0, H, dtype=torch.bfloat16, device=dev)
    qx, bx, amx = qd(H)
    mgq.moe_permute_routed(x, k, E, qx, R_cap, rim, src, off, cnt)
    qy, by, amy = qd(H)
    dprobs = torch.empty(0, k, device=dev)
    mgq.moe_unpermute_bwd(torch.empty(0, H, dtype=torch.bfloat16, device=dev),
                          torch.zeros(R_cap, H, dtype=torch.bfloat16, device=dev), rim, src,
                          torch.empty(0, k, device=dev), R_cap, off, E, qy, dprobs)
    bufs, ams = bx + by, [amx, amy]
    if nv:
        gu = torch.zeros(R_cap, 2 * F, dtype=torch.bfloat16, device=dev)
        h = torch.full((R_cap, F), 3.0, dtype=torch.bfloat16, device=dev)
        qh, bh, amh = qd(F)
        mgq.swiglu_quantize(gu, R_cap, F, off, E, qh, h)
        dgu = torch.full((R_cap, 2 * F), 3.0, dtype=torch.bfloat16, device=dev)
        qg, bg, amg = qd(2 * F)
        mgq.dswiglu_quantize(torch.zeros(R_cap, F, dtype=torch.bfloat16, device=dev), gu, R_cap, F, off, E, qg, dgu)
        bufs, ams = bufs + bh + bg, ams + [amh, amg]
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    assert torch.all(off == 0) and torch.all(cnt == 0)
    for b in bufs:
        assert torch.all((b == 0xAB) | (b == 0xCD)).item()      # nothing written
    if nv:
        assert all(float(a.item()) == 0.0 for a in ams)
        assert torch.all(h == 3.0).item() and torch.all(dgu == 3.0).item()


def test_tile_pass_beyond_the_grid_row_limit(mgq):
    """An MX row-wise + column-wise pass over 66560 row tiles (more than a
    grid dimension holds): the CTAs stride over the row tiles; the first, a
    middle, the 65536th and the last tiles equal the oracle's."""
    dev = torch.device(DEV)
    K = 128
    M = 66560 * 128
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    x = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    codes = torch.empty(M, K, dtype=torch.uint8, device=dev)
    sc = torch.empty(mgq.mx_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    col = torch.empty(K, M, dtype=torch.uint8, device=dev)
    csc = torch.empty(mgq.mx_scale_bytes(K, M), dtype=torch.uint8, device=dev)
    mgq.block_quantize(x, mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, codes, sc, col, csc))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    s_nat = untile_mx_scales(u8_np(sc), M, K)
    for t in (0, 12345, 65535, 66559):
        r0 = t * 128
        xt = bf16_np(x[r0:r0 + 128])
        c, s_ = OQ.quantize_mx(xt)
        assert np.array_equal(u8_np(codes[r0:r0 + 128]), c), t
        assert np.array_equal(s_nat[r0:r0 + 128], s_), t
        cc, cs = OQ.quantize_mx(xt.T)
        assert np.array_equal(u8_np(col[:, r0:r0 + 128]), cc), t
    # the column-wise scales of the last tile (natural [K, M/32] view, computed
    # from the tiled layout directly for its 4 blocks)
    kb4 = M // 128
    ks = np.arange(K)[:, None]
    bs = (66559 * 128) // 32 + np.arange(4)[None, :]
    offs = ((ks // 128) * kb4 + bs // 4) * 512 + (ks % 32) * 16 + ((ks // 32) % 4) * 4 + bs % 4
    got = u8_np(csc)[offs]
    _, cs_last = OQ.quantize_mx(bf16_np(x[66559 * 128:]).T)
    assert np.array_equal(got, cs_last)


@pytest.mark.parametrize("mode", ["mx", "nvfp4", "tensor"])
def test_grouped_quantize_ragged_groups(mgq, mode):
    """Row-wise and column-wise codes of a bf16 matrix over ragged groups (an
    empty group, a 32-row group, unpadded rows past the last group): equal to
    the oracle's, column blocks inside each group; a group start off the block
    boundary is reported."""
    rng = np.random.default_rng(81)
    dev = torch.device(DEV)
    C, R_cap = 384, 768
    sizes = [160, 0, 32, 320, 64]                 # multiples of 32 (MX) and 16 (NVFP4)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    E, Rp = len(sizes), int(off[-1])
    x = _bf16(rng, (R_cap, C), 2.0)
    x[Rp:] = 1e4                                  # rows past the groups: never read
    xf = bf16_np(x)[:Rp]
    nv = mode == "nvfp4"
    cb = C // 2 if nv else C
    codes = torch.full((R_cap, cb), 0xAB, dtype=torch.uint8, device=dev)
    col = torch.full((C, R_cap // 2 if nv else R_cap), 0xAB, dtype=torch.uint8, device=dev)
    if nv:
        sc = torch.full((mgq.nv_scale_bytes(R_cap, C),), 0xCD, dtype=torch.uint8, device=dev)
        csc = torch.full((mgq.nv_scale_bytes(C, R_cap),), 0xCD, dtype=torch.uint8, device=dev)
        am, sg = torch.full((1,), 7.0, device=dev), torch.zeros(1, device=dev)
        q = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, codes, sc, col, csc, tensor_scale=sg, amax_out=am)
    elif mode == "mx":
        sc = torch.full((mgq.mx_scale_bytes(R_cap, C),), 0xCD, dtype=torch.uint8, device=dev)
        csc = torch.full((mgq.mx_scale_bytes(C, R_cap),), 0xCD, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, codes, sc, col, csc)
    else:
        s = torch.tensor([3.0], device=dev)
        am = torch.zeros(1, device=dev)
        q = mgq.qdesc(mgq.E4M3, mgq.TENSOR_F32, codes, None, col, None, s, am)
    offd = torch.from_numpy(off).to(dev)
    mgq.grouped_quantize(x.to(dev), offd, E, q)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    if nv:
        amv = float(np.max(np.abs(xf)))
        s_g = OQ.nvfp4_global_scale(amv)
        assert float(am.item()) == amv and float(sg.item()) == float(s_g)
        c, s_ = OQ.quantize_nvfp4(xf, s_g)
        assert np.array_equal(u8_np(codes)[:Rp], c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), R_cap, C, 16)[:Rp], s_)
        for e in range(E):
            lo, hi = int(off[e]), int(off[e + 1])
            if hi == lo:
                continue
            cc, cs = OQ.quantize_nvfp4(xf[lo:hi].T, s_g)
            assert np.array_equal(u8_np(col)[:, lo // 2:hi // 2], cc), e
            assert np.array_equal(untile_mx_scales(u8_np(csc), C, R_cap, 16)[:, lo // 16:hi // 16], cs), e
    elif mode == "mx":
        c, s_ = OQ.quantize_mx(xf)
        assert np.array_equal(u8_np(codes)[:Rp], c)
        assert np.array_equal(untile_mx_scales(u8_np(sc), R_cap, C)[:Rp], s_)
        for e in range(E):
            lo, hi = int(off[e]), int(off[e + 1])
            if hi == lo:
                continue
            cc, cs = OQ.quantize_mx(xf[lo:hi].T)
            assert np.array_equal(u8_np(col)[:, lo:hi], cc), e
            assert np.array_equal(untile_mx_scales(u8_np(csc), C, R_cap)[:, lo // 32:hi // 32], cs), e
    else:
        c, amv = OQ.quantize_tensor(xf, np.float32(3.0))
        assert np.array_equal(u8_np(codes)[:Rp], c)
        assert np.array_equal(u8_np(col)[:, :Rp], c.T)
        assert float(am.item()) == amv
    assert torch.all(codes[Rp:] == 0xAB).item()     # rows past the groups untouched
    if mode != "tensor":
        # a group start off the column-block boundary is reported
        bad = torch.from_numpy(np.array([0, 48, Rp], dtype=np.int32)).to(dev)
        mgq.grouped_quantize(x.to(dev), bad, 2, q)
        torch.cuda.synchronize()
        assert mgq.get_error() == (mgq.ERR_INVALID_ARG if mode == "mx" else mgq.OK)   # 48: an NVFP4 block start


def test_empty_batch_through_every_call(mgq):
    """T = 0 tokens: routing gives empty groups (offsets all zero), the
    permute writes nothing, the GEMMs compute nothing (wgrad writes zeros for
    the empty groups, or keeps dW with beta = 1), and the combine steps return
    at once; no call reports an error."""
    dev = torch.device(DEV)
    E, k, H, N = 4, 2, 256, 256
    T = 0
    R_cap = mgq.r_cap(T, k, E, 128)
    idx = torch.empty(0, k, dtype=torch.int32, device=dev)
    rim = torch.empty(0, k, dtype=torch.int32, device=dev)
    src = torch.full((R_cap,), -9, dtype=torch.int32, device=dev)
    off = torch.full((E + 1,), -9, dtype=torch.int32, device=dev)
    cnt = torch.full((E,), -9, dtype=torch.int32, device=dev)
    ws = torch.empty(max(16, mgq.permute_workspace_size(T, k, E)), dtype=torch.uint8, device=dev)
    mgq.moe_route(idx, E, 128, R_cap, rim, src, off, cnt, ws)
    x = torch.empty(0, H, dtype=torch.bfloat16, device=dev)
    codes = torch.full((R_cap, H), 0xAB, dtype=torch.uint8, device=dev)
    s = torch.tensor([1.0], device=dev)
    q = mgq.qdesc(mgq.E4M3, mgq.TENSOR_F32, codes, None, None, None, s, None)
    mgq.moe_permute_routed(x, k, E, q, R_cap, rim, src, off, cnt)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    assert torch.all(off == 0) and torch.all(cnt == 0)
    assert torch.all(codes == 0xAB)
    # GEMMs over all-empty groups
    w = torch.zeros(E * N, H, dtype=torch.uint8, device=dev)
    A = mgq.operand(codes, s, H, mgq.E4M3)
    sw = torch.ones(E, device=dev)              # (tensors kept alive: operands hold addresses)
    W = mgq.operand(w, sw, H, mgq.E4M3)
    Y = torch.full((R_cap, N), 3.0, dtype=torch.bfloat16, device=dev)
    mgq.grouped_gemm_fwd(A, W, mgq.TENSOR_F32, off, E, R_cap, N, H, Y)
    dW = torch.full((E, N, H), 5.0, dtype=torch.float32, device=dev)
    dyc_codes = torch.zeros(N, R_cap, dtype=torch.uint8, device=dev)
    ac_codes = torch.zeros(H, R_cap, dtype=torch.uint8, device=dev)
    dYc = mgq.operand(dyc_codes, s, R_cap, mgq.E5M2)
    Ac = mgq.operand(ac_codes, s, R_cap, mgq.E4M3)
    mgq.grouped_gemm_wgrad(dYc, Ac, mgq.TENSOR_F32, off, E, R_cap, N, H, dW, 0.0)
    dW1 = torch.full((E, N, H), 5.0, dtype=torch.float32, device=dev)
    mgq.grouped_gemm_wgrad(dYc, Ac, mgq.TENSOR_F32, off, E, R_cap, N, H, dW1, 1.0)
    out = torch.empty(0, H, dtype=torch.bfloat16, device=dev)
    mgq.moe_unpermute(Y, rim, torch.empty(0, k, device=dev), out)
    mgq.moe_permute_bwd(Y, rim, out)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    assert torch.all(Y == 3.0)                 # no rows to compute
    assert torch.all(dW == 0.0)                # empty groups: zeros
    assert torch.all(dW1 == 5.0)               # beta = 1: untouched

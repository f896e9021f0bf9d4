"""End-to-end parity of the expert layer through the C ABI: every step of a
forward (MXFP8) and of a training step (hybrid e4m3/e5m2, delayed per-tensor
scaling) against the oracle on the same inputs, plus the SQNR of the
quantised GEMMs against unquantised bf16 operands (pytorch/ao PR #2275,
testing)."""
import numpy as np
import pytest
import torch

from oracle import formats as OF
from oracle import gemm as OG
from oracle import layer as OL
from oracle import quant as OQ
from oracle import routing as OR
from tests.layer_check import (GEMM_TOL_BF16, GEMM_TOL_F32, bf16_np, check_elementwise, rel_fro,
                               run_fwd_and_check, u8_np)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_tiny_forward_mxfp8():
    from fp8_grouped_gemm_gb300.workloads import WORKLOADS
    res = run_fwd_and_check(WORKLOADS["tiny"], DEV)
    assert res["gemm1_sqnr_vs_bf16"] >= 28.0, res


def test_mixtral_shaped_forward_scaled_down():
    """Mixtral-like proportions (outlier channels, top-2 of 8) at a size the
    oracle checks in full: several 128x256 tiles per expert, ragged groups."""
    from fp8_grouped_gemm_gb300.workloads import WORKLOADS
    w = WORKLOADS["mixtral_fwd"].scaled(T=1500, H=1024, F=1792)
    res = run_fwd_and_check(w, DEV)
    assert res["gemm1_sqnr_vs_bf16"] >= 28.0, res


def test_scout_forward_blockwise_scaled_down():
    """Llama4-Scout proportions (Zipf(1.2) expert loads, two empty experts,
    top-1) with 1x128 / 128x128 blockwise FP8 at a size checked in full."""
    from fp8_grouped_gemm_gb300.workloads import WORKLOADS
    w = WORKLOADS["scout_fwd"].scaled(T=2048, H=768, F=1024)
    res = run_fwd_and_check(w, DEV, recipe="blockwise")
    assert res["gemm1_sqnr_vs_bf16"] >= 28.0, res


@pytest.mark.parametrize("recipe", ["mxfp8", "nvfp4"])
def test_skewed_routing_forward_scaled_down(recipe):
    """The degenerate load: top-1 Zipf(3) routing over two of eight experts
    (about 89% of the tokens in one group, six groups empty), checked in full."""
    from fp8_grouped_gemm_gb300.workloads import WORKLOADS
    w = WORKLOADS["mixtral_fwd"].scaled(T=1500, H=512, F=768, k=1, routing="zipf", zipf_s=3.0, n_empty=6,
                                        recipe=recipe)
    res = run_fwd_and_check(w, DEV, recipe=recipe)
    assert res["gemm1_sqnr_vs_bf16"] >= (28.0 if recipe == "mxfp8" else 15.0), res


@pytest.mark.parametrize("image_min_k", [1 << 30, 0], ids=["scales", "scale_image"])
def test_finegrained_forward_nvfp4_scaled_down(image_min_k):
    """Fine-grained MoE proportions (uniform top-8 routing) in NVFP4 (e2m1,
    16-element ue4m3 scales, float32 global scales) at a size checked in full;
    SQNR bar 15 dB against bf16. Both with the weights' scales read as they
    are and through their GEMM scale images."""
    from fp8_grouped_gemm_gb300.workloads import WORKLOADS
    w = WORKLOADS["finegrained_fwd"].scaled(T=1024, E=32, H=512, F=768)
    kw = {"nv_image_min_k": image_min_k}
    res = run_fwd_and_check(w, DEV, recipe="nvfp4", **kw)
    assert res["gemm1_sqnr_vs_bf16"] >= 15.0, res


def _tensor_deq(codes, s, fmt="e4m3"):
    return OQ.dequantize_tensor(codes, np.float32(s), fmt)


@pytest.mark.parametrize("col_copies,skewed", [(False, False), (True, False), (False, True)],
                         ids=["mn_major", "col_copies", "skewed"])
def test_delayed_training_steps(col_copies, skewed):
    """Three delayed-scaling training steps: every code bit-exact, GEMMs within
    tolerance, amaxes and next scales exact. By default the backward GEMMs read
    the row-wise codes MN-major; col_copies=True writes and uses the explicit
    column-wise copies (which must be the transposed row-wise codes). skewed:
    top-1 Zipf(3) routing over two of the four experts (two groups empty, one
    holding most of the tokens)."""
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    w = W.WORKLOADS["mixtral_fwdbwd"].scaled(T=700, H=512, F=768, E=4)
    if skewed:
        w = w.scaled(k=1, routing="zipf", zipf_s=3.0, n_empty=2)
    E, k, T, H, F = w.E, w.k, w.T, w.H, w.F
    x = W.make_activations(w)
    w1, w2 = W.make_weights(w)
    idx, probs = W.make_routing(w)
    dout = W.make_dout(w)
    lay = L.ExpertLayer(w, DEV, recipe="delayed", keep_bf16=True, history=16, col_copies=col_copies)
    xd, w1d, w2d, dd = x.to(DEV), w1.to(DEV), w2.to(DEV), dout.to(DEV)
    idxd, pd = torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV)
    xf, w1f, w2f, df = bf16_np(x), bf16_np(w1), bf16_np(w2), bf16_np(dout)
    rim, src, off, cnt = OR.permute_indices(idx, E, L.ALIGN)
    Rp = int(off[-1])
    fwd_ds = [OL.DelayedScaling("e4m3", 16) for _ in range(2 + 2 * E)]
    bwd_ds = [OL.DelayedScaling("e5m2", 16) for _ in range(2)]
    for step in range(3):
        fs = lay.fwd_scale.cpu().numpy().copy()
        bs = lay.bwd_scale.cpu().numpy().copy()
        assert np.array_equal(fs, np.array([d.scale for d in fwd_ds], dtype=np.float32))
        assert np.array_equal(bs, np.array([d.scale for d in bwd_ds], dtype=np.float32))
        lay.quantize_weights(w1d, w2d)
        lay.forward(xd, idxd, pd)
        lay.backward(dd, pd)
        torch.cuda.synchronize()
        assert mgq.get_error() == mgq.OK
        # --- forward -----------------------------------------------------
        cx, am_x = OQ.quantize_tensor(xf, fs[0])
        want = OR.permute_rows(cx, rim, Rp)
        assert np.array_equal(u8_np(lay.xq)[:Rp], want)
        if col_copies:
            assert np.array_equal(u8_np(lay.xcol)[:, :Rp], want.T)
        else:
            assert lay.xcol is None and lay.w1col is None and lay.dy1col is None
        w1c = [OQ.quantize_tensor(w1f[e], fs[2 + e]) for e in range(E)]
        w2c = [OQ.quantize_tensor(w2f[e], fs[2 + E + e]) for e in range(E)]
        for e in range(E):
            assert np.array_equal(u8_np(lay.w1q)[e], w1c[e][0])
            assert np.array_equal(u8_np(lay.w2q)[e], w2c[e][0])
            if col_copies:
                assert np.array_equal(u8_np(lay.w1col)[e], w1c[e][0].T)
                assert np.array_equal(u8_np(lay.w2col)[e], w2c[e][0].T)
        xdq = _tensor_deq(want, fs[0])
        w1dq = np.stack([_tensor_deq(w1c[e][0], fs[2 + e]) for e in range(E)])
        w2dq = np.stack([_tensor_deq(w2c[e][0], fs[2 + E + e]) for e in range(E)])
        gu = bf16_np(lay.gu)[:Rp]
        assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_fwd(xdq, w1dq, off)), gu) <= GEMM_TOL_BF16
        hg = bf16_np(lay.h_bf16)[:Rp]
        check_elementwise(OL.swiglu(gu, F), hg, "swiglu")
        ch, am_h = OQ.quantize_tensor(hg, fs[1])
        assert np.array_equal(u8_np(lay.hq)[:Rp], ch)
        if col_copies:
            assert np.array_equal(u8_np(lay.hcol)[:, :Rp], ch.T)
        hdq = _tensor_deq(ch, fs[1])
        y = bf16_np(lay.y)[:Rp]
        assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_fwd(hdq, w2dq, off)), y) <= GEMM_TOL_BF16
        check_elementwise(OR.unpermute(y, rim, probs), bf16_np(lay.out), "unpermute")
        # --- backward ----------------------------------------------------
        dy32, dp = OR.unpermute_bwd(df, y, rim, probs, Rp)
        c2, am_dy2 = OQ.quantize_tensor(dy32.astype(np.float64), bs[0], "e5m2")
        assert np.array_equal(u8_np(lay.dy2q)[:Rp], c2)
        if col_copies:
            assert np.array_equal(u8_np(lay.dy2col)[:, :Rp], c2.T)
        assert rel_fro(dp, lay.dprobs.cpu().numpy()) <= 1e-5
        dy2dq = _tensor_deq(c2, bs[0], "e5m2")
        dh = bf16_np(lay.dh)[:Rp]
        assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_dgrad(dy2dq, w2dq, off)), dh) <= GEMM_TOL_BF16
        assert rel_fro(OG.grouped_gemm_wgrad(dy2dq, hdq, off, E), lay.dw2.cpu().numpy()) <= GEMM_TOL_F32
        dgu = bf16_np(lay.dgu_bf16)[:Rp]
        check_elementwise(OL.dswiglu(dh, gu, F), dgu, "dswiglu")
        c1, am_dy1 = OQ.quantize_tensor(dgu, bs[1], "e5m2")
        assert np.array_equal(u8_np(lay.dy1q)[:Rp], c1)
        if col_copies:
            assert np.array_equal(u8_np(lay.dy1col)[:, :Rp], c1.T)
        dy1dq = _tensor_deq(c1, bs[1], "e5m2")
        dxp = bf16_np(lay.dxp)[:Rp]
        assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_dgrad(dy1dq, w1dq, off)), dxp) <= GEMM_TOL_BF16
        assert rel_fro(OG.grouped_gemm_wgrad(dy1dq, xdq, off, E), lay.dw1.cpu().numpy()) <= GEMM_TOL_F32
        check_elementwise(OR.permute_bwd(dxp, rim), bf16_np(lay.dx), "permute_bwd")
        # --- amaxes and the next step's scales ----------------------------
        amaxes = [am_x, am_h] + [w1c[e][1] for e in range(E)] + [w2c[e][1] for e in range(E)]
        assert np.array_equal(lay.fwd_amax.cpu().numpy(), np.array(amaxes, dtype=np.float32))
        assert np.array_equal(lay.bwd_amax.cpu().numpy(), np.array([am_dy2, am_dy1], dtype=np.float32))
        if step >= 1:
            # after one step of history the e4m3 GEMMs keep the SQNR bar
            ref = OG.grouped_gemm_fwd(OR.permute_rows(xf, rim, Rp), w1f, off)
            assert OG.sqnr_db(ref, gu) >= 28.0
        lay.update_scaling()
        for d, a in zip(fwd_ds, amaxes):
            d.update(a)
        for d, a in zip(bwd_ds, [am_dy2, am_dy1]):
            d.update(a)


def test_mxfp8_training_step_scaled_down():
    """MXFP8 in both passes (e4m3 forward, e5m2 gradients, E8M0 per 32): the
    column-wise copies requantise with 32x1 blocks along each expert's tokens
    (and along N for the weights) instead of transposing the row codes."""
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    from tests.layer_check import untile_mx_scales
    w = W.WORKLOADS["mixtral_fwdbwd_mx"].scaled(T=700, H=512, F=768, E=4)
    E, k, T, H, F = w.E, w.k, w.T, w.H, w.F
    x = W.make_activations(w)
    w1, w2 = W.make_weights(w)
    idx, probs = W.make_routing(w)
    dout = W.make_dout(w)
    lay = L.ExpertLayer(w, DEV, keep_bf16=True)
    assert lay.train and not lay.delayed
    lay.quantize_weights(w1.to(DEV), w2.to(DEV))
    lay.forward(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV))
    lay.backward(dout.to(DEV), torch.from_numpy(probs).to(DEV))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    R = lay.R_cap
    rim, src, off, cnt = OR.permute_indices(idx, E, L.ALIGN)
    Rp = int(off[-1])
    sc = lambda t, rows, ld: untile_mx_scales(u8_np(t), rows, ld)

    def row_col(m, fmt, rq, rs, cq, cs):
        """m [Rp, C]: check the row-wise and column-wise MX copies; returns both dequantised."""
        c, s = OQ.quantize_mx(m, fmt)
        assert np.array_equal(u8_np(rq)[:Rp], c)
        assert np.array_equal(sc(rs, R, m.shape[1])[:Rp], s)
        ct, st = OQ.quantize_mx(m.T, fmt)
        assert np.array_equal(u8_np(cq)[:, :Rp], ct)
        assert np.array_equal(sc(cs, m.shape[1], R)[:, :Rp // 32], st)
        return OQ.dequantize_mx(c, s, fmt), OQ.dequantize_mx(ct, st, fmt).T

    xp = OR.permute_rows(bf16_np(x), rim, Rp)
    x_r, x_c = row_col(xp, "e4m3", lay.xq, lay.xs, lay.xcol, lay.xcs)
    w1f, w2f = bf16_np(w1), bf16_np(w2)
    w1_r, w1_c, w2_r, w2_c = [], [], [], []
    w1cs = sc(lay.w1cs, E * H, 2 * F).reshape(E, H, 2 * F // 32)
    w2cs = sc(lay.w2cs, E * F, H).reshape(E, F, H // 32)
    for e in range(E):
        ct, st = OQ.quantize_mx(w1f[e].T)
        assert np.array_equal(u8_np(lay.w1col)[e], ct) and np.array_equal(w1cs[e], st)
        w1_c.append(OQ.dequantize_mx(ct, st).T)
        ct, st = OQ.quantize_mx(w2f[e].T)
        assert np.array_equal(u8_np(lay.w2col)[e], ct) and np.array_equal(w2cs[e], st)
        w2_c.append(OQ.dequantize_mx(ct, st).T)
    w1_c, w2_c = np.stack(w1_c), np.stack(w2_c)
    w1_r = OQ.dequantize_mx(*OQ.quantize_mx(w1f.reshape(E * 2 * F, H))).reshape(E, 2 * F, H)
    w2_r = OQ.dequantize_mx(*OQ.quantize_mx(w2f.reshape(E * H, F))).reshape(E, H, F)
    gu = bf16_np(lay.gu)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_fwd(x_r, w1_r, off)), gu) <= GEMM_TOL_BF16
    hg = bf16_np(lay.h_bf16)[:Rp]
    check_elementwise(OL.swiglu(gu, F), hg, "swiglu")
    h_r, h_c = row_col(hg, "e4m3", lay.hq, lay.hs, lay.hcol, lay.hcs)
    y = bf16_np(lay.y)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_fwd(h_r, w2_r, off)), y) <= GEMM_TOL_BF16
    # backward
    dy32, dp = OR.unpermute_bwd(bf16_np(dout), y, rim, probs, Rp)
    assert rel_fro(dp, lay.dprobs.cpu().numpy()) <= 1e-5
    dy2_r, dy2_c = row_col(dy32.astype(np.float64), "e5m2", lay.dy2q, lay.dy2s, lay.dy2col, lay.dy2cs)
    dh = bf16_np(lay.dh)[:Rp]
    dh_q = OG.grouped_gemm_dgrad(dy2_r, w2_c, off)
    assert rel_fro(OF.round_to_bf16(dh_q), dh) <= GEMM_TOL_BF16
    dw2_q = OG.grouped_gemm_wgrad(dy2_c, h_c, off, E)
    assert rel_fro(dw2_q, lay.dw2.cpu().numpy()) <= GEMM_TOL_F32
    # GEMMs with an e5m2 operand against the unquantised operands: at least
    # 23 dB, and within 0.5 dB of the oracle's own quantised GEMM
    for ref, q_oracle, got in [(OG.grouped_gemm_dgrad(dy32.astype(np.float64), w2f, off), dh_q, dh),
                               (OG.grouped_gemm_wgrad(dy32.astype(np.float64), hg, off, E), dw2_q,
                                lay.dw2.cpu().numpy().astype(np.float64))]:
        s_gpu, s_orc = OG.sqnr_db(ref, got), OG.sqnr_db(ref, q_oracle)
        assert s_gpu >= 23.0 and abs(s_gpu - s_orc) <= 0.5, (s_gpu, s_orc)
    dgu = bf16_np(lay.dgu_bf16)[:Rp]
    check_elementwise(OL.dswiglu(dh, gu, F), dgu, "dswiglu")
    dy1_r, dy1_c = row_col(dgu, "e5m2", lay.dy1q, lay.dy1s, lay.dy1col, lay.dy1cs)
    dxp = bf16_np(lay.dxp)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_dgrad(dy1_r, w1_c, off)), dxp) <= GEMM_TOL_BF16
    assert rel_fro(OG.grouped_gemm_wgrad(dy1_c, x_c, off, E), lay.dw1.cpu().numpy()) <= GEMM_TOL_F32
    check_elementwise(OR.permute_bwd(dxp, rim), bf16_np(lay.dx), "permute_bwd")
    # quantised-vs-bf16 SQNR of the e4m3 forward GEMM
    assert OG.sqnr_db(OG.grouped_gemm_fwd(xp, w1f, off), gu) >= 28.0


@pytest.mark.parametrize("image_min_k", [1 << 30, 0], ids=["scales", "scale_image"])
def test_nvfp4_training_step_scaled_down(image_min_k):
    """NVFP4 in both passes: activations and gradients e2m1 with 16-element
    ue4m3 scales and one s_g per tensor (row-wise for fwd/dgrad, 16x1 blocks
    along each expert's tokens for wgrad), weights with 16x16 blocks (one pass,
    both copies), groups padded to 256 rows for the NVFP4 wgrad. Both with the
    second operands' scales read as they are and through their scale images."""
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    from tests.layer_check import untile_mx_scales
    w = W.WORKLOADS["mixtral_fwdbwd_nvfp4"].scaled(T=700, H=512, F=768, E=4)
    E, k, T, H, F = w.E, w.k, w.T, w.H, w.F
    x = W.make_activations(w)
    w1, w2 = W.make_weights(w)
    idx, probs = W.make_routing(w)
    dout = W.make_dout(w)
    kw = {"nv_image_min_k": image_min_k}
    lay = L.ExpertLayer(w, DEV, keep_bf16=True, **kw)
    assert lay.train and lay.nv and lay.align == 256 and lay.fused_swiglu
    assert (lay.xcimg is not None) == (image_min_k == 0)
    lay.quantize_weights(w1.to(DEV), w2.to(DEV))
    lay.forward(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV))
    lay.backward(dout.to(DEV), torch.from_numpy(probs).to(DEV))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    R = lay.R_cap
    rim, src, off, cnt = OR.permute_indices(idx, E, lay.align)
    Rp = int(off[-1])
    amax, sg = lay.nv_amax.cpu().numpy(), lay.nv_sg.cpu().numpy()
    sc = lambda t, rows, ld: untile_mx_scales(u8_np(t), rows, ld, 16)

    def row_col(m, i, rq, rs, cq, cs):
        """m [Rp, C] with its own s_g (slot i): both NVFP4 copies; returns them dequantised [Rp, C]."""
        am = float(np.max(np.abs(m)))
        s_g = OQ.nvfp4_global_scale(am)
        assert amax[i] == np.float32(am) and sg[i] == s_g
        C = m.shape[1]
        c, s = OQ.quantize_nvfp4(m, s_g)
        assert np.array_equal(u8_np(rq)[:Rp], c)
        assert np.array_equal(sc(rs, R, C)[:Rp], s)
        ct, st = OQ.quantize_nvfp4(m.T, s_g)
        assert np.array_equal(u8_np(cq)[:, :Rp // 2], ct)
        assert np.array_equal(sc(cs, C, R)[:, :Rp // 16], st)
        return OQ.dequantize_nvfp4(c, s, s_g, C), OQ.dequantize_nvfp4(ct, st, s_g, Rp).T

    xp = OR.permute_rows(bf16_np(x), rim, Rp)
    x_r, x_c = row_col(xp, 0, lay.xq, lay.xs, lay.xcol, lay.xcs)
    w1f, w2f = bf16_np(w1), bf16_np(w2)

    def weight(wf, q, s, col, cs, base, N, Kd):
        """16x16-block copies of each expert [N, Kd]; returns the dequantised weight [E, N, Kd]."""
        rs_all = sc(s, E * N, Kd).reshape(E, N, Kd // 16)
        cs_all = sc(cs, E * Kd, N).reshape(E, Kd, N // 16)
        out = []
        for e in range(E):
            am = float(np.max(np.abs(wf[e])))
            s_g = OQ.nvfp4_global_scale(am)
            assert amax[base + e] == np.float32(am) and sg[base + e] == s_g
            rc, rs, cc, css = OQ.quantize_nvfp4_2d(wf[e], s_g)
            assert np.array_equal(u8_np(q)[e], rc) and np.array_equal(rs_all[e], rs)
            assert np.array_equal(u8_np(col)[e], cc) and np.array_equal(cs_all[e], css)
            out.append(OQ.dequantize_nvfp4(rc, rs, s_g, Kd))
        return np.stack(out)

    w1_d = weight(w1f, lay.w1q, lay.w1s, lay.w1col, lay.w1cs, 2, 2 * F, H)
    w2_d = weight(w2f, lay.w2q, lay.w2s, lay.w2col, lay.w2cs, 2 + E, H, F)
    gu = bf16_np(lay.gu)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_fwd(x_r, w1_d, off)), gu) <= GEMM_TOL_BF16
    hg = bf16_np(lay.h_bf16)[:Rp]
    check_elementwise(OL.swiglu(gu, F), hg, "swiglu")
    h_r, h_c = row_col(hg, 1, lay.hq, lay.hs, lay.hcol, lay.hcs)
    y = bf16_np(lay.y)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_fwd(h_r, w2_d, off)), y) <= GEMM_TOL_BF16
    # backward
    i2, i1 = 2 + 2 * E, 3 + 2 * E
    dy32, dp = OR.unpermute_bwd(bf16_np(dout), y, rim, probs, Rp)
    assert rel_fro(dp, lay.dprobs.cpu().numpy()) <= 1e-5
    dy2_r, dy2_c = row_col(dy32.astype(np.float64), i2, lay.dy2q, lay.dy2s, lay.dy2col, lay.dy2cs)
    dh = bf16_np(lay.dh)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_dgrad(dy2_r, w2_d, off)), dh) <= GEMM_TOL_BF16
    assert rel_fro(OG.grouped_gemm_wgrad(dy2_c, h_c, off, E), lay.dw2.cpu().numpy()) <= GEMM_TOL_F32
    dgu = bf16_np(lay.dgu_bf16)[:Rp]
    check_elementwise(OL.dswiglu(dh, gu, F), dgu, "dswiglu")
    dy1_r, dy1_c = row_col(dgu, i1, lay.dy1q, lay.dy1s, lay.dy1col, lay.dy1cs)
    dxp = bf16_np(lay.dxp)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_dgrad(dy1_r, w1_d, off)), dxp) <= GEMM_TOL_BF16
    assert rel_fro(OG.grouped_gemm_wgrad(dy1_c, x_c, off, E), lay.dw1.cpu().numpy()) <= GEMM_TOL_F32
    check_elementwise(OR.permute_bwd(dxp, rim), bf16_np(lay.dx), "permute_bwd")
    # quantised-vs-bf16 SQNR of the NVFP4 forward GEMM (the NVFP4 bar)
    assert OG.sqnr_db(OG.grouped_gemm_fwd(xp, w1f, off), gu) >= 15.0


def test_blockwise_training_step_scaled_down():
    """Blockwise FP8 in both passes (TransformerEngine issue #2393: 1x128
    forward blocks, 128x1 backward blocks, 128x128 weight tiles; e4m3
    forward, e5m2 gradients) on the Scout-shaped experts scaled down (Zipf
    loads with two empty experts, top-1): every code and scale_inv of both
    copies of X, h, dY2, dY1 and the weights equal the oracle's, and every
    GEMM is within tolerance of the oracle's GEMM on the same quantised
    operands."""
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    w = W.WORKLOADS["scout_fwdbwd"].scaled(T=900, H=512, F=768, E=6)
    E, k, T, H, F = w.E, w.k, w.T, w.H, w.F
    x = W.make_activations(w)
    w1, w2 = W.make_weights(w)
    idx, probs = W.make_routing(w)
    dout = W.make_dout(w)
    lay = L.ExpertLayer(w, DEV, keep_bf16=True)
    assert lay.train and lay.recipe == "blockwise" and not lay.fused_swiglu
    lay.quantize_weights(w1.to(DEV), w2.to(DEV))
    lay.forward(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV))
    lay.backward(dout.to(DEV), torch.from_numpy(probs).to(DEV))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    rim, src, off, cnt = OR.permute_indices(idx, E, L.ALIGN)
    assert np.sum(cnt == 0) >= 1
    Rp = int(off[-1])
    filler = src < 0

    def row_col(m, fmt, rq, rs, cq, cs, zero_filler):
        """m [Rp, C]: the row-wise (1x128) and column-wise (128x1 inside each
        group) copies; returns both dequantised ([Rp, C])."""
        c, si = OQ.quantize_block_1x128(m, fmt)
        r_deq = OQ.dequantize_block_1x128(c, si, fmt)
        if zero_filler:
            si = si.copy()
            si[filler] = 0.0                 # padding rows: zero codes and zero scales
        assert np.array_equal(u8_np(rq)[:Rp], c)
        assert np.array_equal(rs.cpu().numpy().T[:Rp], si)
        c_deq = np.zeros_like(m)
        for e in range(E):
            lo, hi = int(off[e]), int(off[e + 1])
            if hi == lo:
                continue
            ct, st = OQ.quantize_block_1x128(np.ascontiguousarray(m[lo:hi].T), fmt)
            assert np.array_equal(u8_np(cq)[:, lo:hi], ct), e
            assert np.array_equal(cs.cpu().numpy()[lo // 128:hi // 128].T, st), e
            c_deq[lo:hi] = OQ.dequantize_block_1x128(ct, st, fmt).T
        return r_deq, c_deq

    xp = OR.permute_rows(bf16_np(x), rim, Rp)
    x_r, x_c = row_col(xp, "e4m3", lay.xq, lay.xs, lay.xcol, lay.xcs, True)
    w1f, w2f = bf16_np(w1), bf16_np(w2)
    w1_r, w2_r, w1_c, w2_c = [], [], [], []
    for e in range(E):
        for wf, q, s, qc, sc_, rl, cl in ((w1f, lay.w1q, lay.w1s, lay.w1col, lay.w1cs, w1_r, w1_c),
                                          (w2f, lay.w2q, lay.w2s, lay.w2col, lay.w2cs, w2_r, w2_c)):
            c, si = OQ.quantize_block_128x128(wf[e])
            ct, sit = OQ.quantize_block_128x128(np.ascontiguousarray(wf[e].T))
            assert np.array_equal(u8_np(q[e]), c) and np.array_equal(s[e].cpu().numpy(), si), e
            assert np.array_equal(u8_np(qc[e]), ct) and np.array_equal(sc_[e].cpu().numpy(), sit), e
            rl.append(OQ.dequantize_block_128x128(c, si))
            cl.append(OQ.dequantize_block_128x128(ct, sit))
    w1_r, w2_r, w1_c, w2_c = map(np.stack, (w1_r, w2_r, w1_c, w2_c))
    gu = bf16_np(lay.gu)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_fwd(x_r, w1_r, off)), gu) <= GEMM_TOL_BF16
    hg = bf16_np(lay.h_bf16)[:Rp]
    check_elementwise(OL.swiglu(gu, F), hg, "swiglu")
    h_r, h_c = row_col(hg, "e4m3", lay.hq, lay.hs, lay.hcol, lay.hcs, False)
    y = bf16_np(lay.y)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_fwd(h_r, w2_r, off)), y) <= GEMM_TOL_BF16
    # backward
    dy32, dp = OR.unpermute_bwd(bf16_np(dout), y, rim, probs, Rp)
    assert rel_fro(dp, lay.dprobs.cpu().numpy()) <= 1e-5
    dy2_r, dy2_c = row_col(dy32.astype(np.float64), "e5m2", lay.dy2q, lay.dy2s, lay.dy2col, lay.dy2cs, True)
    dh = bf16_np(lay.dh)[:Rp]
    # dgrad through the column-wise weight copy: dY2 (W2col)^T = dY2 W2
    dh_q = OG.grouped_gemm_fwd(dy2_r, w2_c, off)
    assert rel_fro(OF.round_to_bf16(dh_q), dh) <= GEMM_TOL_BF16
    dw2_q = OG.grouped_gemm_wgrad(dy2_c, h_c, off, E)
    assert rel_fro(dw2_q, lay.dw2.cpu().numpy()) <= GEMM_TOL_F32
    for ref, q_oracle, got in [(OG.grouped_gemm_dgrad(dy32.astype(np.float64), w2f, off), dh_q, dh),
                               (OG.grouped_gemm_wgrad(dy32.astype(np.float64), hg, off, E), dw2_q,
                                lay.dw2.cpu().numpy().astype(np.float64))]:
        s_gpu, s_orc = OG.sqnr_db(ref, got), OG.sqnr_db(ref, q_oracle)
        assert s_gpu >= 23.0 and abs(s_gpu - s_orc) <= 0.5, (s_gpu, s_orc)
    dgu = bf16_np(lay.dgu_bf16)[:Rp]
    check_elementwise(OL.dswiglu(dh, gu, F), dgu, "dswiglu")
    dy1_r, dy1_c = row_col(dgu, "e5m2", lay.dy1q, lay.dy1s, lay.dy1col, lay.dy1cs, False)
    dxp = bf16_np(lay.dxp)[:Rp]
    assert rel_fro(OF.round_to_bf16(OG.grouped_gemm_fwd(dy1_r, w1_c, off)), dxp) <= GEMM_TOL_BF16
    assert rel_fro(OG.grouped_gemm_wgrad(dy1_c, x_c, off, E), lay.dw1.cpu().numpy()) <= GEMM_TOL_F32
    dw = lay.dw1.cpu().numpy()
    for e in np.flatnonzero(cnt == 0):
        assert np.all(dw[e] == 0.0)         # empty experts: zero weight gradients
    check_elementwise(OR.permute_bwd(dxp, rim), bf16_np(lay.dx), "permute_bwd")
    assert OG.sqnr_db(OG.grouped_gemm_fwd(xp, w1f, off), gu) >= 28.0

"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (ExpertLayer, persistent GEMM grid over all SMs), on sampled outputs the
oracle computes one by one: for every expert its first and last rows plus
random rows, and random output columns. Routing indices are checked in full.
"""
import numpy as np
import pytest
import torch

from oracle import formats as OF
from oracle import layer as OL
from oracle import quant as OQ
from oracle import routing as OR
from tests.layer_check import GEMM_TOL_BF16, bf16_np, check_elementwise, rel_fro, u8_np, untile_mx_scales

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _weights_on_device(w):
    g = torch.Generator(device=DEV)
    g.manual_seed(w.seed * 1000 + 4)
    w1 = (torch.randn(w.E, 2 * w.F, w.H, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn(w.E, w.H, w.F, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    return w1, w2


def _sample_rows(off, cnt, rng, n_random=4):
    rows = []
    for e in range(len(cnt)):
        c = int(cnt[e])
        if c == 0:
            continue
        lo = int(off[e])
        pick = {lo, lo + c - 1} | {lo + int(i) for i in rng.integers(0, c, n_random)}
        rows += [(e, r) for r in sorted(pick)]
    return rows


def _mx_deq_rows(codes_u8, scales_nat, fmt="e4m3"):
    return OQ.dequantize_mx(codes_u8, scales_nat, fmt)


def test_mixtral_forward_full_size_sampled():
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    w = W.WORKLOADS["mixtral_fwd"]
    E, H, F = w.E, w.H, w.F
    rng = np.random.default_rng(0)
    x = W.make_activations(w)
    idx, probs = W.make_routing(w)
    w1, w2 = _weights_on_device(w)
    lay = L.ExpertLayer(w, DEV, keep_bf16=True)
    lay.quantize_weights(w1, w2)
    lay.forward(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    rim, src, off, cnt = OR.permute_indices(idx, E, L.ALIGN)
    Rp = int(off[-1])
    assert np.array_equal(lay.offsets.cpu().numpy(), off)
    assert np.array_equal(lay.row_id_map.cpu().numpy(), rim)
    assert np.array_equal(lay.src_row.cpu().numpy()[:Rp], src)
    rows = _sample_rows(off, cnt, rng)
    rr = np.array([r for _, r in rows])
    ee = np.array([e for e, _ in rows])
    toks = src[rr] // w.k
    xf = bf16_np(x)
    # permuted activation codes / scales of the sampled rows
    cx, sx = OQ.quantize_mx(xf[toks])
    xq = u8_np(lay.xq[torch.from_numpy(rr).to(DEV)])
    xs_all = untile_mx_scales(u8_np(lay.xs), lay.R_cap, H)
    assert np.array_equal(xq, cx) and np.array_equal(xs_all[rr], sx)
    # gate/up outputs at sampled columns (gate and matching up columns)
    cols = np.sort(rng.choice(F, 48, replace=False))
    cols2 = np.concatenate([cols, cols + F])
    w1s = w1[:, torch.from_numpy(cols2).to(DEV)]                   # [E, 96, H]
    w1s_f = bf16_np(w1s)
    gu_gpu = bf16_np(lay.gu[torch.from_numpy(rr).to(DEV)])        # [S, 2F]
    w1_rows_q = u8_np(lay.w1q[:, torch.from_numpy(cols2).to(DEV)])
    w1s_all = untile_mx_scales(u8_np(lay.w1s), E * 2 * F, H).reshape(E, 2 * F, H // 32)
    refs, gots = [], []
    for e in range(E):
        cw, sw = OQ.quantize_mx(w1s_f[e])
        assert np.array_equal(w1_rows_q[e], cw)
        assert np.array_equal(w1s_all[e, cols2], sw)
        sel = ee == e
        if sel.any():
            refs.append(_mx_deq_rows(cx[sel], sx[sel]) @ _mx_deq_rows(cw, sw).T)
            gots.append(gu_gpu[sel][:, cols2])
    assert rel_fro(OF.round_to_bf16(np.concatenate(refs)), np.concatenate(gots)) <= GEMM_TOL_BF16
    # SwiGLU + quantisation of the sampled rows (from the GPU's gate/up row)
    h_gpu = bf16_np(lay.h_bf16[torch.from_numpy(rr).to(DEV)])
    check_elementwise(OL.swiglu(gu_gpu, F), h_gpu, "swiglu")
    ch, sh = OQ.quantize_mx(h_gpu)
    assert np.array_equal(u8_np(lay.hq[torch.from_numpy(rr).to(DEV)]), ch)
    assert np.array_equal(untile_mx_scales(u8_np(lay.hs), lay.R_cap, F)[rr], sh)
    # down projection at sampled columns
    ocols = np.sort(rng.choice(H, 48, replace=False))
    w2s_f = bf16_np(w2[:, torch.from_numpy(ocols).to(DEV)])        # [E, 48, F]
    y_gpu = bf16_np(lay.y[torch.from_numpy(rr).to(DEV)])
    refs, gots = [], []
    for e in range(E):
        sel = ee == e
        if not sel.any():
            continue
        cw, sw = OQ.quantize_mx(w2s_f[e])
        refs.append(_mx_deq_rows(ch[sel], sh[sel]) @ _mx_deq_rows(cw, sw).T)
        gots.append(y_gpu[sel][:, ocols])
    assert rel_fro(OF.round_to_bf16(np.concatenate(refs)), np.concatenate(gots)) <= GEMM_TOL_BF16
    # combine of sampled tokens from the GPU's expert outputs
    tsel = np.unique(toks)[:64]
    y_rows = bf16_np(lay.y[torch.from_numpy(rim[tsel].reshape(-1)).to(DEV)]).reshape(len(tsel), w.k, H)
    ref = np.einsum("tk,tkh->th", probs[tsel].astype(np.float64), y_rows)
    check_elementwise(ref, bf16_np(lay.out[torch.from_numpy(tsel).to(DEV)]), "unpermute")


@pytest.mark.parametrize("name", ["scout_fwd", "finegrained_fwd"])
def test_blockwise_and_nvfp4_forward_full_size_sampled(name):
    """The Scout-shaped blockwise FP8 forward (1x128 activations, 128x128
    weights, Zipf loads with empty experts) and the fine-grained NVFP4 forward
    (128 experts, top-8) at full size: routing in full; sampled rows of the X
    and h codes and scales, every s_g (NVFP4); gate/up and down outputs at
    sampled rows and columns against the oracle's GEMM on the identical
    quantised inputs (blockwise weights requantised by the 128x128 slabs that
    hold the sampled columns); SwiGLU from the GPU's own gate/up rows; the
    combine of sampled tokens."""
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    from tests.layer_check import _gpu_row_scales, _q_rows
    w = W.WORKLOADS[name]
    recipe = w.recipe
    nv = recipe == "nvfp4"
    E, H, F, k = w.E, w.H, w.F, w.k
    rng = np.random.default_rng(3)
    x = W.make_activations(w)
    idx, probs = W.make_routing(w)
    w1, w2 = _weights_on_device(w)
    lay = L.ExpertLayer(w, DEV, keep_bf16=True)
    assert not lay.train and lay.recipe == recipe
    lay.quantize_weights(w1, w2)
    lay.forward(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    rim, src, off, cnt = OR.permute_indices(idx, E, lay.align)
    Rp = int(off[-1])
    assert np.array_equal(lay.offsets.cpu().numpy(), off)
    assert np.array_equal(lay.counts.cpu().numpy(), cnt)
    assert np.array_equal(lay.row_id_map.cpu().numpy(), rim)
    assert np.array_equal(lay.src_row.cpu().numpy()[:Rp], src)
    rows = _sample_rows(off, cnt, rng, n_random=2 if nv else 4)
    rr = np.array([r for _, r in rows])
    ee = np.array([e for e, _ in rows])
    rrd = torch.from_numpy(rr).to(DEV)
    toks = src[rr] // k
    xf = bf16_np(x)
    # X: the tensor's s_g (NVFP4) and the sampled rows' codes and scales
    if nv:
        sg_x = OQ.nvfp4_global_scale(np.max(np.abs(xf)))
        assert float(lay.nv_sg[0].item()) == float(sg_x)
        cx, sx = OQ.quantize_nvfp4(xf[toks], sg_x)
        x_deq = OQ.dequantize_nvfp4(cx, sx, sg_x, H)
    else:
        cx, sx, x_deq = _q_rows(xf[toks], recipe)
    assert np.array_equal(u8_np(lay.xq[rrd]), cx)
    assert np.array_equal(_gpu_row_scales(lay, lay.xs, lay.R_cap, H, recipe)[rr], sx)

    def weight_rows(wt, wscales, e, sel_rows, slot):
        """Codes and dequantised values of rows `sel_rows` of expert e's weight
        [N, K] (bf16 on the device), quantised here: NVFP4 with the s_g of the
        whole expert (checked against the GPU's), blockwise through the
        128x128 slabs holding the rows (their scales checked against the
        GPU's)."""
        we = wt[e]
        if nv:
            sg = OQ.nvfp4_global_scale(np.max(np.abs(bf16_np(we))))
            assert float(lay.nv_sg[slot + e].item()) == float(sg)
            c, sc = OQ.quantize_nvfp4(bf16_np(we[torch.from_numpy(sel_rows).to(DEV)]), sg)
            return c, OQ.dequantize_nvfp4(c, sc, sg, we.shape[1])
        gpu_si = wscales[e].cpu().numpy()                               # [N/128, K/128]
        slabs = {}
        for b in np.unique(sel_rows // 128):
            c, si = OQ.quantize_block_128x128(bf16_np(we[128 * b:128 * b + 128]), "e4m3")
            assert np.array_equal(gpu_si[b], si[0])
            slabs[b] = (c, OQ.dequantize_block_128x128(c, si))
        return (np.stack([slabs[n // 128][0][n % 128] for n in sel_rows]),
                np.stack([slabs[n // 128][1][n % 128] for n in sel_rows]))

    def sample_cols(n_total, n_blocks=3, per_block=8):
        blocks = rng.choice(n_total // 128, n_blocks, replace=False)
        return np.sort(np.concatenate([128 * b + rng.choice(128, per_block, replace=False) for b in blocks]))

    # gate/up at sampled gate columns and the matching up columns
    cols = sample_cols(F)
    cols2 = np.concatenate([cols, cols + F])
    gu_gpu = bf16_np(lay.gu[rrd])                                   # [S, 2F]
    w1q_s = u8_np(lay.w1q[:, torch.from_numpy(cols2).to(DEV)])
    refs, gots = [], []
    for e in range(E):
        sel = ee == e
        if not sel.any():
            continue
        c, d = weight_rows(w1, lay.w1s, e, cols2, 2)
        assert np.array_equal(w1q_s[e], c)
        refs.append(x_deq[sel] @ d.T)
        gots.append(gu_gpu[sel][:, cols2])
    assert rel_fro(OF.round_to_bf16(np.concatenate(refs)), np.concatenate(gots)) <= GEMM_TOL_BF16
    # SwiGLU of the GPU's gate/up rows; h codes from the GPU's h
    h_gpu = bf16_np(lay.h_bf16[rrd])
    check_elementwise(OL.swiglu(gu_gpu, F), h_gpu, "swiglu")
    if nv:
        # s_g of h from the GPU's whole h (the quantiser's input), reduced here in row chunks
        h_all = max(float(np.max(np.abs(bf16_np(lay.h_bf16[r0:min(r0 + 32768, Rp)]))))
                    for r0 in range(0, Rp, 32768))
        sg_h = OQ.nvfp4_global_scale(h_all)
        assert float(lay.nv_sg[1].item()) == float(sg_h)
        ch, sh = OQ.quantize_nvfp4(h_gpu, sg_h)
        h_deq = OQ.dequantize_nvfp4(ch, sh, sg_h, F)
    else:
        ch, sh, h_deq = _q_rows(h_gpu, recipe)
    assert np.array_equal(u8_np(lay.hq[rrd]), ch)
    assert np.array_equal(_gpu_row_scales(lay, lay.hs, lay.R_cap, F, recipe)[rr], sh)
    # down projection at sampled columns
    ocols = sample_cols(H)
    y_gpu = bf16_np(lay.y[rrd])
    w2q_s = u8_np(lay.w2q[:, torch.from_numpy(ocols).to(DEV)])
    refs, gots = [], []
    for e in range(E):
        sel = ee == e
        if not sel.any():
            continue
        c, d = weight_rows(w2, lay.w2s, e, ocols, 2 + E)
        assert np.array_equal(w2q_s[e], c)
        refs.append(h_deq[sel] @ d.T)
        gots.append(y_gpu[sel][:, ocols])
    assert rel_fro(OF.round_to_bf16(np.concatenate(refs)), np.concatenate(gots)) <= GEMM_TOL_BF16
    # combine of sampled tokens from the GPU's expert outputs
    tsel = np.unique(toks)[:64]
    y_rows = bf16_np(lay.y[torch.from_numpy(rim[tsel].reshape(-1)).to(DEV)]).reshape(len(tsel), k, H)
    ref = np.einsum("tk,tkh->th", probs[tsel].astype(np.float64), y_rows)
    check_elementwise(ref, bf16_np(lay.out[torch.from_numpy(tsel).to(DEV)]), "unpermute")


def test_mixtral_training_step_full_size_sampled():
    """The fwd+bwd step of the bench workload (hybrid e4m3/e5m2, delayed
    scaling), after two warm-up steps so the scales are non-trivial; sampled
    dgrad rows and sampled wgrad elements against the oracle."""
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    w = W.WORKLOADS["mixtral_fwdbwd"]
    E, H, F = w.E, w.H, w.F
    rng = np.random.default_rng(1)
    x = W.make_activations(w)
    idx, probs = W.make_routing(w)
    dout = W.make_dout(w)
    w1, w2 = _weights_on_device(w)
    lay = L.ExpertLayer(w, DEV, keep_bf16=True)
    xd, idxd, pd, dd = x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV), dout.to(DEV)
    for _ in range(2):
        lay.quantize_weights(w1, w2)
        lay.forward(xd, idxd, pd)
        lay.backward(dd, pd)
        lay.update_scaling()
    fs = lay.fwd_scale.cpu().numpy().copy()
    bs = lay.bwd_scale.cpu().numpy().copy()
    lay.quantize_weights(w1, w2)
    lay.forward(xd, idxd, pd)
    lay.backward(dd, pd)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    assert np.all(fs != 1.0) and np.all(bs != 1.0)
    rim, src, off, cnt = OR.permute_indices(idx, E, L.ALIGN)
    rows = _sample_rows(off, cnt, rng)
    rr = np.array([r for _, r in rows])
    ee = np.array([e for e, _ in rows])
    toks = src[rr] // w.k
    slots = src[rr] % w.k
    # dY2 codes of the sampled rows: float32(probs * dout) cast with the e5m2 scale
    dy32 = (probs[toks, slots][:, None].astype(np.float32) * bf16_np(dout[torch.from_numpy(toks)]).astype(np.float32))
    c2, _ = OQ.quantize_tensor(dy32.astype(np.float64), bs[0], "e5m2")
    rrd = torch.from_numpy(rr).to(DEV)
    assert np.array_equal(u8_np(lay.dy2q[rrd]), c2)
    # dgrad of the down projection (dh) at sampled columns
    fcols = np.sort(rng.choice(F, 48, replace=False))
    w2c = bf16_np(w2[:, :, torch.from_numpy(fcols).to(DEV)])          # [E, H, 48]
    dh_gpu = bf16_np(lay.dh[rrd])
    refs, gots = [], []
    for e in range(E):
        sel = ee == e
        if not sel.any():
            continue
        cw, _ = OQ.quantize_tensor(w2c[e], fs[2 + E + e])
        refs.append(OQ.dequantize_tensor(c2[sel], bs[0], "e5m2") @ OQ.dequantize_tensor(cw, fs[2 + E + e]))
        gots.append(dh_gpu[sel][:, fcols])
    assert rel_fro(OF.round_to_bf16(np.concatenate(refs)), np.concatenate(gots)) <= GEMM_TOL_BF16
    # wgrad of the gate/up projection at sampled (n, k) of every expert:
    # dW1[e, n, k] = sum over the expert's rows of dY1[r, n] * X[r, k]; the
    # GEMM read the row-wise codes dY1 [R, 2F] and X [R, H] MN-major
    assert lay.mn and lay.xcol is None
    ns = np.sort(rng.choice(2 * F, 8, replace=False))
    ks = np.sort(rng.choice(H, 8, replace=False))
    dw1 = lay.dw1
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        dyc = u8_np(lay.dy1q[lo:hi][:, torch.from_numpy(ns).to(DEV)]).T     # [8, rows]
        xc = u8_np(lay.xq[lo:hi][:, torch.from_numpy(ks).to(DEV)]).T        # [8, rows]
        ref = OQ.dequantize_tensor(dyc, bs[1], "e5m2") @ OQ.dequantize_tensor(xc, fs[0]).T
        got = dw1[e][torch.from_numpy(ns).to(DEV)][:, torch.from_numpy(ks).to(DEV)].cpu().numpy()
        assert rel_fro(ref, got) <= 1e-5, e


@pytest.mark.parametrize("recipe", ["mxfp8", "nvfp4"])
def test_block_scaled_training_step_full_size_sampled(recipe):
    """The MXFP8 and NVFP4 training steps at the full Mixtral size: routing in
    full; the row-wise dY2 codes and scales of sampled rows (NVFP4: with s_g
    from the dY amax, max |fl(p d)| = fl(|p| max |d|)); dh at sampled rows and
    columns against the oracle's GEMM of the dequantised dY2 rows and the weight
    copy requantised here; sampled gate/up wgrad elements from the column-wise
    copies."""
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    w = W.WORKLOADS["mixtral_fwdbwd_mx" if recipe == "mxfp8" else "mixtral_fwdbwd_nvfp4"]
    E, H, F, k = w.E, w.H, w.F, w.k
    nv = recipe == "nvfp4"
    rng = np.random.default_rng(2)
    x = W.make_activations(w)
    idx, probs = W.make_routing(w)
    dout = W.make_dout(w)
    w1, w2 = _weights_on_device(w)
    # (MXFP8: dh comes out of the dSwiGLU epilogue of the down dgrad only when asked for)
    lay = L.ExpertLayer(w, DEV, keep_bf16=not nv)
    assert lay.train
    lay.quantize_weights(w1, w2)
    lay.forward(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV))
    lay.backward(dout.to(DEV), torch.from_numpy(probs).to(DEV))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    rim, src, off, cnt = OR.permute_indices(idx, E, lay.align)
    Rp = int(off[-1])
    R = lay.R_cap
    assert np.array_equal(lay.offsets.cpu().numpy(), off)
    assert np.array_equal(lay.row_id_map.cpu().numpy(), rim)
    assert np.array_equal(lay.src_row.cpu().numpy()[:Rp], src)
    rows = _sample_rows(off, cnt, rng)
    rr = np.array([r for _, r in rows])
    ee = np.array([e for e, _ in rows])
    toks, slots = src[rr] // k, src[rr] % k
    df = bf16_np(dout).astype(np.float32)
    dy32 = probs[toks, slots][:, None].astype(np.float32) * df[toks]
    rrd = torch.from_numpy(rr).to(DEV)
    if nv:
        i2, i1 = 2 + 2 * E, 3 + 2 * E
        am = float(np.max(np.abs(probs).astype(np.float32) * np.max(np.abs(df), axis=1)[:, None]))
        s_g = OQ.nvfp4_global_scale(am)
        assert float(lay.nv_amax[i2].item()) == am and float(lay.nv_sg[i2].item()) == float(s_g)
        c2, s2 = OQ.quantize_nvfp4(dy32.astype(np.float64), s_g)
        got_s = untile_mx_scales(u8_np(lay.dy2s), R, H, 16)[rr]
        dy2_deq = OQ.dequantize_nvfp4(c2, s2, s_g, H)
    else:
        c2, s2 = OQ.quantize_mx(dy32.astype(np.float64), "e5m2")
        got_s = untile_mx_scales(u8_np(lay.dy2s), R, H)[rr]
        dy2_deq = OQ.dequantize_mx(c2, s2, "e5m2")
    assert np.array_equal(u8_np(lay.dy2q[rrd]), c2)
    assert np.array_equal(got_s, s2)
    # dh = dY2 W2_e at sampled columns; the dgrad reads W2's column-wise copy
    # (blocks along H), requantised here from the bf16 weight
    fcols = np.sort(rng.choice(F, 24, replace=False))
    dh_gpu = bf16_np(lay.dh[rrd])
    refs, gots = [], []
    for e in range(E):
        sel = ee == e
        if not sel.any():
            continue
        if nv:
            w2e = w2[e].float().cpu().numpy()                          # [H, F]
            sg_w = OQ.nvfp4_global_scale(float(np.max(np.abs(w2e))))
            cols = []
            for f in fcols:
                fb = f // 16
                _, _, cc, cs = OQ.quantize_nvfp4_2d(w2e[:, 16 * fb:16 * fb + 16], sg_w)
                cols.append(OQ.dequantize_nvfp4(cc, cs, sg_w, H)[f - 16 * fb])
            wcol = np.stack(cols)                                      # [24, H]
        else:
            w2c = bf16_np(w2[e][:, torch.from_numpy(fcols).to(DEV)])   # [H, 24]
            cc, cs = OQ.quantize_mx(np.ascontiguousarray(w2c.T))
            wcol = OQ.dequantize_mx(cc, cs)
        refs.append(dy2_deq[sel] @ wcol.T)
        gots.append(dh_gpu[sel][:, fcols])
    assert rel_fro(OF.round_to_bf16(np.concatenate(refs)), np.concatenate(gots)) <= GEMM_TOL_BF16
    # gate/up wgrad at sampled (n, k): sum over the expert's rows of the
    # column-wise dY1 and X copies, dequantised
    ns = np.sort(rng.choice(2 * F, 6, replace=False))
    ks = np.sort(rng.choice(H, 6, replace=False))
    nsd, ksd = torch.from_numpy(ns).to(DEV), torch.from_numpy(ks).to(DEV)
    blk = 16 if nv else 32
    dyc_s = untile_mx_scales(u8_np(lay.dy1cs), 2 * F, R, blk)[ns]
    xc_s = untile_mx_scales(u8_np(lay.xcs), H, R, blk)[ks]
    dyc_all, xc_all = u8_np(lay.dy1col[nsd]), u8_np(lay.xcol[ksd])
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        # (the columns past the rows in use are never written: dequantise [0, Rp) only)
        if nv:
            dq = OQ.dequantize_nvfp4(dyc_all[:, :Rp // 2], dyc_s[:, :Rp // 16], float(lay.nv_sg[i1].item()),
                                     Rp)[:, lo:hi]
            xq = OQ.dequantize_nvfp4(xc_all[:, :Rp // 2], xc_s[:, :Rp // 16], float(lay.nv_sg[0].item()),
                                     Rp)[:, lo:hi]
        else:
            dq = OQ.dequantize_mx(dyc_all[:, :Rp], dyc_s[:, :Rp // 32], "e5m2")[:, lo:hi]
            xq = OQ.dequantize_mx(xc_all[:, :Rp], xc_s[:, :Rp // 32])[:, lo:hi]
        ref = dq @ xq.T
        got = lay.dw1[e][nsd][:, ksd].cpu().numpy()
        assert rel_fro(ref, got) <= 1e-5, e

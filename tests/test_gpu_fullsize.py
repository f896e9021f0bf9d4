"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (ExpertLayer, persistent GEMM grid over all SMs).

What is compared, for every workload:
* routing indices (offsets, counts, row_id_map, src_row): in full, bit-exact;
* permute + quantise: the codes and scales of every routed row, bit-exact
  (the oracle quantises every token, tests/fullsize_pool.py spreads that over
  the host cores); training also the column-wise copies in full;
* weight quantisation: every code and scale of both weights, bit-exact (and
  the column-wise copies where the recipe writes them);
* grouped GEMMs (forward, and for training the dgrads): for every expert its
  first and last rows plus 126 random rows, against ALL output columns, as the
  oracle's float64 GEMM of the same quantised operands;
* SwiGLU / dSwiGLU and the codes quantised from them on the sampled rows,
  from the GPU's bf16 operands (exp is not reproducible bit for bit);
* unpermute, permute-backward and the unpermute-backward's dY codes and
  dprobs: every token;
* wgrads: 16 x 16 sampled (n, k) elements of every expert.
Training runs for the per-tensor (delayed) headline, MXFP8, NVFP4 and
blockwise recipes.
"""
import numpy as np
import pytest
import torch

from oracle import formats as OF
from oracle import layer as OL
from oracle import quant as OQ
from oracle import routing as OR
from tests import fullsize_pool as FP
from tests.layer_check import (GEMM_TOL_BF16, GEMM_TOL_F32, bf16_np, check_elementwise, rel_fro, u8_np,
                               untile_mx_scales)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
N_RANDOM = 126          # random rows per expert beside its first and last


def _weights_on_device(w):
    g = torch.Generator(device=DEV)
    g.manual_seed(w.seed * 1000 + 4)
    w1 = (torch.randn(w.E, 2 * w.F, w.H, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    w2 = (torch.randn(w.E, w.H, w.F, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    return w1, w2


def _bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its bit patterns (uint16) on the host."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _amax_bits(bits: np.ndarray) -> float:
    """max |x| of finite bf16 values from their bit patterns (the magnitude
    bits order like the values)."""
    return float(OF.bf16_bits_to_f64(np.array([np.max(bits & 0x7FFF)], dtype=np.uint16))[0])


def _sample_rows(off, cnt, rng, n_random=N_RANDOM):
    """(expert, row) pairs: every non-empty group's first and last rows plus
    n_random distinct random rows (all rows of a smaller group)."""
    rows = []
    for e in range(len(cnt)):
        c = int(cnt[e])
        if c == 0:
            continue
        lo = int(off[e])
        pick = {lo, lo + c - 1} | {lo + int(i) for i in rng.choice(c, min(c, n_random), replace=False)}
        rows += [(e, r) for r in sorted(pick)]
    return np.array([e for e, _ in rows]), np.array([r for _, r in rows])


def _gather(t, rows):
    return t[torch.from_numpy(np.asarray(rows)).to(t.device)]


def _by_expert(ee, arr):
    return {int(e): arr[ee == e] for e in np.unique(ee)}


def _gemm_check(fwd_by_e, gpu_rows, ee, what):
    """Oracle float64 rows (per expert, sampled-row order) rounded to bf16
    against the GPU's rows: relative Frobenius error within the bf16 GEMM
    tolerance."""
    ref = np.concatenate([fwd_by_e[int(e)] for e in np.unique(ee)])
    got = np.concatenate([gpu_rows[ee == e] for e in np.unique(ee)])
    err = rel_fro(OF.round_to_bf16(ref), got)
    assert err <= GEMM_TOL_BF16, f"{what}: rel Frobenius {err:.3e}"
    return err


def _routing(lay, idx, E):
    rim, src, off, cnt = OR.permute_indices(idx, E, lay.align)
    Rp = int(off[-1])
    assert np.array_equal(lay.offsets.cpu().numpy(), off)
    assert np.array_equal(lay.counts.cpu().numpy(), cnt)
    assert np.array_equal(lay.row_id_map.cpu().numpy(), rim)
    assert np.array_equal(lay.src_row.cpu().numpy()[:Rp], src)
    return rim, src, off, cnt, Rp


def _check_permuted(gpu_codes, gpu_scales, codes, scales, rim, Rp, what):
    """Every routed row (and every filler row: zero codes, zero scales) of the
    GPU's permuted copy against the oracle's per-token quantisation."""
    assert np.array_equal(gpu_codes[:Rp], OR.permute_rows(codes, rim, Rp)), f"{what} codes"
    if scales is not None:
        assert np.array_equal(gpu_scales[:Rp], OR.permute_rows(scales, rim, Rp)), f"{what} scales"


def _wgrad_samples(lay_dw, e, ns, ks, dy_cols, a_cols):
    """dW[e, n, k] = sum over the expert's rows of dY[r, n] A[r, k] at the
    sampled (n, k): dy_cols [rows, |ns|], a_cols [rows, |ks|] dequantised."""
    ref = dy_cols.T @ a_cols
    got = lay_dw[e][torch.from_numpy(ns).to(DEV)][:, torch.from_numpy(ks).to(DEV)].cpu().numpy()
    err = rel_fro(ref, got)
    assert err <= GEMM_TOL_F32, (e, err)


# ---------------------------------------------------------------------------- forward configurations

@pytest.mark.parametrize("name", ["mixtral_fwd", "scout_fwd", "finegrained_fwd"])
def test_forward_full_size(name):
    """The three forward configurations: MXFP8 Mixtral (outlier channels),
    blockwise FP8 Scout (1x128 / 128x128, Zipf loads with empty experts),
    NVFP4 fine-grained (128 experts, top-8)."""
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    w = W.WORKLOADS[name]
    E, H, F, k, recipe = w.E, w.H, w.F, w.k, w.recipe
    nv, blk = recipe == "nvfp4", recipe == "blockwise"
    rng = np.random.default_rng(7)
    x = W.make_activations(w)
    idx, probs = W.make_routing(w)
    w1, w2 = _weights_on_device(w)
    lay = L.ExpertLayer(w, DEV, keep_bf16=True)
    assert not lay.train and lay.recipe == recipe
    lay.quantize_weights(w1, w2)
    lay.forward(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV))
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    rim, src, off, cnt, Rp = _routing(lay, idx, E)
    R = lay.R_cap

    def row_scales(buf, rows, ld):
        if nv:
            return untile_mx_scales(u8_np(buf), rows, ld, 16)
        if blk:
            return buf.cpu().numpy().T            # [ld/128][rows] -> [rows, ld/128]
        return untile_mx_scales(u8_np(buf), rows, ld)

    # permute + quantise, every routed row
    xb = _bits(x)
    if nv:
        sg_x = OQ.nvfp4_global_scale(_amax_bits(xb))
        assert float(lay.nv_sg[0].item()) == float(sg_x)
        cx, sx = FP.quantize_rows(xb, "nv", s_g=float(sg_x))
    else:
        cx, sx = FP.quantize_rows(xb, "blk" if blk else "mx")
    _check_permuted(u8_np(lay.xq), row_scales(lay.xs, R, H), cx, sx, rim, Rp, "X")
    ee, rr = _sample_rows(off, cnt, rng)
    toks = src[rr] // k
    if nv:
        x_deq = OQ.dequantize_nvfp4(cx[toks], sx[toks], sg_x, H)
    elif blk:
        x_deq = OQ.dequantize_block_1x128(cx[toks], sx[toks])
    else:
        x_deq = OQ.dequantize_mx(cx[toks], sx[toks])

    # weights in full; gate/up at the sampled rows against all 2F columns
    def weight_gpu(q, s, N, K):
        g = {"codes": u8_np(q)}
        if nv:
            g["scales"] = untile_mx_scales(u8_np(s), E * N, K, 16).reshape(E, N, K // 16)
        elif blk:
            g["scales"] = s.cpu().numpy()
        else:
            g["scales"] = untile_mx_scales(u8_np(s), E * N, K).reshape(E, N, K // 32)
        return g

    wrec = "nv" if nv else ("blk" if blk else "mx")

    def per_expert(wb, slot):
        if not nv:
            return None
        sg = np.array([OQ.nvfp4_global_scale(_amax_bits(wb[e])) for e in range(E)], dtype=np.float32)
        assert np.array_equal(lay.nv_sg[slot:slot + E].cpu().numpy(), sg)
        return {"s_g": sg}

    w1b = _bits(w1)
    tot, fwd1, _ = FP.weight_sweep(w1b, wrec, gpu=weight_gpu(lay.w1q, lay.w1s, 2 * F, H),
                                   a_rows=_by_expert(ee, x_deq), per_expert=per_expert(w1b, 2))
    del w1b
    assert all(v == 0 for v in tot.values()), tot
    gu_gpu = bf16_np(_gather(lay.gu, rr))
    _gemm_check(fwd1, gu_gpu, ee, "gate/up")

    # SwiGLU and h's codes on the sampled rows, from the GPU's gate/up rows
    h_gpu = bf16_np(_gather(lay.h_bf16, rr))
    check_elementwise(OL.swiglu(gu_gpu, F), h_gpu, "swiglu")
    if nv:
        # s_g of h: the amax of the whole materialised h
        h_amax = max(_amax_bits(_bits(lay.h_bf16[r0:min(r0 + 32768, Rp)])) for r0 in range(0, Rp, 32768))
        sg_h = OQ.nvfp4_global_scale(h_amax)
        assert float(lay.nv_sg[1].item()) == float(sg_h)
        ch, sh = OQ.quantize_nvfp4(h_gpu, sg_h)
        h_deq = OQ.dequantize_nvfp4(ch, sh, sg_h, F)
    elif blk:
        ch, sh = OQ.quantize_block_1x128(h_gpu)
        h_deq = OQ.dequantize_block_1x128(ch, sh)
    else:
        ch, sh = OQ.quantize_mx(h_gpu)
        h_deq = OQ.dequantize_mx(ch, sh)
    assert np.array_equal(u8_np(_gather(lay.hq, rr)), ch)
    assert np.array_equal(row_scales(lay.hs, R, F)[rr], sh)

    # down projection at the sampled rows against all H columns
    w2b = _bits(w2)
    tot, fwd2, _ = FP.weight_sweep(w2b, wrec, gpu=weight_gpu(lay.w2q, lay.w2s, H, F),
                                   a_rows=_by_expert(ee, h_deq), per_expert=per_expert(w2b, 2 + E))
    del w2b
    assert all(v == 0 for v in tot.values()), tot
    _gemm_check(fwd2, bf16_np(_gather(lay.y, rr)), ee, "down")

    # unpermute of every token from the GPU's expert outputs
    check_elementwise(OR.unpermute(bf16_np(lay.y[:Rp]), rim, probs), bf16_np(lay.out), "unpermute")


# ---------------------------------------------------------------------------- training configurations

def _train_layer(name, warm_steps, keep_bf16=True):
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import mgq
    from fp8_grouped_gemm_gb300 import workloads as W
    w = W.WORKLOADS[name]
    x = W.make_activations(w)
    idx, probs = W.make_routing(w)
    dout = W.make_dout(w)
    w1, w2 = _weights_on_device(w)
    lay = L.ExpertLayer(w, DEV, keep_bf16=keep_bf16)
    assert lay.train
    xd, idxd, pd, dd = x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(probs).to(DEV), dout.to(DEV)
    for _ in range(warm_steps):
        lay.quantize_weights(w1, w2)
        lay.forward(xd, idxd, pd)
        lay.backward(dd, pd)
        lay.update_scaling()
    fs = lay.fwd_scale.cpu().numpy().copy() if lay.delayed else None
    bs = lay.bwd_scale.cpu().numpy().copy() if lay.delayed else None
    lay.quantize_weights(w1, w2)
    lay.forward(xd, idxd, pd)
    lay.backward(dd, pd)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    return w, lay, x, idx, probs, dout, w1, w2, fs, bs


def test_mixtral_training_step_full_size():
    """The bench's headline step (hybrid e4m3 / e5m2, delayed scaling, history
    1024) after two warm-up steps, so every scale is non-trivial. Scales of X,
    the weights and dY2 come from the oracle's own amaxes and must equal the
    GPU's; h's and dY1's scales come from the GPU's bf16 intermediates of the
    earlier steps and are taken as given."""
    w, lay, x, idx, probs, dout, w1, w2, fs, bs = _train_layer("mixtral_fwdbwd", 2)
    E, H, F, k = w.E, w.H, w.F, w.k
    rng = np.random.default_rng(11)
    assert lay.mn and lay.delayed
    rim, src, off, cnt, Rp = _routing(lay, idx, E)
    f32 = np.float32
    # delayed scales of the roles the oracle can compute: max_finite / amax
    xb, w1b, w2b = _bits(x), _bits(w1), _bits(w2)
    s_x = f32(448.0) / f32(_amax_bits(xb))
    s_w1 = np.array([f32(448.0) / f32(_amax_bits(w1b[e])) for e in range(E)], dtype=f32)
    s_w2 = np.array([f32(448.0) / f32(_amax_bits(w2b[e])) for e in range(E)], dtype=f32)
    assert fs[0] == s_x and np.array_equal(fs[2:2 + E], s_w1) and np.array_equal(fs[2 + E:2 + 2 * E], s_w2)
    dy32, dprobs_ref = OR.unpermute_bwd(bf16_np(dout), bf16_np(lay.y[:Rp]), rim, probs, Rp)
    s_dy2 = f32(57344.0) / f32(np.max(np.abs(dy32)))
    assert bs[0] == s_dy2
    s_h, s_dy1 = fs[1], bs[1]

    # permute + quantise: every row
    cx, _ = FP.quantize_rows(xb, "tensor", scale=float(s_x))
    _check_permuted(u8_np(lay.xq), None, cx, None, rim, Rp, "X")
    ee, rr = _sample_rows(off, cnt, rng)
    toks = src[rr] // k
    x_deq = OQ.dequantize_tensor(cx[toks], s_x)

    # unpermute backward: every dY2 code, every dprobs
    c2, _ = FP.quantize_rows(dy32, "tensor_e5m2", scale=float(s_dy2))
    assert np.array_equal(u8_np(lay.dy2q[:Rp]), c2)
    assert rel_fro(dprobs_ref, lay.dprobs.cpu().numpy()) <= 1e-5
    dy2_deq = OQ.dequantize_tensor(c2[rr], s_dy2, "e5m2")

    # W1 in full: gate/up forward at the sampled rows (all 2F columns); the
    # dY1 rows for the gate/up dgrad are filled in below, after dSwiGLU
    gu_gpu = bf16_np(_gather(lay.gu, rr))
    h_gpu = bf16_np(_gather(lay.h_bf16, rr))
    check_elementwise(OL.swiglu(gu_gpu, F), h_gpu, "swiglu")
    ch, _ = OQ.quantize_tensor(h_gpu, s_h)
    assert np.array_equal(u8_np(_gather(lay.hq, rr)), ch)
    h_deq = OQ.dequantize_tensor(ch, s_h)

    # W2 in full: down forward (all H columns) and down dgrad dh (all F
    # columns) at the sampled rows, from one sweep
    tot, fwd2, dgr2 = FP.weight_sweep(w2b, "tensor", gpu={"codes": u8_np(lay.w2q)}, a_rows=_by_expert(ee, h_deq),
                                      dy_rows=_by_expert(ee, dy2_deq), per_expert={"scale": s_w2})
    assert tot == {"codes": 0}, tot
    _gemm_check(fwd2, bf16_np(_gather(lay.y, rr)), ee, "down fwd")
    dh_gpu = bf16_np(_gather(lay.dh, rr))
    _gemm_check(dgr2, dh_gpu, ee, "down dgrad")

    # dSwiGLU and dY1's codes on the sampled rows, from the GPU's dh and g | u
    dgu_gpu = bf16_np(_gather(lay.dgu_bf16, rr))
    check_elementwise(OL.dswiglu(dh_gpu, gu_gpu, F), dgu_gpu, "dswiglu")
    c1, _ = OQ.quantize_tensor(dgu_gpu, s_dy1, "e5m2")
    assert np.array_equal(u8_np(_gather(lay.dy1q, rr)), c1)
    dy1_deq = OQ.dequantize_tensor(c1, s_dy1, "e5m2")

    tot, fwd1, dgr1 = FP.weight_sweep(w1b, "tensor", gpu={"codes": u8_np(lay.w1q)}, a_rows=_by_expert(ee, x_deq),
                                      dy_rows=_by_expert(ee, dy1_deq), per_expert={"scale": s_w1})
    assert tot == {"codes": 0}, tot
    _gemm_check(fwd1, gu_gpu, ee, "gate/up fwd")
    _gemm_check(dgr1, bf16_np(_gather(lay.dxp, rr)), ee, "gate/up dgrad")

    # unpermute and permute backward: every token
    check_elementwise(OR.unpermute(bf16_np(lay.y[:Rp]), rim, probs), bf16_np(lay.out), "unpermute")
    check_elementwise(OR.permute_bwd(bf16_np(lay.dxp[:Rp]), rim), bf16_np(lay.dx), "permute_bwd")

    # wgrads at 16 x 16 sampled (n, k) of every expert (the GEMMs read the
    # row-wise codes MN-major)
    ns2, ks2 = np.sort(rng.choice(H, 16, replace=False)), np.sort(rng.choice(F, 16, replace=False))
    ns1, ks1 = np.sort(rng.choice(2 * F, 16, replace=False)), np.sort(rng.choice(H, 16, replace=False))
    cx_perm = OR.permute_rows(cx, rim, Rp)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        # down: dY2 (oracle codes) x h (GPU h quantised here) over the expert's rows
        hk = bf16_np(lay.h_bf16[lo:hi][:, torch.from_numpy(ks2).to(DEV)])
        hk_c, _ = OQ.quantize_tensor(hk, s_h)
        assert np.array_equal(u8_np(lay.hq[lo:hi][:, torch.from_numpy(ks2).to(DEV)]), hk_c)
        _wgrad_samples(lay.dw2, e, ns2, ks2, OQ.dequantize_tensor(c2[lo:hi][:, ns2], s_dy2, "e5m2"),
                       OQ.dequantize_tensor(hk_c, s_h))
        # gate/up: dY1 (GPU dG | dU quantised here) x X (oracle codes)
        dn = bf16_np(lay.dgu_bf16[lo:hi][:, torch.from_numpy(ns1).to(DEV)])
        dn_c, _ = OQ.quantize_tensor(dn, s_dy1, "e5m2")
        assert np.array_equal(u8_np(lay.dy1q[lo:hi][:, torch.from_numpy(ns1).to(DEV)]), dn_c)
        _wgrad_samples(lay.dw1, e, ns1, ks1, OQ.dequantize_tensor(dn_c, s_dy1, "e5m2"),
                       OQ.dequantize_tensor(cx_perm[lo:hi][:, ks1], s_x))


@pytest.mark.parametrize("recipe", ["mxfp8", "nvfp4"])
def test_block_scaled_training_step_full_size(recipe):
    """The MXFP8 and NVFP4 training steps at the full Mixtral size. Besides
    the forward checks: the column-wise copies of X and dY2 in full (blocks
    along each expert's tokens), both copies of every weight, the dgrads at
    the sampled rows against all columns (through the column-wise weight
    copies), and sampled wgrad elements from the column-wise copies."""
    nv = recipe == "nvfp4"
    name = "mixtral_fwdbwd_nvfp4" if nv else "mixtral_fwdbwd_mx"
    w, lay, x, idx, probs, dout, w1, w2, _, _ = _train_layer(name, 0)
    E, H, F, k = w.E, w.H, w.F, w.k
    rng = np.random.default_rng(12)
    rim, src, off, cnt, Rp = _routing(lay, idx, E)
    R = lay.R_cap
    blk = 16 if nv else 32

    def sc(buf, rows, ld):
        return untile_mx_scales(u8_np(buf), rows, ld, blk)

    # X row-wise (every routed row) and column-wise ([H, R_cap], in full)
    xb = _bits(x)
    if nv:
        sg_x = OQ.nvfp4_global_scale(_amax_bits(xb))
        assert float(lay.nv_sg[0].item()) == float(sg_x)
        cx, sx = FP.quantize_rows(xb, "nv", s_g=float(sg_x))
    else:
        cx, sx = FP.quantize_rows(xb, "mx")
    _check_permuted(u8_np(lay.xq), sc(lay.xs, R, H), cx, sx, rim, Rp, "X")
    xperm_t = np.ascontiguousarray(OR.permute_rows(xb, rim, Rp).T)       # bf16 bits [H, Rp], filler rows 0
    if nv:
        ccx, csx = FP.quantize_rows(xperm_t, "nv", s_g=float(sg_x))
        assert np.array_equal(u8_np(lay.xcol)[:, :Rp // 2], ccx)
    else:
        ccx, csx = FP.quantize_rows(xperm_t, "mx")
        assert np.array_equal(u8_np(lay.xcol)[:, :Rp], ccx)
    assert np.array_equal(sc(lay.xcs, H, R)[:, :Rp // blk], csx)
    del xperm_t
    ee, rr = _sample_rows(off, cnt, rng)
    toks = src[rr] // k
    x_deq = OQ.dequantize_nvfp4(cx[toks], sx[toks], sg_x, H) if nv else OQ.dequantize_mx(cx[toks], sx[toks])

    # dY2 = float32(probs * dout): row-wise and column-wise, in full; dprobs
    dy32, dprobs_ref = OR.unpermute_bwd(bf16_np(dout), bf16_np(lay.y[:Rp]), rim, probs, Rp)
    assert rel_fro(dprobs_ref, lay.dprobs.cpu().numpy()) <= 1e-5
    dy32_t = np.ascontiguousarray(dy32.T)
    if nv:
        i2, i1 = 2 + 2 * E, 3 + 2 * E
        am = float(np.max(np.abs(dy32)))
        sg_dy2 = OQ.nvfp4_global_scale(am)
        assert float(lay.nv_amax[i2].item()) == am and float(lay.nv_sg[i2].item()) == float(sg_dy2)
        c2, s2 = FP.quantize_rows(dy32, "nv", s_g=float(sg_dy2))
        cc2, cs2 = FP.quantize_rows(dy32_t, "nv", s_g=float(sg_dy2))
        assert np.array_equal(u8_np(lay.dy2col)[:, :Rp // 2], cc2)
        dy2_deq = OQ.dequantize_nvfp4(c2[rr], s2[rr], sg_dy2, H)
    else:
        c2, s2 = FP.quantize_rows(dy32, "mx_e5m2")
        cc2, cs2 = FP.quantize_rows(dy32_t, "mx_e5m2")
        assert np.array_equal(u8_np(lay.dy2col)[:, :Rp], cc2)
        dy2_deq = OQ.dequantize_mx(c2[rr], s2[rr], "e5m2")
    assert np.array_equal(u8_np(lay.dy2q[:Rp]), c2)
    assert np.array_equal(sc(lay.dy2s, R, H)[:Rp], s2)
    assert np.array_equal(sc(lay.dy2cs, H, R)[:, :Rp // blk], cs2)
    del dy32, dy32_t

    # weights: both copies of each in full, the forward GEMMs and the dgrads
    # at the sampled rows against all columns
    def weight_gpu(q, s, qc, scs, N, K):
        return {"codes": u8_np(q), "scales": sc(s, E * N, K).reshape(E, N, K // blk),
                "col_codes": u8_np(qc), "col_scales": sc(scs, E * K, N).reshape(E, K, N // blk)}

    wrec = "nv2d" if nv else "mx"

    def per_expert(wb, slot):
        if not nv:
            return None
        sg = np.array([OQ.nvfp4_global_scale(_amax_bits(wb[e])) for e in range(E)], dtype=np.float32)
        assert np.array_equal(lay.nv_sg[slot:slot + E].cpu().numpy(), sg)
        return {"s_g": sg}

    gu_gpu = bf16_np(_gather(lay.gu, rr))
    h_gpu = bf16_np(_gather(lay.h_bf16, rr))
    check_elementwise(OL.swiglu(gu_gpu, F), h_gpu, "swiglu")
    if nv:
        h_amax = max(_amax_bits(_bits(lay.h_bf16[r0:min(r0 + 32768, Rp)])) for r0 in range(0, Rp, 32768))
        sg_h = OQ.nvfp4_global_scale(h_amax)
        assert float(lay.nv_sg[1].item()) == float(sg_h)
        ch, sh = OQ.quantize_nvfp4(h_gpu, sg_h)
        h_deq = OQ.dequantize_nvfp4(ch, sh, sg_h, F)
    else:
        ch, sh = OQ.quantize_mx(h_gpu)
        h_deq = OQ.dequantize_mx(ch, sh)
    assert np.array_equal(u8_np(_gather(lay.hq, rr)), ch)
    assert np.array_equal(sc(lay.hs, R, F)[rr], sh)

    w2b = _bits(w2)
    tot, fwd2, dgr2 = FP.weight_sweep(w2b, wrec, gpu=weight_gpu(lay.w2q, lay.w2s, lay.w2col, lay.w2cs, H, F),
                                      a_rows=_by_expert(ee, h_deq), dy_rows=_by_expert(ee, dy2_deq), col=True,
                                      per_expert=per_expert(w2b, 2 + E))
    del w2b
    assert all(v == 0 for v in tot.values()) and len(tot) == 4, tot
    _gemm_check(fwd2, bf16_np(_gather(lay.y, rr)), ee, "down fwd")
    dh_gpu = bf16_np(_gather(lay.dh, rr))
    _gemm_check(dgr2, dh_gpu, ee, "down dgrad")

    # dSwiGLU and dY1's row-wise codes on the sampled rows
    dgu_gpu = bf16_np(_gather(lay.dgu_bf16, rr))
    check_elementwise(OL.dswiglu(dh_gpu, gu_gpu, F), dgu_gpu, "dswiglu")
    if nv:
        d_amax = max(_amax_bits(_bits(lay.dgu_bf16[r0:min(r0 + 16384, Rp)])) for r0 in range(0, Rp, 16384))
        sg_dy1 = OQ.nvfp4_global_scale(d_amax)
        assert float(lay.nv_sg[i1].item()) == float(sg_dy1)
        c1, s1 = OQ.quantize_nvfp4(dgu_gpu, sg_dy1)
        dy1_deq = OQ.dequantize_nvfp4(c1, s1, sg_dy1, 2 * F)
    else:
        c1, s1 = OQ.quantize_mx(dgu_gpu, "e5m2")
        dy1_deq = OQ.dequantize_mx(c1, s1, "e5m2")
    assert np.array_equal(u8_np(_gather(lay.dy1q, rr)), c1)
    assert np.array_equal(sc(lay.dy1s, R, 2 * F)[rr], s1)

    w1b = _bits(w1)
    tot, fwd1, dgr1 = FP.weight_sweep(w1b, wrec, gpu=weight_gpu(lay.w1q, lay.w1s, lay.w1col, lay.w1cs, 2 * F, H),
                                      a_rows=_by_expert(ee, x_deq), dy_rows=_by_expert(ee, dy1_deq), col=True,
                                      per_expert=per_expert(w1b, 2))
    del w1b
    assert all(v == 0 for v in tot.values()) and len(tot) == 4, tot
    _gemm_check(fwd1, gu_gpu, ee, "gate/up fwd")
    _gemm_check(dgr1, bf16_np(_gather(lay.dxp, rr)), ee, "gate/up dgrad")

    check_elementwise(OR.unpermute(bf16_np(lay.y[:Rp]), rim, probs), bf16_np(lay.out), "unpermute")
    check_elementwise(OR.permute_bwd(bf16_np(lay.dxp[:Rp]), rim), bf16_np(lay.dx), "permute_bwd")

    # wgrads at 16 x 16 sampled (n, k) of every expert, from the column-wise
    # copies (dequantised over the rows in use)
    def col_deq(codes, scales, s_g, fmt):
        if nv:
            return OQ.dequantize_nvfp4(codes[:, :Rp // 2], scales[:, :Rp // 16], s_g, Rp)
        return OQ.dequantize_mx(codes[:, :Rp], scales[:, :Rp // 32], fmt)

    ns2, ks2 = np.sort(rng.choice(H, 16, replace=False)), np.sort(rng.choice(F, 16, replace=False))
    ns1, ks1 = np.sort(rng.choice(2 * F, 16, replace=False)), np.sort(rng.choice(H, 16, replace=False))
    sel = lambda t, idx_: t[torch.from_numpy(idx_).to(DEV)]                     # noqa: E731
    # the column-wise dY2 (checked in full above) and X; h's and dY1's column
    # copies were cast from the GPU's bf16 h / dG | dU: requantised here from
    # those columns and compared first
    dy2c = col_deq(cc2[ns2], cs2[ns2], float(sg_dy2) if nv else None, "e5m2")
    xc = col_deq(ccx[ks1], csx[ks1], float(sg_x) if nv else None, "e4m3")
    h_cols_bits = np.ascontiguousarray(_bits(lay.h_bf16[:Rp][:, torch.from_numpy(ks2).to(DEV)]).T)
    d_cols_bits = np.ascontiguousarray(_bits(lay.dgu_bf16[:Rp][:, torch.from_numpy(ns1).to(DEV)]).T)
    if nv:
        hc_c, hc_s = OQ.quantize_nvfp4(OF.bf16_bits_to_f64(h_cols_bits), sg_h)
        dc_c, dc_s = OQ.quantize_nvfp4(OF.bf16_bits_to_f64(d_cols_bits), sg_dy1)
        assert np.array_equal(u8_np(sel(lay.hcol, ks2))[:, :Rp // 2], hc_c)
        assert np.array_equal(u8_np(sel(lay.dy1col, ns1))[:, :Rp // 2], dc_c)
    else:
        hc_c, hc_s = OQ.quantize_mx(OF.bf16_bits_to_f64(h_cols_bits))
        dc_c, dc_s = OQ.quantize_mx(OF.bf16_bits_to_f64(d_cols_bits), "e5m2")
        assert np.array_equal(u8_np(sel(lay.hcol, ks2))[:, :Rp], hc_c)
        assert np.array_equal(u8_np(sel(lay.dy1col, ns1))[:, :Rp], dc_c)
    assert np.array_equal(sc(lay.hcs, F, R)[ks2][:, :Rp // blk], hc_s)
    assert np.array_equal(sc(lay.dy1cs, 2 * F, R)[ns1][:, :Rp // blk], dc_s)
    hc = OQ.dequantize_nvfp4(hc_c, hc_s, sg_h, Rp) if nv else OQ.dequantize_mx(hc_c, hc_s)
    dc = OQ.dequantize_nvfp4(dc_c, dc_s, sg_dy1, Rp) if nv else OQ.dequantize_mx(dc_c, dc_s, "e5m2")
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        _wgrad_samples(lay.dw2, e, ns2, ks2, dy2c[:, lo:hi].T, hc[:, lo:hi].T)
        _wgrad_samples(lay.dw1, e, ns1, ks1, dc[:, lo:hi].T, xc[:, lo:hi].T)


def test_blockwise_training_step_full_size():
    """The Scout-shaped experts trained with blockwise FP8 at full size (1x128
    row blocks and 128x1 column blocks of activations and gradients, 128x128
    weight tiles; e4m3 forward, e5m2 gradients; Zipf loads with two empty
    experts, top-1). Both copies of X and dY2 in full, both copies of every
    weight in full, the forward GEMMs and the dgrads at the sampled rows
    against all columns, h's and dY1's codes on the sampled rows and their
    column copies on sampled columns, and sampled wgrad elements of every
    expert from the column-wise copies."""
    w, lay, x, idx, probs, dout, w1, w2, _, _ = _train_layer("scout_fwdbwd", 0)
    E, H, F, k = w.E, w.H, w.F, w.k
    rng = np.random.default_rng(13)
    rim, src, off, cnt, Rp = _routing(lay, idx, E)
    assert np.sum(cnt == 0) >= 1
    filler = src < 0

    def rows_si(buf):                      # row-wise scale_inv [C/128][R_cap] -> [R_cap, C/128]
        return buf.cpu().numpy().T

    def cols_si(buf, cols=None):           # column-wise [R_cap/128][C] -> [C, Rp/128]
        a = buf.cpu().numpy()[:Rp // 128]
        return (a if cols is None else a[:, cols]).T

    # X: every routed row; the column-wise copy ([H, R_cap], 128x1 blocks along
    # each group's tokens) in full
    xb = _bits(x)
    cx, sx = FP.quantize_rows(xb, "blk")
    _check_permuted(u8_np(lay.xq), rows_si(lay.xs), cx, sx, rim, Rp, "X")
    xperm_t = np.ascontiguousarray(OR.permute_rows(xb, rim, Rp).T)      # bf16 bits [H, Rp], filler rows 0
    ccx, csx = FP.quantize_rows(xperm_t, "blk")
    del xperm_t
    assert np.array_equal(u8_np(lay.xcol)[:, :Rp], ccx)
    assert np.array_equal(cols_si(lay.xcs), csx)
    ee, rr = _sample_rows(off, cnt, rng)
    toks = src[rr] // k
    x_deq = OQ.dequantize_block_1x128(cx[toks], sx[toks])

    # dY2 = float32(probs * dout): both copies in full; dprobs
    dy32, dprobs_ref = OR.unpermute_bwd(bf16_np(dout), bf16_np(lay.y[:Rp]), rim, probs, Rp)
    assert rel_fro(dprobs_ref, lay.dprobs.cpu().numpy()) <= 1e-5
    c2, s2 = FP.quantize_rows(dy32, "blk_e5m2")
    assert np.array_equal(u8_np(lay.dy2q[:Rp]), c2)
    s2z = s2.copy()
    s2z[filler] = 0.0
    assert np.array_equal(rows_si(lay.dy2s)[:Rp], s2z)
    cc2, cs2 = FP.quantize_rows(np.ascontiguousarray(dy32.T), "blk_e5m2")
    assert np.array_equal(u8_np(lay.dy2col)[:, :Rp], cc2)
    assert np.array_equal(cols_si(lay.dy2cs), cs2)
    dy2_deq = OQ.dequantize_block_1x128(c2[rr], s2[rr], "e5m2")
    del dy32

    def weight_gpu(q, s, qc, scs):
        return {"codes": u8_np(q), "scales": s.cpu().numpy(), "col_codes": u8_np(qc), "col_scales": scs.cpu().numpy()}

    # forward: gate/up rows, SwiGLU, h's row codes on the sampled rows
    gu_gpu = bf16_np(_gather(lay.gu, rr))
    h_gpu = bf16_np(_gather(lay.h_bf16, rr))
    check_elementwise(OL.swiglu(gu_gpu, F), h_gpu, "swiglu")
    ch, sh = OQ.quantize_block_1x128(h_gpu)
    assert np.array_equal(u8_np(_gather(lay.hq, rr)), ch)
    assert np.array_equal(rows_si(lay.hs)[rr], sh)
    h_deq = OQ.dequantize_block_1x128(ch, sh)

    # W2 in full (both copies): down forward (all H columns) and down dgrad
    # through the column copy (all F columns) at the sampled rows
    w2b = _bits(w2)
    tot, fwd2, dgr2 = FP.weight_sweep(w2b, "blk", gpu=weight_gpu(lay.w2q, lay.w2s, lay.w2col, lay.w2cs),
                                      a_rows=_by_expert(ee, h_deq), dy_rows=_by_expert(ee, dy2_deq), col=True)
    del w2b
    assert all(v == 0 for v in tot.values()) and len(tot) == 4, tot
    _gemm_check(fwd2, bf16_np(_gather(lay.y, rr)), ee, "down fwd")
    dh_gpu = bf16_np(_gather(lay.dh, rr))
    _gemm_check(dgr2, dh_gpu, ee, "down dgrad")

    # dSwiGLU and dY1's row codes on the sampled rows
    dgu_gpu = bf16_np(_gather(lay.dgu_bf16, rr))
    check_elementwise(OL.dswiglu(dh_gpu, gu_gpu, F), dgu_gpu, "dswiglu")
    c1, s1 = OQ.quantize_block_1x128(dgu_gpu, "e5m2")
    assert np.array_equal(u8_np(_gather(lay.dy1q, rr)), c1)
    assert np.array_equal(rows_si(lay.dy1s)[rr], s1)
    dy1_deq = OQ.dequantize_block_1x128(c1, s1, "e5m2")

    # W1 in full (both copies): gate/up forward and gate/up dgrad
    w1b = _bits(w1)
    tot, fwd1, dgr1 = FP.weight_sweep(w1b, "blk", gpu=weight_gpu(lay.w1q, lay.w1s, lay.w1col, lay.w1cs),
                                      a_rows=_by_expert(ee, x_deq), dy_rows=_by_expert(ee, dy1_deq), col=True)
    del w1b
    assert all(v == 0 for v in tot.values()) and len(tot) == 4, tot
    _gemm_check(fwd1, gu_gpu, ee, "gate/up fwd")
    _gemm_check(dgr1, bf16_np(_gather(lay.dxp, rr)), ee, "gate/up dgrad")

    check_elementwise(OR.unpermute(bf16_np(lay.y[:Rp]), rim, probs), bf16_np(lay.out), "unpermute")
    check_elementwise(OR.permute_bwd(bf16_np(lay.dxp[:Rp]), rim), bf16_np(lay.dx), "permute_bwd")

    # wgrads at 16 x 16 sampled (n, k) of every expert from the column-wise
    # copies: dY2's and X's checked in full above; h's and dY1's requantised
    # here from the GPU's bf16 columns and compared first
    ns2, ks2 = np.sort(rng.choice(H, 16, replace=False)), np.sort(rng.choice(F, 16, replace=False))
    ns1, ks1 = np.sort(rng.choice(2 * F, 16, replace=False)), np.sort(rng.choice(H, 16, replace=False))
    sel = lambda t, idx_: t[torch.from_numpy(idx_).to(DEV)]                     # noqa: E731
    dy2c = OQ.dequantize_block_1x128(cc2[ns2], cs2[ns2], "e5m2")
    xc = OQ.dequantize_block_1x128(ccx[ks1], csx[ks1])
    h_cols = OF.bf16_bits_to_f64(np.ascontiguousarray(_bits(lay.h_bf16[:Rp][:, torch.from_numpy(ks2).to(DEV)]).T))
    d_cols = OF.bf16_bits_to_f64(np.ascontiguousarray(_bits(lay.dgu_bf16[:Rp][:, torch.from_numpy(ns1).to(DEV)]).T))
    hc_c, hc_s = OQ.quantize_block_1x128(h_cols)
    dc_c, dc_s = OQ.quantize_block_1x128(d_cols, "e5m2")
    assert np.array_equal(u8_np(sel(lay.hcol, ks2))[:, :Rp], hc_c)
    assert np.array_equal(u8_np(sel(lay.dy1col, ns1))[:, :Rp], dc_c)
    assert np.array_equal(cols_si(lay.hcs, ks2), hc_s)
    assert np.array_equal(cols_si(lay.dy1cs, ns1), dc_s)
    hc = OQ.dequantize_block_1x128(hc_c, hc_s)
    dc = OQ.dequantize_block_1x128(dc_c, dc_s, "e5m2")
    dw1, dw2 = lay.dw1, lay.dw2
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            # empty expert: zero weight gradients
            assert float(dw1[e].abs().max()) == 0.0 and float(dw2[e].abs().max()) == 0.0
            continue
        _wgrad_samples(dw2, e, ns2, ks2, dy2c[:, lo:hi].T, hc[:, lo:hi].T)
        _wgrad_samples(dw1, e, ns1, ks1, dc[:, lo:hi].T, xc[:, lo:hi].T)

"""Helpers shared by the GPU parity tests, smoke() and bench: run pieces of the
CUDA path through the C ABI and compare them with the CPU oracle on the same
inputs.

Tolerances (written here, used by every GPU test):
* codes, scales and index arrays: bit-exact;
* grouped GEMM outputs: relative Frobenius error <= 2e-3 against the oracle's
  float64 result on the same quantised inputs, rounded to the output dtype
  (bf16 rounding alone costs about 1.7e-3 of that budget); float32 outputs
  <= 1e-5 against the unrounded float64 result;
* elementwise float steps (SwiGLU, combine, ...): relative Frobenius <= 1e-3
  and at most 1 bf16 ulp on >= 99.99% of the elements.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import formats as OF
from oracle import gemm as OG
from oracle import layer as OL
from oracle import quant as OQ
from oracle import routing as OR

GEMM_TOL_BF16 = 2e-3
GEMM_TOL_F32 = 1e-5
ELEM_TOL = 1e-3


def untile_mx_scales(buf, rows: int, ld: int, block: int = 32) -> np.ndarray:
    """The 128x4-tiled scale bytes of a [rows, ld] matrix -> natural
    [rows, ld/block] (layout documented in include/mgq.h)."""
    b = np.asarray(buf).reshape(-1)
    kb = ld // block
    rp = (rows + 127) // 128 * 128
    t = b[: rp * kb].reshape(rp // 128, kb // 4, 32, 4, 4)
    return t.transpose(0, 3, 2, 1, 4).reshape(rp, kb)[:rows]


def tile_mx_scales(nat: np.ndarray) -> np.ndarray:
    """Inverse of untile_mx_scales (rows padded to 128 with zero bytes)."""
    rows, kb = nat.shape
    rp = (rows + 127) // 128 * 128
    full = np.zeros((rp, kb), dtype=np.uint8)
    full[:rows] = nat
    t = full.reshape(rp // 128, 4, 32, kb // 4, 4)      # [rt, q, i, kg, bb]
    return np.ascontiguousarray(t.transpose(0, 3, 2, 1, 4)).reshape(-1)


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def u8_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def rel_fro(ref, got) -> float:
    return OG.rel_frobenius(ref, got)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    return np.exp2(np.maximum(e - 8, -133).astype(np.float64))


def check_elementwise(ref: np.ndarray, got: np.ndarray, what: str):
    """ref: oracle float64 (unrounded); got: GPU bf16 values (float64).
    Compared with the oracle rounded to bf16: at most 1 bf16 ulp apart on
    >= 99.99% of the elements and relative Frobenius <= 1e-3."""
    refr = OF.round_to_bf16(ref)
    rf = rel_fro(refr, got)
    ulp = np.maximum(ulp_bf16(refr), ulp_bf16(got))
    bad = np.abs(got - refr) > ulp * 1.0000001
    frac = float(np.mean(bad)) if bad.size else 0.0
    assert rf <= ELEM_TOL, f"{what}: rel Frobenius {rf:.3e}"
    assert frac <= 1e-4, f"{what}: {frac:.2e} of elements beyond 1 bf16 ulp"
    return rf


def _q_rows(x, recipe):
    """Oracle row-wise quantisation of activations: (codes, scales, dequantised)."""
    if recipe == "nvfp4":
        sg = OQ.nvfp4_global_scale(np.max(np.abs(x)) if x.size else 0.0)
        c, s = OQ.quantize_nvfp4(x, sg)
        return c, s, OQ.dequantize_nvfp4(c, s, sg, x.shape[1])
    if recipe == "mxfp8":
        c, s = OQ.quantize_mx(x, "e4m3")
        return c, s, OQ.dequantize_mx(c, s)
    c, s = OQ.quantize_block_1x128(x, "e4m3")
    return c, s, OQ.dequantize_block_1x128(c, s)


def _q_weight(w, recipe):
    if recipe == "nvfp4":
        return _q_rows(w, recipe)
    if recipe == "mxfp8":
        c, s = OQ.quantize_mx(w, "e4m3")
        return c, s, OQ.dequantize_mx(c, s)
    c, s = OQ.quantize_block_128x128(w, "e4m3")
    return c, s, OQ.dequantize_block_128x128(c, s)


def _gpu_row_scales(lay, buf, rows_cap, ld, recipe):
    if recipe == "nvfp4":
        return untile_mx_scales(u8_np(buf), rows_cap, ld, block=16)
    if recipe == "mxfp8":
        return untile_mx_scales(u8_np(buf), rows_cap, ld)
    return buf.detach().cpu().numpy().T          # [K/128][R_cap] -> [R_cap, K/128]


def run_fwd_and_check(w, device, recipe: str = "mxfp8", **layer_kw) -> dict:
    """One forward of workload ``w`` through ExpertLayer (MXFP8 or blockwise
    FP8), every step compared with the oracle. Returns the measured errors."""
    from fp8_grouped_gemm_gb300 import layer as L
    from fp8_grouped_gemm_gb300 import workloads as W
    from fp8_grouped_gemm_gb300 import mgq

    x = W.make_activations(w)
    w1, w2 = W.make_weights(w)
    idx, probs = W.make_routing(w)
    lay = L.ExpertLayer(w, device, recipe=recipe, keep_bf16=True, **layer_kw)
    xd, w1d, w2d = x.to(device), w1.to(device), w2.to(device)
    idxd = torch.from_numpy(idx).to(device)
    pd = torch.from_numpy(probs).to(device)
    lay.quantize_weights(w1d, w2d)
    lay.forward(xd, idxd, pd)
    torch.cuda.synchronize()
    assert mgq.get_error() == mgq.OK
    res = {}
    E, H, F = w.E, w.H, w.F
    # routing: bit-exact
    rim, src, off, cnt = OR.permute_indices(idx, E, L.ALIGN)
    Rp = int(off[-1])
    assert np.array_equal(lay.offsets.cpu().numpy(), off)
    assert np.array_equal(lay.counts.cpu().numpy(), cnt)
    assert np.array_equal(lay.row_id_map.cpu().numpy(), rim)
    assert np.array_equal(lay.src_row.cpu().numpy()[:Rp], src)
    # permute + quantise: bit-exact codes and scales (filler rows zero)
    xf = W.bf16_to_f64(x)
    cx, sx, _ = _q_rows(xf, recipe)
    want_c = OR.permute_rows(cx, rim, Rp)
    want_s = OR.permute_rows(sx, rim, Rp)
    assert np.array_equal(u8_np(lay.xq)[:Rp], want_c)
    assert np.array_equal(_gpu_row_scales(lay, lay.xs, lay.R_cap, H, recipe)[:Rp], want_s)
    # weights: bit-exact
    w1f, w2f = W.bf16_to_f64(w1), W.bf16_to_f64(w2)
    if recipe == "mxfp8":
        cw1, sw1, dw1 = _q_weight(w1f.reshape(E * 2 * F, H), recipe)
        cw2, sw2, dw2 = _q_weight(w2f.reshape(E * H, F), recipe)
        assert np.array_equal(untile_mx_scales(u8_np(lay.w1s), E * 2 * F, H), sw1)
        assert np.array_equal(untile_mx_scales(u8_np(lay.w2s), E * H, F), sw2)
    elif recipe == "nvfp4":
        q1 = [_q_weight(w1f[e], recipe) for e in range(E)]
        q2 = [_q_weight(w2f[e], recipe) for e in range(E)]
        cw1 = np.concatenate([q[0] for q in q1]); dw1 = np.concatenate([q[2] for q in q1])
        cw2 = np.concatenate([q[0] for q in q2]); dw2 = np.concatenate([q[2] for q in q2])
        assert np.array_equal(untile_mx_scales(u8_np(lay.w1s), E * 2 * F, H, 16), np.concatenate([q[1] for q in q1]))
        assert np.array_equal(untile_mx_scales(u8_np(lay.w2s), E * H, F, 16), np.concatenate([q[1] for q in q2]))
        sgs = [OQ.nvfp4_global_scale(np.max(np.abs(w1f[e]))) for e in range(E)] + \
              [OQ.nvfp4_global_scale(np.max(np.abs(w2f[e]))) for e in range(E)]
        assert np.array_equal(lay.nv_sg.cpu().numpy()[2:2 + 2 * E], np.array(sgs, dtype=np.float32))
    else:
        q1 = [_q_weight(w1f[e], recipe) for e in range(E)]
        q2 = [_q_weight(w2f[e], recipe) for e in range(E)]
        cw1 = np.concatenate([q[0] for q in q1]); dw1 = np.concatenate([q[2] for q in q1])
        cw2 = np.concatenate([q[0] for q in q2]); dw2 = np.concatenate([q[2] for q in q2])
        assert np.array_equal(lay.w1s.cpu().numpy(), np.stack([q[1] for q in q1]))
        assert np.array_equal(lay.w2s.cpu().numpy(), np.stack([q[1] for q in q2]))
    assert np.array_equal(u8_np(lay.w1q).reshape(E * 2 * F, -1), cw1)
    assert np.array_equal(u8_np(lay.w2q).reshape(E * H, -1), cw2)
    # gate/up GEMM on the identical quantised inputs
    a_deq = _q_rows(xf, recipe)[2]
    a_deq = OR.permute_rows(a_deq, rim, Rp, fill=0.0)
    gu_ref = OG.grouped_gemm_fwd(a_deq, dw1.reshape(E, 2 * F, H), off)
    gu = bf16_np(lay.gu)[:Rp]
    res["gemm1_relfro"] = rel_fro(OF.round_to_bf16(gu_ref), gu)
    res["gemm1_sqnr_vs_bf16"] = OG.sqnr_db(
        OG.grouped_gemm_fwd(OR.permute_rows(xf, rim, Rp), w1f, off), gu)
    assert res["gemm1_relfro"] <= GEMM_TOL_BF16, res
    # SwiGLU on the GPU's gate/up output; codes from the GPU-materialised h
    h_gpu = bf16_np(lay.h_bf16)[:Rp]
    res["swiglu_relfro"] = check_elementwise(OL.swiglu(gu, F), h_gpu, "swiglu")
    ch, sh, hdq = _q_rows(h_gpu, recipe)
    assert np.array_equal(u8_np(lay.hq)[:Rp], ch)
    assert np.array_equal(_gpu_row_scales(lay, lay.hs, lay.R_cap, F, recipe)[:Rp], sh)
    # down GEMM
    y_ref = OG.grouped_gemm_fwd(hdq, dw2.reshape(E, H, F), off)
    y = bf16_np(lay.y)[:Rp]
    res["gemm2_relfro"] = rel_fro(OF.round_to_bf16(y_ref), y)
    assert res["gemm2_relfro"] <= GEMM_TOL_BF16, res
    # unpermute on the GPU's y
    out_ref = OR.unpermute(y, rim, probs)
    res["unpermute_relfro"] = check_elementwise(out_ref, bf16_np(lay.out), "unpermute")
    return res

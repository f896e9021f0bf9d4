"""The worker pool of the full-size parity tests (CPU only): on small arrays
its sweeps equal direct calls of the oracle, count planted mismatches, and
assemble the sampled-row products in the right places."""
import numpy as np
import pytest

from oracle import formats as OF
from oracle import quant as OQ
from tests import fullsize_pool as FP


def _bits(x):
    return OF.f64_to_bf16_bits(OF.round_to_bf16(x)).astype(np.uint16)


@pytest.mark.parametrize("recipe", ["mx", "blk", "nv", "nv2d", "tensor"])
def test_weight_sweep_equals_direct_oracle(recipe):
    rng = np.random.default_rng(0)
    E, N, K = 2, 256, 256
    wb = _bits(rng.standard_normal((E, N, K)) * 0.02)
    w = OF.bf16_bits_to_f64(wb)
    a = {e: rng.standard_normal((5, K)) for e in range(E)}
    dy = {e: rng.standard_normal((5, N)) for e in range(E)}
    per = {}
    gpu = {}
    deq, deq_col = [], []
    for e in range(E):
        if recipe == "mx":
            c, s = OQ.quantize_mx(w[e])
            cc, cs = OQ.quantize_mx(np.ascontiguousarray(w[e].T))
            deq.append(OQ.dequantize_mx(c, s))
            deq_col.append(OQ.dequantize_mx(cc, cs))
            gpu.setdefault("codes", []).append(c)
            gpu.setdefault("scales", []).append(s)
            gpu.setdefault("col_codes", []).append(cc)
            gpu.setdefault("col_scales", []).append(cs)
        elif recipe == "blk":
            c, si = OQ.quantize_block_128x128(w[e])
            cc, cs = OQ.quantize_block_128x128(np.ascontiguousarray(w[e].T))
            deq.append(OQ.dequantize_block_128x128(c, si))
            deq_col.append(OQ.dequantize_block_128x128(cc, cs))
            for key, v in (("codes", c), ("scales", si), ("col_codes", cc), ("col_scales", cs)):
                gpu.setdefault(key, []).append(v)
        elif recipe in ("nv", "nv2d"):
            sg = OQ.nvfp4_global_scale(float(np.max(np.abs(w[e]))))
            per.setdefault("s_g", []).append(float(sg))
            if recipe == "nv":
                c, s = OQ.quantize_nvfp4(w[e], sg)
                deq.append(OQ.dequantize_nvfp4(c, s, sg, K))
                gpu.setdefault("codes", []).append(c)
                gpu.setdefault("scales", []).append(s)
            else:
                rc, rs, cc, cs = OQ.quantize_nvfp4_2d(w[e], sg)
                deq.append(OQ.dequantize_nvfp4(rc, rs, sg, K))
                deq_col.append(OQ.dequantize_nvfp4(cc, cs, sg, N))
                for key, v in (("codes", rc), ("scales", rs), ("col_codes", cc), ("col_scales", cs)):
                    gpu.setdefault(key, []).append(v)
        else:
            sc = np.float32(448.0 / np.max(np.abs(w[e])))
            per.setdefault("scale", []).append(float(sc))
            c, _ = OQ.quantize_tensor(w[e], sc)
            deq.append(OQ.dequantize_tensor(c, sc))
            gpu.setdefault("codes", []).append(c)
    gpu = {k: np.stack(v) for k, v in gpu.items()}
    # plant one wrong byte in the GPU codes of expert 1
    gpu["codes"][1, 3, 5] ^= 1
    tot, fwd, dgrad = FP.weight_sweep(wb, recipe, gpu=gpu, a_rows=a, dy_rows=dy, chunk=128,
                                      col=(recipe in ("mx", "blk")), per_expert={k: np.array(v) for k, v in per.items()})
    assert tot["codes"] == 1
    assert all(v == 0 for k, v in tot.items() if k != "codes")
    for e in range(E):
        np.testing.assert_allclose(fwd[e], a[e] @ deq[e].T, rtol=1e-12, atol=1e-12)
        wcol = deq_col[e] if deq_col else deq[e].T                    # [K, N]
        np.testing.assert_allclose(dgrad[e], dy[e] @ wcol.T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("recipe", ["mx", "mx_e5m2", "blk", "blk_e5m2", "nv", "tensor_e5m2"])
def test_quantize_rows_equals_direct_oracle(recipe):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((300, 256))
    xb = _bits(x)
    xf = OF.bf16_bits_to_f64(xb)
    kw = {"s_g": 100.0} if recipe == "nv" else ({"scale": 3.0} if recipe.startswith("tensor") else {})
    c, s = FP.quantize_rows(xb, recipe, chunk=64, **kw)
    if recipe in ("mx", "mx_e5m2"):
        wc, ws = OQ.quantize_mx(xf, "e5m2" if recipe == "mx_e5m2" else "e4m3")
    elif recipe in ("blk", "blk_e5m2"):
        wc, ws = OQ.quantize_block_1x128(xf, "e5m2" if recipe == "blk_e5m2" else "e4m3")
    elif recipe == "nv":
        wc, ws = OQ.quantize_nvfp4(xf, np.float32(100.0))
    else:
        wc, ws = OQ.quantize_tensor(xf, np.float32(3.0), "e5m2")[0], None
    np.testing.assert_array_equal(c, wc)
    if ws is None:
        assert s is None
    else:
        np.testing.assert_array_equal(s, ws)
    # float32 inputs (dY = probs * dout) go through unchanged
    x32 = xf.astype(np.float32) * np.float32(0.37)
    c32, _ = FP.quantize_rows(x32, "tensor_e5m2", chunk=100, scale=3.0)
    np.testing.assert_array_equal(c32, OQ.quantize_tensor(x32.astype(np.float64), np.float32(3.0), "e5m2")[0])

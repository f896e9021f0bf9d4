"""Host-side wiring of ExpertLayer (no GPU): which steps each recipe fuses,
the order of the calls of a step, and the kernel launches per step that
bench.py reports (the training counts are those of the ncu launch lists of
the three Mixtral-shaped training steps); and the binding's buffer-size
helpers. The layer is built over CPU tensors; building the op list issues no
call."""
import pytest
import torch

from fp8_grouped_gemm_gb300 import layer as L
from fp8_grouped_gemm_gb300 import workloads as W

FWD = ["weight_quant", "weight_quant", "route", "permute_quant"]

CASES = {
    # workload: (recipe, train, ops after the weights / routing / permute, launches per step)
    "mixtral_fwdbwd": ("delayed", True,
                       ["gemm_fwd_gateup_swiglu", "gemm_fwd_down", "unpermute", "unpermute_bwd_quant",
                        "gemm_dgrad_down_dswiglu", "gemm_wgrad_down", "gemm_dgrad_gateup", "gemm_wgrad_gateup",
                        "permute_bwd", "scaling_update"], 17),
    "mixtral_fwdbwd_mx": ("mxfp8", True,
                          ["gemm_fwd_gateup_swiglu", "gemm_fwd_down", "unpermute", "unpermute_bwd_quant",
                           "gemm_dgrad_down", "gemm_wgrad_down", "dswiglu_quant", "gemm_dgrad_gateup",
                           "gemm_wgrad_gateup", "permute_bwd"], 17),
    "mixtral_fwdbwd_nvfp4": ("nvfp4", True,
                             ["gemm_fwd_gateup_swiglu", "gemm_fwd_down", "unpermute", "unpermute_bwd_quant",
                              "gemm_dgrad_down", "gemm_wgrad_down", "dswiglu_quant", "gemm_dgrad_gateup",
                              "gemm_wgrad_gateup", "permute_bwd"], 23),
    "scout_fwdbwd": ("blockwise", True,
                     ["gemm_fwd_gateup", "swiglu_quant", "gemm_fwd_down", "unpermute", "unpermute_bwd_quant",
                      "gemm_dgrad_down", "gemm_wgrad_down", "dswiglu_quant", "gemm_dgrad_gateup",
                      "gemm_wgrad_gateup", "permute_bwd"], 18),
    "mixtral_fwd": ("mxfp8", False, ["gemm_fwd_gateup_swiglu", "gemm_fwd_down", "unpermute"], 9),
    "scout_fwd": ("blockwise", False, ["gemm_fwd_gateup", "swiglu_quant", "gemm_fwd_down", "unpermute"], 10),
    "finegrained_fwd": ("nvfp4", False, ["gemm_fwd_gateup_swiglu", "gemm_fwd_down", "unpermute"], 14),
}


def _layer_and_ops(name, **kw):
    w = W.WORKLOADS[name].scaled(T=256, H=256, F=512, E=4)
    lay = L.ExpertLayer(w, "cpu", **kw)
    E, H, F, T, k = w.E, w.H, w.F, w.T, w.k
    bf = dict(dtype=torch.bfloat16)
    ops = lay.step_ops(torch.zeros(E, 2 * F, H, **bf), torch.zeros(E, H, F, **bf), torch.zeros(T, H, **bf),
                       torch.zeros(T, k, dtype=torch.int32), torch.zeros(T, k),
                       torch.zeros(T, H, **bf) if lay.train else None)
    return lay, [n for n, _ in ops]


@pytest.mark.parametrize("name", sorted(CASES))
def test_step_wiring_and_launch_count(name):
    recipe, train, rest, launches = CASES[name]
    lay, names = _layer_and_ops(name)
    assert (lay.recipe, lay.train) == (recipe, train)
    assert names == FWD + rest
    assert lay.gpu_launches_per_step() == launches


def test_explicit_column_copies_unfuse_the_delayed_epilogues():
    """Per-tensor with explicit column-wise copies: the SwiGLU / dSwiGLU
    epilogues write row-wise codes only, so the separate passes come back,
    with the column copies of X and dY2 as two more launches."""
    lay, names = _layer_and_ops("mixtral_fwdbwd", col_copies=True)
    assert not lay.mn and not lay.fused_swiglu
    assert "swiglu_quant" in names and "dswiglu_quant" in names
    assert "gemm_fwd_gateup_swiglu" not in names and "gemm_dgrad_down_dswiglu" not in names
    assert lay.gpu_launches_per_step() == 17 + 2 + 2


def test_unfused_mx_training_has_the_separate_swiglu_pass():
    lay, names = _layer_and_ops("mixtral_fwdbwd_mx", fuse_swiglu=False)
    assert names[4:6] == ["gemm_fwd_gateup", "swiglu_quant"]
    assert lay.gpu_launches_per_step() == 18


@pytest.mark.parametrize("name", ["mixtral_fwdbwd_nvfp4", "finegrained_fwd"])
def test_nvfp4_scale_images_follow_their_quantisers(name):
    """NVFP4 GEMMs whose contraction reaches the threshold read the scale image
    of their second operand; its op follows the quantiser that writes the
    scales: the weights (training: also their column-wise copies), the column
    copy of x after the permute and that of h after the gate/up GEMM. (The
    scaled-down shapes above stay below the default threshold.)"""
    recipe, train, rest, launches = CASES[name]
    lay, names = _layer_and_ops(name, nv_image_min_k=0)
    n_img = 6 if train else 2
    head = ["weight_quant", "weight_quant"] + ["scale_image"] * (4 if train else 2) + ["route", "permute_quant"]
    if train:
        head += ["scale_image"]
        rest = rest[:1] + ["scale_image"] + rest[1:]
    assert names == head + rest
    assert lay.gpu_launches_per_step() == launches + n_img


def test_nvfp4_training_pads_groups_to_256_rows():
    lay, _ = _layer_and_ops("mixtral_fwdbwd_nvfp4")
    assert lay.align == L.ALIGN_NV_TRAIN == 256 and lay.R_cap % 256 == 0


def test_buffer_sizes_bound_the_layouts():
    """The binding's size helpers: r_cap holds the oracle's padded group layout
    in the worst case, and the tiled-scale byte counts equal the length of the
    128x4 tiling of [rows, ld / block] scales."""
    import numpy as np
    from fp8_grouped_gemm_gb300 import mgq
    from oracle import routing as OR
    from tests.layer_check import tile_mx_scales
    rng = np.random.default_rng(5)
    for T, E, k, align in [(1000, 8, 2, 128), (37, 16, 1, 32), (4096, 128, 8, 128), (5, 4, 4, 256)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        _, _, off, _ = OR.permute_indices(idx, E, align)
        rc = mgq.r_cap(T, k, E, align)
        assert int(off[-1]) <= rc and rc % 128 == 0 and rc - (T * k + E * (align - 1)) < 128
    for rows, ld in [(128, 128), (300, 512), (4096, 4096)]:
        assert mgq.mx_scale_bytes(rows, ld) == tile_mx_scales(np.zeros((rows, ld // 32), np.uint8)).size
        assert mgq.nv_scale_bytes(rows, ld) == tile_mx_scales(np.zeros((rows, ld // 16), np.uint8)).size

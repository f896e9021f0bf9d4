"""The routed-expert layer as a sequence of libmgq calls.

``ExpertLayer`` owns the device buffers of one workload (allocated once with
PyTorch) and issues the C-ABI calls of a forward step and, for the delayed
per-tensor recipe, of the backward step:

forward:  moe_permute (+ quantise) -> grouped_gemm_fwd (gate/up) ->
          swiglu_quantize -> grouped_gemm_fwd (down) -> moe_unpermute
backward: moe_unpermute_bwd (+ quantise dY, dprobs) -> grouped_gemm_dgrad and
          grouped_gemm_wgrad (down) -> dswiglu_quantize -> grouped_gemm_dgrad
          and grouped_gemm_wgrad (gate/up) -> moe_permute_bwd
then:     amax_history_update (delayed scaling)

Every step runs in the library's kernels; this module only allocates buffers
and passes pointers.
"""
from __future__ import annotations

import torch

from . import mgq
from .workloads import Workload

ALIGN = 128       # group padding: the grouped GEMM tiles rows by 128


class ExpertLayer:
    def __init__(self, w: Workload, device, recipe: str | None = None, keep_bf16: bool = False,
                 history: int = 1024):
        self.w = w
        self.dev = torch.device(device)
        self.recipe = recipe or w.recipe
        if self.recipe not in ("mxfp8", "delayed", "blockwise", "nvfp4"):
            raise NotImplementedError(self.recipe)
        self.train = self.recipe == "delayed"
        self.scaling = {"mxfp8": mgq.MX32_E8M0, "delayed": mgq.TENSOR_F32,
                        "blockwise": mgq.BLK_1x128_F32, "nvfp4": mgq.NV16_UE4M3}[self.recipe]
        self.nv = self.recipe == "nvfp4"
        E, k, T, H, F = w.E, w.k, w.T, w.H, w.F
        self.R_cap = mgq.r_cap(T, k, E, ALIGN)
        R = self.R_cap
        d = self.dev
        u8 = dict(dtype=torch.uint8, device=d)
        i32 = dict(dtype=torch.int32, device=d)
        bf = dict(dtype=torch.bfloat16, device=d)
        f32 = dict(dtype=torch.float32, device=d)
        mx = self.scaling == mgq.MX32_E8M0
        blk = self.scaling == mgq.BLK_1x128_F32
        # routing
        self.row_id_map = torch.empty(T, k, **i32)
        self.src_row = torch.empty(R, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.counts = torch.empty(E, **i32)
        self.ws = torch.empty(max(16, mgq.permute_workspace_size(T, k, E)), **u8)
        if self.nv:
            self._alloc_nvfp4(w, R)
            return
        # activations
        self.xq = torch.empty(R, H, **u8)
        self.xs = torch.empty(mgq.mx_scale_bytes(R, H), **u8) if mx else None
        if blk:   # 1x128 scale_inv, k-block major [K/128][R_cap]
            self.xs = torch.empty(H // 128, R, **f32)
        self.gu = torch.empty(R, 2 * F, **bf)
        self.hq = torch.empty(R, F, **u8)
        self.hs = torch.empty(mgq.mx_scale_bytes(R, F), **u8) if mx else None
        if blk:
            self.hs = torch.empty(F // 128, R, **f32)
        self.h_bf16 = torch.empty(R, F, **bf) if keep_bf16 else None
        self.y = torch.empty(R, H, **bf)
        self.out = torch.empty(T, H, **bf)
        # weights
        self.w1q = torch.empty(E, 2 * F, H, **u8)
        self.w1s = torch.empty(mgq.mx_scale_bytes(E * 2 * F, H), **u8) if mx else None
        self.w2q = torch.empty(E, H, F, **u8)
        self.w2s = torch.empty(mgq.mx_scale_bytes(E * H, F), **u8) if mx else None
        if blk:   # 128x128 scale_inv [E][N/128][K/128]
            self.w1s = torch.empty(E, 2 * F // 128, H // 128, **f32)
            self.w2s = torch.empty(E, H // 128, F // 128, **f32)
        if self.train:
            # per-tensor scales (delayed): [x, h, w1 x E, w2 x E] in e4m3, [dy2, dy1] in e5m2
            nf = 2 + 2 * E
            self.fwd_scale = torch.ones(nf, **f32)
            self.fwd_amax = torch.zeros(nf, **f32)
            self.fwd_hist = torch.zeros(nf, history, **f32)
            self.bwd_scale = torch.ones(2, **f32)
            self.bwd_amax = torch.zeros(2, **f32)
            self.bwd_hist = torch.zeros(2, history, **f32)
            self.heads = torch.zeros(2, **i32)
            self.xcol = torch.empty(H, R, **u8)
            self.hcol = torch.empty(F, R, **u8)
            self.w1col = torch.empty(E, H, 2 * F, **u8)
            self.w2col = torch.empty(E, F, H, **u8)
            self.dy2q = torch.empty(R, H, **u8)
            self.dy2col = torch.empty(H, R, **u8)
            self.dprobs = torch.empty(T, k, **f32)
            self.dh = torch.empty(R, F, **bf)
            self.dy1q = torch.empty(R, 2 * F, **u8)
            self.dy1col = torch.empty(2 * F, R, **u8)
            self.dgu_bf16 = torch.empty(R, 2 * F, **bf) if keep_bf16 else None
            self.dw1 = torch.empty(E, 2 * F, H, **f32)
            self.dw2 = torch.empty(E, H, F, **f32)
            self.dxp = torch.empty(R, H, **bf)
            self.dx = torch.empty(T, H, **bf)

    def _alloc_nvfp4(self, w, R):
        """NVFP4 buffers: e2m1 codes two per byte, tiled ue4m3 scales, and the
        per-tensor (per-expert for weights) amax and global scale s_g:
        [x, h, w1 x E, w2 x E]."""
        E, T, H, F = w.E, w.T, w.H, w.F
        d = self.dev
        u8 = dict(dtype=torch.uint8, device=d)
        self.xq = torch.empty(R, H // 2, **u8)
        self.xs = torch.empty(mgq.nv_scale_bytes(R, H), **u8)
        self.gu = torch.empty(R, 2 * F, dtype=torch.bfloat16, device=d)
        self.h_bf16 = torch.empty(R, F, dtype=torch.bfloat16, device=d)
        self.hq = torch.empty(R, F // 2, **u8)
        self.hs = torch.empty(mgq.nv_scale_bytes(R, F), **u8)
        self.y = torch.empty(R, H, dtype=torch.bfloat16, device=d)
        self.out = torch.empty(T, H, dtype=torch.bfloat16, device=d)
        self.w1q = torch.empty(E, 2 * F, H // 2, **u8)
        self.w1s = torch.empty(mgq.nv_scale_bytes(E * 2 * F, H), **u8)
        self.w2q = torch.empty(E, H, F // 2, **u8)
        self.w2s = torch.empty(mgq.nv_scale_bytes(E * H, F), **u8)
        self.nv_amax = torch.zeros(2 + 2 * E, dtype=torch.float32, device=d)
        self.nv_sg = torch.ones(2 + 2 * E, dtype=torch.float32, device=d)

    def _nv_forward(self, x, topk_idx, probs, stream):
        E, H, F, R = self.w.E, self.w.H, self.w.F, self.R_cap
        a, g = self.nv_amax, self.nv_sg
        qx = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, self.xq, self.xs, tensor_scale=g[0:1], amax_out=a[0:1])
        mgq.moe_permute(x, topk_idx, E, ALIGN, qx, R, self.row_id_map, self.src_row, self.offsets,
                        self.counts, self.ws, None, stream)
        mgq.grouped_gemm_fwd(mgq.operand(self.xq, self.xs, H, mgq.E2M1, g[0:1]),
                             mgq.operand(self.w1q, self.w1s, H, mgq.E2M1, g[2:2 + E]),
                             mgq.NV16_UE4M3, self.offsets, E, R, 2 * F, H, self.gu, mgq.OUT_BF16, stream)
        qh = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, self.hq, self.hs, tensor_scale=g[1:2], amax_out=a[1:2])
        mgq.swiglu_quantize(self.gu, R, F, self.offsets, E, qh, self.h_bf16, stream)
        mgq.grouped_gemm_fwd(mgq.operand(self.hq, self.hs, F, mgq.E2M1, g[1:2]),
                             mgq.operand(self.w2q, self.w2s, F, mgq.E2M1, g[2 + E:2 + 2 * E]),
                             mgq.NV16_UE4M3, self.offsets, E, R, H, F, self.y, mgq.OUT_BF16, stream)
        mgq.moe_unpermute(self.y, self.row_id_map, probs, self.out, stream)
        return self.out

    # ---- scale views (delayed recipe) ------------------------------------------
    def _fs(self, i, n=1):
        return self.fwd_scale[i:i + n]

    def _fa(self, i, n=1):
        return self.fwd_amax[i:i + n]

    # ---- weights ------------------------------------------------------------------
    def quantize_weights(self, w1, w2, stream=None):
        """w1 bf16 [E, 2F, H], w2 bf16 [E, H, F] on the device."""
        E = self.w.E
        if self.nv:
            a, g = self.nv_amax, self.nv_sg
            mgq.block_quantize(w1, mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, self.w1q, self.w1s,
                                             tensor_scale=g[2:2 + E], amax_out=a[2:2 + E]), stream)
            mgq.block_quantize(w2, mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, self.w2q, self.w2s,
                                             tensor_scale=g[2 + E:], amax_out=a[2 + E:]), stream)
        elif self.scaling == mgq.MX32_E8M0:
            mgq.block_quantize(w1, mgq.qdesc(mgq.E4M3, self.scaling, self.w1q, self.w1s), stream)
            mgq.block_quantize(w2, mgq.qdesc(mgq.E4M3, self.scaling, self.w2q, self.w2s), stream)
        elif self.scaling == mgq.BLK_1x128_F32:
            mgq.block_quantize(w1, mgq.qdesc(mgq.E4M3, mgq.BLK_128x128_F32, self.w1q, self.w1s), stream)
            mgq.block_quantize(w2, mgq.qdesc(mgq.E4M3, mgq.BLK_128x128_F32, self.w2q, self.w2s), stream)
        else:
            mgq.block_quantize(w1, mgq.qdesc(mgq.E4M3, self.scaling, self.w1q, None, self.w1col, None,
                                             self._fs(2, E), self._fa(2, E)), stream)
            mgq.block_quantize(w2, mgq.qdesc(mgq.E4M3, self.scaling, self.w2q, None, self.w2col, None,
                                             self._fs(2 + E, E), self._fa(2 + E, E)), stream)

    # ---- forward ------------------------------------------------------------------
    def forward(self, x, topk_idx, probs, stream=None):
        if self.nv:
            return self._nv_forward(x, topk_idx, probs, stream)
        w, E, H, F, R = self.w, self.w.E, self.w.H, self.w.F, self.R_cap
        mx = self.scaling in (mgq.MX32_E8M0, mgq.BLK_1x128_F32)    # scales beside the codes
        if mx:
            qx = mgq.qdesc(mgq.E4M3, self.scaling, self.xq, self.xs)
        else:
            qx = mgq.qdesc(mgq.E4M3, self.scaling, self.xq, None, self.xcol, None, self._fs(0), self._fa(0))
        mgq.moe_permute(x, topk_idx, E, ALIGN, qx, R, self.row_id_map, self.src_row, self.offsets,
                        self.counts, self.ws, None, stream)
        sa = self.xs if mx else self._fs(0)
        sw1 = self.w1s if mx else self._fs(2, E)
        mgq.grouped_gemm_fwd(mgq.operand(self.xq, sa, H, mgq.E4M3), mgq.operand(self.w1q, sw1, H, mgq.E4M3),
                             self.scaling, self.offsets, E, R, 2 * F, H, self.gu, mgq.OUT_BF16, stream)
        if mx:
            qh = mgq.qdesc(mgq.E4M3, self.scaling, self.hq, self.hs)
        else:
            qh = mgq.qdesc(mgq.E4M3, self.scaling, self.hq, None, self.hcol, None, self._fs(1), self._fa(1))
        mgq.swiglu_quantize(self.gu, R, F, self.offsets, E, qh, self.h_bf16, stream)
        sh = self.hs if mx else self._fs(1)
        sw2 = self.w2s if mx else self._fs(2 + E, E)
        mgq.grouped_gemm_fwd(mgq.operand(self.hq, sh, F, mgq.E4M3), mgq.operand(self.w2q, sw2, F, mgq.E4M3),
                             self.scaling, self.offsets, E, R, H, F, self.y, mgq.OUT_BF16, stream)
        mgq.moe_unpermute(self.y, self.row_id_map, probs, self.out, stream)
        return self.out

    # ---- backward (delayed per-tensor recipe) --------------------------------------
    def backward(self, dout, probs, stream=None):
        assert self.train
        E, H, F, R = self.w.E, self.w.H, self.w.F, self.R_cap
        sdy2, sdy1 = self.bwd_scale[0:1], self.bwd_scale[1:2]
        q2 = mgq.qdesc(mgq.E5M2, mgq.TENSOR_F32, self.dy2q, None, self.dy2col, None, sdy2, self.bwd_amax[0:1])
        mgq.moe_unpermute_bwd(dout, self.y, self.row_id_map, self.src_row, probs, R, self.offsets, E, q2,
                              self.dprobs, stream)
        # down projection: dh = dY2 W2 ; dW2 = dY2^T h
        mgq.grouped_gemm_dgrad(mgq.operand(self.dy2q, sdy2, H, mgq.E5M2),
                               mgq.operand(self.w2col, self._fs(2 + E, E), H, mgq.E4M3),
                               mgq.TENSOR_F32, self.offsets, E, R, H, F, self.dh, mgq.OUT_BF16, stream)
        mgq.grouped_gemm_wgrad(mgq.operand(self.dy2col, sdy2, R, mgq.E5M2),
                               mgq.operand(self.hcol, self._fs(1), R, mgq.E4M3),
                               mgq.TENSOR_F32, self.offsets, E, R, H, F, self.dw2, 0.0, mgq.OUT_F32, stream)
        q1 = mgq.qdesc(mgq.E5M2, mgq.TENSOR_F32, self.dy1q, None, self.dy1col, None, sdy1, self.bwd_amax[1:2])
        mgq.dswiglu_quantize(self.dh, self.gu, R, F, self.offsets, E, q1, self.dgu_bf16, stream)
        # gate/up projection: dXp = dY1 W1 ; dW1 = dY1^T X
        mgq.grouped_gemm_dgrad(mgq.operand(self.dy1q, sdy1, 2 * F, mgq.E5M2),
                               mgq.operand(self.w1col, self._fs(2, E), 2 * F, mgq.E4M3),
                               mgq.TENSOR_F32, self.offsets, E, R, 2 * F, H, self.dxp, mgq.OUT_BF16, stream)
        mgq.grouped_gemm_wgrad(mgq.operand(self.dy1col, sdy1, R, mgq.E5M2),
                               mgq.operand(self.xcol, self._fs(0), R, mgq.E4M3),
                               mgq.TENSOR_F32, self.offsets, E, R, 2 * F, H, self.dw1, 0.0, mgq.OUT_F32, stream)
        mgq.moe_permute_bwd(self.dxp, self.row_id_map, self.dx, stream)
        return self.dx

    def update_scaling(self, stream=None):
        """Delayed scaling: push this step's amaxes into the histories and
        derive the scales of the next step."""
        assert self.train
        mgq.amax_history_update(self.fwd_hist, self.heads[0:1], self.fwd_amax, self.fwd_scale,
                                mgq.FMAX[mgq.E4M3], stream)
        mgq.amax_history_update(self.bwd_hist, self.heads[1:2], self.bwd_amax, self.bwd_scale,
                                mgq.FMAX[mgq.E5M2], stream)

    def gpu_launches_per_step(self) -> int:
        """Kernels this object launches per forward (+ backward) step."""
        E = self.w.E
        n_route = 3 if self.w.T * self.w.k > 0 else 1
        fwd = n_route + 1 + 1 + 1 + 1 + 1               # route, permute-quant, gemm1, swiglu, gemm2, unpermute
        if self.nv:
            return fwd + 2 + 4                          # + amax passes (x, h); weights: 2 x (amax + rows)
        if not self.train:
            return fwd + 2                              # weight quantisation (row)
        fwd += 2                                        # col transposes of x and h
        wq = 2 + 2 * E                                  # weight rows + per-expert col transposes
        bwd = 2 + 2 + 2 + 2 + 1                         # unpermute_bwd(+T), dgrad/wgrad x2, dswiglu(+T), permute_bwd
        return fwd + wq + bwd + 2                       # + two history updates

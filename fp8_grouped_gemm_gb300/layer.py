"""The routed-expert layer as a sequence of libmgq calls.

``ExpertLayer`` owns the device buffers of one workload (allocated once with
PyTorch) and issues the C-ABI calls of a forward step and, for the delayed
per-tensor recipe, of the backward step:

forward:  moe_permute (+ quantise) -> grouped_gemm_fwd (gate/up) ->
          swiglu_quantize -> grouped_gemm_fwd (down) -> moe_unpermute
          (MXFP8, NVFP4 and the delayed recipe fuse the gate/up GEMM and
          SwiGLU + quantise into grouped_gemm_fwd_swiglu, MXFP8 training with
          the column-wise copy of h; delayed training also fuses the down
          dgrad and dSwiGLU + quantise into grouped_gemm_dgrad_dswiglu, whose
          MX form, with its column-wise copy, runs no faster than the two
          separate steps on the Mixtral shapes, so MXFP8 training keeps those)
backward: moe_unpermute_bwd (+ quantise dY, dprobs) -> grouped_gemm_dgrad and
          grouped_gemm_wgrad (down) -> dswiglu_quantize -> grouped_gemm_dgrad
          and grouped_gemm_wgrad (gate/up) -> moe_permute_bwd
then:     amax_history_update (delayed scaling)

The backward GEMMs contract over the other dimension of their operands (dgrad
over the weight's rows, wgrad over the tokens). With block scales (MXFP8,
NVFP4, blockwise 1x128 / 128x128) each of those operands is requantised
column-wise with blocks along the new contraction (blockwise: 128x1 blocks
along each expert's tokens; weights' 128x128 tiles are simply transposed). With per-tensor scales the column-wise copy would hold the same
codes transposed, so by default the delayed recipe writes none and hands the
row-wise codes to the GEMMs as MN-major operands (``col_copies=True`` keeps
the explicit copies).

Every step runs in the library's kernels; this module only allocates buffers
and passes pointers.
"""
from __future__ import annotations

import torch

from . import mgq
from .workloads import Workload

ALIGN = 128       # group padding: the grouped GEMM tiles rows by 128
ALIGN_NV_TRAIN = 256   # NVFP4 wgrad: a 128-byte stage holds 256 rows of a group
# NVFP4 GEMMs read the scale image of their second operand
# (mgq_nv_scale_image) when the contraction is at least this long: measured on
# the Mixtral shapes (contractions of 4096 and more) every GEMM gained 4-9%,
# more than the image costs; in the fine-grained forward the gate/up GEMM
# (contraction 2048) gains 6%, the down GEMM (768) less than its image costs
NV_IMAGE_MIN_K = 2048


class ExpertLayer:
    def __init__(self, w: Workload, device, recipe: str | None = None, keep_bf16: bool = False,
                 history: int = 1024, train: bool | None = None, col_copies: bool = False,
                 fuse_swiglu: bool = True, nv_image_min_k: int = NV_IMAGE_MIN_K):
        self.w = w
        self.dev = torch.device(device)
        self.recipe = recipe or w.recipe
        if self.recipe not in ("mxfp8", "delayed", "blockwise", "nvfp4"):
            raise NotImplementedError(self.recipe)
        self.train = (w.backward or self.recipe == "delayed") if train is None else train
        self.delayed = self.recipe == "delayed"
        # per-tensor backward GEMMs read the row-wise codes MN-major
        self.mn = self.delayed and not col_copies
        self.keep_bf16 = keep_bf16
        self.nv_image_min_k = nv_image_min_k
        # SwiGLU in the gate/up GEMM epilogue: MX (training: the epilogue also
        # writes the column-wise copy of h), NVFP4 (the epilogue writes h and
        # its amax; a second pass casts both copies) or per-tensor without a
        # column-wise copy (the blockwise 1x128 block spans both epilogue
        # halves); dSwiGLU in the down dgrad epilogue for per-tensor training
        self.fused_swiglu = fuse_swiglu and (self.recipe in ("mxfp8", "nvfp4") or self.mn)
        if self.train and self.recipe not in ("delayed", "mxfp8", "nvfp4", "blockwise"):
            raise NotImplementedError(f"backward with {self.recipe}")
        self.scaling = {"mxfp8": mgq.MX32_E8M0, "delayed": mgq.TENSOR_F32,
                        "blockwise": mgq.BLK_1x128_F32, "nvfp4": mgq.NV16_UE4M3}[self.recipe]
        self.nv = self.recipe == "nvfp4"
        self.align = ALIGN_NV_TRAIN if (self.nv and self.train) else ALIGN
        E, k, T, H, F = w.E, w.k, w.T, w.H, w.F
        self.R_cap = mgq.r_cap(T, k, E, self.align)
        if self.align == ALIGN_NV_TRAIN:          # the NVFP4 wgrad reads whole 256-row stages
            self.R_cap = (self.R_cap + 255) // 256 * 256
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
            if self.delayed:
                # per-tensor scales (delayed): [x, h, w1 x E, w2 x E] in e4m3, [dy2, dy1] in e5m2
                nf = 2 + 2 * E
                self.fwd_scale = torch.ones(nf, **f32)
                self.fwd_amax = torch.zeros(nf, **f32)
                self.fwd_hist = torch.zeros(nf, history, **f32)
                self.bwd_scale = torch.ones(2, **f32)
                self.bwd_amax = torch.zeros(2, **f32)
                self.bwd_hist = torch.zeros(2, history, **f32)
                self.heads = torch.zeros(2, **i32)
            # column-wise copies (MX: with their own E8M0 scales, blocks along the old rows)
            cols = not self.mn
            self.xcol = torch.empty(H, R, **u8) if cols else None
            self.hcol = torch.empty(F, R, **u8) if cols else None
            self.w1col = torch.empty(E, H, 2 * F, **u8) if cols else None
            self.w2col = torch.empty(E, F, H, **u8) if cols else None
            self.dy2q = torch.empty(R, H, **u8)
            self.dy2col = torch.empty(H, R, **u8) if cols else None
            self.dprobs = torch.empty(T, k, **f32)
            self.dh = torch.empty(R, F, **bf)
            self.dy1q = torch.empty(R, 2 * F, **u8)
            self.dy1col = torch.empty(2 * F, R, **u8) if cols else None
            self.dgu_bf16 = torch.empty(R, 2 * F, **bf) if keep_bf16 else None
            self.dw1 = torch.empty(E, 2 * F, H, **f32)
            self.dw2 = torch.empty(E, H, F, **f32)
            self.dxp = torch.empty(R, H, **bf)
            self.dx = torch.empty(T, H, **bf)
            if blk:
                # float32 scale_inv: row-wise [C/128][R_cap], column-wise
                # [R_cap/128][C] (128x1 blocks along each expert's tokens);
                # weights' column-wise copies carry the transposed 128x128
                # tile scales [E][K/128][N/128]
                self.xcs = torch.empty(R // 128, H, **f32)
                self.hcs = torch.empty(R // 128, F, **f32)
                self.w1cs = torch.empty(E, H // 128, 2 * F // 128, **f32)
                self.w2cs = torch.empty(E, F // 128, H // 128, **f32)
                self.dy2s = torch.empty(H // 128, R, **f32)
                self.dy2cs = torch.empty(R // 128, H, **f32)
                self.dy1s = torch.empty(2 * F // 128, R, **f32)
                self.dy1cs = torch.empty(R // 128, 2 * F, **f32)
            if mx:
                ms = mgq.mx_scale_bytes
                self.xcs = torch.empty(ms(H, R), **u8)
                self.hcs = torch.empty(ms(F, R), **u8)
                self.w1cs = torch.empty(ms(E * H, 2 * F), **u8)
                self.w2cs = torch.empty(ms(E * F, H), **u8)
                self.dy2s = torch.empty(ms(R, H), **u8)
                self.dy2cs = torch.empty(ms(H, R), **u8)
                self.dy1s = torch.empty(ms(R, 2 * F), **u8)
                self.dy1cs = torch.empty(ms(2 * F, R), **u8)

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
        # amax and s_g: [x, h, w1 x E, w2 x E, dy2, dy1]
        self.nv_amax = torch.zeros(4 + 2 * E, dtype=torch.float32, device=d)
        self.nv_sg = torch.ones(4 + 2 * E, dtype=torch.float32, device=d)
        # scale images of the GEMMs' second operands (mgq_nv_scale_image), for
        # the GEMMs whose contraction (ld, the operand's row pitch) is long enough
        img = lambda rows, ld: (torch.empty(mgq.nv_scale_image_bytes(rows, ld), **u8)
                                if ld >= self.nv_image_min_k else None)
        self.w1img, self.w2img = img(E * 2 * F, H), img(E * H, F)
        if not self.train:
            return
        self.w1cimg, self.w2cimg = img(E * H, 2 * F), img(E * F, H)
        self.xcimg, self.hcimg = img(H, R), img(F, R)
        ns = mgq.nv_scale_bytes
        # column-wise copies (16x1 blocks along the tokens; weights: the same
        # 16x16 block scales as their row-wise copies), e2m1 packed along them
        self.xcol, self.xcs = torch.empty(H, R // 2, **u8), torch.empty(ns(H, R), **u8)
        self.hcol, self.hcs = torch.empty(F, R // 2, **u8), torch.empty(ns(F, R), **u8)
        self.w1col, self.w1cs = torch.empty(E, H, F, **u8), torch.empty(ns(E * H, 2 * F), **u8)
        self.w2col, self.w2cs = torch.empty(E, F, H // 2, **u8), torch.empty(ns(E * F, H), **u8)
        self.dy2q, self.dy2s = torch.empty(R, H // 2, **u8), torch.empty(ns(R, H), **u8)
        self.dy2col, self.dy2cs = torch.empty(H, R // 2, **u8), torch.empty(ns(H, R), **u8)
        self.dy1q, self.dy1s = torch.empty(R, F, **u8), torch.empty(ns(R, 2 * F), **u8)
        self.dy1col, self.dy1cs = torch.empty(2 * F, R // 2, **u8), torch.empty(ns(2 * F, R), **u8)
        bf = dict(dtype=torch.bfloat16, device=d)
        f32 = dict(dtype=torch.float32, device=d)
        self.dprobs = torch.empty(T, w.k, **f32)
        self.dh = torch.empty(R, F, **bf)
        self.dgu_bf16 = torch.empty(R, 2 * F, **bf)      # materialised: its amax precedes the cast
        self.dw1 = torch.empty(E, 2 * F, H, **f32)
        self.dw2 = torch.empty(E, H, F, **f32)
        self.dxp = torch.empty(R, H, **bf)
        self.dx = torch.empty(T, H, **bf)

    # ---- scale views (delayed recipe) ------------------------------------------
    def _fs(self, i, n=1):
        return self.fwd_scale[i:i + n]

    def _fa(self, i, n=1):
        return self.fwd_amax[i:i + n]

    # ---- the call sequence, as named operations (one C-ABI call each) ------------
    # The ops capture only persistent buffers; running them in order is the
    # step. bench.py brackets each with CUDA events to time the kernels.

    def weight_ops(self, w1, w2, stream=None):
        """Quantisation of w1 bf16 [E, 2F, H] and w2 bf16 [E, H, F]."""
        E, Q = self.w.E, mgq.block_quantize
        if self.nv:
            a, g = self.nv_amax, self.nv_sg
            if self.train:
                # 16x16 blocks: one pass writes the row-wise and column-wise copies
                sc2d = mgq.NV16x16_UE4M3
                q1 = mgq.qdesc(mgq.E2M1, sc2d, self.w1q, self.w1s, self.w1col, self.w1cs, tensor_scale=g[2:2 + E],
                               amax_out=a[2:2 + E])
                q2 = mgq.qdesc(mgq.E2M1, sc2d, self.w2q, self.w2s, self.w2col, self.w2cs,
                               tensor_scale=g[2 + E:2 + 2 * E], amax_out=a[2 + E:2 + 2 * E])
            else:
                q1 = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, self.w1q, self.w1s, tensor_scale=g[2:2 + E],
                               amax_out=a[2:2 + E])
                q2 = mgq.qdesc(mgq.E2M1, mgq.NV16_UE4M3, self.w2q, self.w2s, tensor_scale=g[2 + E:2 + 2 * E],
                               amax_out=a[2 + E:2 + 2 * E])
        elif self.scaling == mgq.MX32_E8M0:
            c1 = (self.w1col, self.w1cs) if self.train else (None, None)
            c2 = (self.w2col, self.w2cs) if self.train else (None, None)
            q1 = mgq.qdesc(mgq.E4M3, self.scaling, self.w1q, self.w1s, *c1)
            q2 = mgq.qdesc(mgq.E4M3, self.scaling, self.w2q, self.w2s, *c2)
        elif self.scaling == mgq.BLK_1x128_F32:
            # 128x128 tiles; training: the column-wise copy (transposed codes
            # and tile scales) from the same pass
            c1 = (self.w1col, self.w1cs) if self.train else (None, None)
            c2 = (self.w2col, self.w2cs) if self.train else (None, None)
            q1 = mgq.qdesc(mgq.E4M3, mgq.BLK_128x128_F32, self.w1q, self.w1s, *c1)
            q2 = mgq.qdesc(mgq.E4M3, mgq.BLK_128x128_F32, self.w2q, self.w2s, *c2)
        else:
            q1 = mgq.qdesc(mgq.E4M3, self.scaling, self.w1q, None, self.w1col, None, self._fs(2, E), self._fa(2, E))
            q2 = mgq.qdesc(mgq.E4M3, self.scaling, self.w2q, None, self.w2col, None, self._fs(2 + E, E),
                           self._fa(2 + E, E))
        ops = [("weight_quant", lambda: Q(w1, q1, stream)), ("weight_quant", lambda: Q(w2, q2, stream))]
        if self.nv:
            H, F = self.w.H, self.w.F
            ops += self._image_ops([(self.w1s, E * 2 * F, H, self.w1img), (self.w2s, E * H, F, self.w2img)], stream)
            if self.train:
                ops += self._image_ops([(self.w1cs, E * H, 2 * F, self.w1cimg), (self.w2cs, E * F, H, self.w2cimg)],
                                       stream)
        return ops

    @staticmethod
    def _image_ops(items, stream):
        """One scale-image op per (scales, rows, ld, image) with an image."""
        return [("scale_image", (lambda s=s, r=r, ld=ld, im=im: mgq.nv_scale_image(s, r, ld, im, stream)))
                for s, r, ld, im in items if im is not None]

    def fwd_ops(self, x, topk_idx, probs, stream=None):
        E, H, F, R = self.w.E, self.w.H, self.w.F, self.R_cap
        sc = self.scaling
        if self.nv:
            a, g = self.nv_amax, self.nv_sg
            dt = mgq.E2M1
            cx = (self.xcol, self.xcs) if self.train else (None, None)
            ch = (self.hcol, self.hcs) if self.train else (None, None)
            qx = mgq.qdesc(dt, sc, self.xq, self.xs, *cx, tensor_scale=g[0:1], amax_out=a[0:1])
            qh = mgq.qdesc(dt, sc, self.hq, self.hs, *ch, tensor_scale=g[1:2], amax_out=a[1:2])
            A1, B1 = (mgq.operand(self.xq, self.xs, H, dt, g[0:1]),
                      mgq.operand(self.w1q, self.w1s, H, dt, g[2:2 + E], scale_image=self.w1img))
            A2, B2 = (mgq.operand(self.hq, self.hs, F, dt, g[1:2]),
                      mgq.operand(self.w2q, self.w2s, F, dt, g[2 + E:2 + 2 * E], scale_image=self.w2img))
        else:
            dt = mgq.E4M3
            if sc in (mgq.MX32_E8M0, mgq.BLK_1x128_F32):       # block scales beside the codes
                cx = (self.xcol, self.xcs) if self.train else (None, None)
                ch = (self.hcol, self.hcs) if self.train else (None, None)
                qx = mgq.qdesc(dt, sc, self.xq, self.xs, *cx)
                qh = mgq.qdesc(dt, sc, self.hq, self.hs, *ch)
                sa, sw1, sh, sw2 = self.xs, self.w1s, self.hs, self.w2s
            else:                                               # delayed per-tensor
                qx = mgq.qdesc(dt, sc, self.xq, None, self.xcol, None, self._fs(0), self._fa(0))
                qh = mgq.qdesc(dt, sc, self.hq, None, self.hcol, None, self._fs(1), self._fa(1))
                sa, sw1, sh, sw2 = self._fs(0), self._fs(2, E), self._fs(1), self._fs(2 + E, E)
            A1, B1 = mgq.operand(self.xq, sa, H, dt), mgq.operand(self.w1q, sw1, H, dt)
            A2, B2 = mgq.operand(self.hq, sh, F, dt), mgq.operand(self.w2q, sw2, F, dt)
        # routing (index work) and the permute + quantise (HBM-bound) as two ops
        permute = [("route", lambda: mgq.moe_route(topk_idx, E, self.align, R, self.row_id_map, self.src_row,
                                                   self.offsets, self.counts, self.ws, stream)),
                   ("permute_quant", lambda: mgq.moe_permute_routed(x, self.w.k, E, qx, R, self.row_id_map,
                                                                    self.src_row, self.offsets, self.counts, None,
                                                                    stream))]
        if self.fused_swiglu:
            # g | u only where something reads them (backward, or checks)
            gu = self.gu if (self.train or self.keep_bf16) else None
            gateup = [("gemm_fwd_gateup_swiglu",
                       lambda: mgq.grouped_gemm_fwd_swiglu(A1, B1, sc, self.offsets, E, R, F, H, qh, gu, self.h_bf16,
                                                           stream))]
        else:
            gateup = [
                ("gemm_fwd_gateup", lambda: mgq.grouped_gemm_fwd(A1, B1, sc, self.offsets, E, R, 2 * F, H, self.gu,
                                                                 mgq.OUT_BF16, stream)),
                ("swiglu_quant", lambda: mgq.swiglu_quantize(self.gu, R, F, self.offsets, E, qh, self.h_bf16,
                                                             stream))]
        if self.nv and self.train:
            # scale images of the column-wise copies of x and h (the wgrads' second operands)
            permute += self._image_ops([(self.xcs, H, R, self.xcimg)], stream)
            gateup += self._image_ops([(self.hcs, F, R, self.hcimg)], stream)
        return permute + gateup + [
            ("gemm_fwd_down", lambda: mgq.grouped_gemm_fwd(A2, B2, sc, self.offsets, E, R, H, F, self.y,
                                                           mgq.OUT_BF16, stream)),
            ("unpermute", lambda: mgq.moe_unpermute(self.y, self.row_id_map, probs, self.out, stream)),
        ]

    def bwd_ops(self, dout, probs, stream=None):
        assert self.train
        E, H, F, R = self.w.E, self.w.H, self.w.F, self.R_cap
        if self.nv:
            return self._bwd_ops_nvfp4(dout, probs, stream)
        if self.delayed:
            sc = mgq.TENSOR_F32
            sdy2, sdy1 = self.bwd_scale[0:1], self.bwd_scale[1:2]
            q2 = mgq.qdesc(mgq.E5M2, sc, self.dy2q, None, self.dy2col, None, sdy2, self.bwd_amax[0:1])
            q1 = mgq.qdesc(mgq.E5M2, sc, self.dy1q, None, self.dy1col, None, sdy1, self.bwd_amax[1:2])
            # per-tensor: the column-wise copy shares the row-wise scale
            s_dy2r = s_dy2c = sdy2
            s_dy1r = s_dy1c = sdy1
            s_w2c, s_w1c = self._fs(2 + E, E), self._fs(2, E)
            s_hc, s_xc = self._fs(1), self._fs(0)
        else:
            # block scales (MX E8M0 per 32, or blockwise float32 1x128 / 128x1):
            # row-wise and column-wise copies of each gradient
            sc = self.scaling
            q2 = mgq.qdesc(mgq.E5M2, sc, self.dy2q, self.dy2s, self.dy2col, self.dy2cs)
            q1 = mgq.qdesc(mgq.E5M2, sc, self.dy1q, self.dy1s, self.dy1col, self.dy1cs)
            s_dy2r, s_dy2c, s_dy1r, s_dy1c = self.dy2s, self.dy2cs, self.dy1s, self.dy1cs
            s_w2c, s_w1c, s_hc, s_xc = self.w2cs, self.w1cs, self.hcs, self.xcs
        O = mgq.operand
        if self.mn:
            # the row-wise codes, read transposed by the tensor cores
            MN = mgq.LAYOUT_MN
            d2 = (O(self.dy2q, s_dy2r, H, mgq.E5M2), O(self.w2q, s_w2c, F, mgq.E4M3, layout=MN))
            w2 = (O(self.dy2q, s_dy2c, H, mgq.E5M2, layout=MN), O(self.hq, s_hc, F, mgq.E4M3, layout=MN))
            d1 = (O(self.dy1q, s_dy1r, 2 * F, mgq.E5M2), O(self.w1q, s_w1c, H, mgq.E4M3, layout=MN))
            w1 = (O(self.dy1q, s_dy1c, 2 * F, mgq.E5M2, layout=MN), O(self.xq, s_xc, H, mgq.E4M3, layout=MN))
        else:
            # down projection: dh = dY2 W2 ; dW2 = dY2^T h
            d2 = (O(self.dy2q, s_dy2r, H, mgq.E5M2), O(self.w2col, s_w2c, H, mgq.E4M3))
            w2 = (O(self.dy2col, s_dy2c, R, mgq.E5M2), O(self.hcol, s_hc, R, mgq.E4M3))
            # gate/up projection: dXp = dY1 W1 ; dW1 = dY1^T X
            d1 = (O(self.dy1q, s_dy1r, 2 * F, mgq.E5M2), O(self.w1col, s_w1c, 2 * F, mgq.E4M3))
            w1 = (O(self.dy1col, s_dy1c, R, mgq.E5M2), O(self.xcol, s_xc, R, mgq.E4M3))
        ops = [
            ("unpermute_bwd_quant", lambda: mgq.moe_unpermute_bwd(dout, self.y, self.row_id_map, self.src_row, probs,
                                                                  R, self.offsets, E, q2, self.dprobs, stream)),
        ]
        wgrad_down = ("gemm_wgrad_down", lambda: mgq.grouped_gemm_wgrad(*w2, sc, self.offsets, E, R, H, F, self.dw2,
                                                                         0.0, mgq.OUT_F32, stream))
        if self.fused_swiglu and self.delayed:
            # dh only where a check reads it
            dh = self.dh if self.keep_bf16 else None
            ops += [("gemm_dgrad_down_dswiglu",
                     lambda: mgq.grouped_gemm_dgrad_dswiglu(*d2, sc, self.offsets, E, R, H, F, self.gu, q1, dh,
                                                            self.dgu_bf16, stream)), wgrad_down]
        else:
            ops += [("gemm_dgrad_down", lambda: mgq.grouped_gemm_dgrad(*d2, sc, self.offsets, E, R, H, F, self.dh,
                                                                       mgq.OUT_BF16, stream)), wgrad_down,
                    ("dswiglu_quant", lambda: mgq.dswiglu_quantize(self.dh, self.gu, R, F, self.offsets, E, q1,
                                                                   self.dgu_bf16, stream))]
        return ops + [
            ("gemm_dgrad_gateup", lambda: mgq.grouped_gemm_dgrad(*d1, sc, self.offsets, E, R, 2 * F, H, self.dxp,
                                                                 mgq.OUT_BF16, stream)),
            ("gemm_wgrad_gateup", lambda: mgq.grouped_gemm_wgrad(*w1, sc, self.offsets, E, R, 2 * F, H, self.dw1,
                                                                 0.0, mgq.OUT_F32, stream)),
            ("permute_bwd", lambda: mgq.moe_permute_bwd(self.dxp, self.row_id_map, self.dx, stream)),
        ]

    def _bwd_ops_nvfp4(self, dout, probs, stream=None):
        """NVFP4 backward: dY2 and dY1 = [dG | dU] quantised row-wise (dgrad)
        and column-wise (wgrad) with their own s_g; weights' column-wise
        copies share the 16x16 block scales of the row-wise ones."""
        E, H, F, R = self.w.E, self.w.H, self.w.F, self.R_cap
        sc, dt, O = mgq.NV16_UE4M3, mgq.E2M1, mgq.operand
        a, g = self.nv_amax, self.nv_sg
        i2, i1 = 2 + 2 * E, 3 + 2 * E
        q2 = mgq.qdesc(dt, sc, self.dy2q, self.dy2s, self.dy2col, self.dy2cs, tensor_scale=g[i2:i2 + 1],
                       amax_out=a[i2:i2 + 1])
        q1 = mgq.qdesc(dt, sc, self.dy1q, self.dy1s, self.dy1col, self.dy1cs, tensor_scale=g[i1:i1 + 1],
                       amax_out=a[i1:i1 + 1])
        gw1, gw2 = g[2:2 + E], g[2 + E:2 + 2 * E]
        # down projection: dh = dY2 W2 ; dW2 = dY2^T h
        d2 = (O(self.dy2q, self.dy2s, H, dt, g[i2:i2 + 1]),
              O(self.w2col, self.w2cs, H, dt, gw2, scale_image=self.w2cimg))
        w2 = (O(self.dy2col, self.dy2cs, R, dt, g[i2:i2 + 1]),
              O(self.hcol, self.hcs, R, dt, g[1:2], scale_image=self.hcimg))
        # gate/up projection: dXp = dY1 W1 ; dW1 = dY1^T X
        d1 = (O(self.dy1q, self.dy1s, 2 * F, dt, g[i1:i1 + 1]),
              O(self.w1col, self.w1cs, 2 * F, dt, gw1, scale_image=self.w1cimg))
        w1 = (O(self.dy1col, self.dy1cs, R, dt, g[i1:i1 + 1]),
              O(self.xcol, self.xcs, R, dt, g[0:1], scale_image=self.xcimg))
        return [
            ("unpermute_bwd_quant", lambda: mgq.moe_unpermute_bwd(dout, self.y, self.row_id_map, self.src_row, probs,
                                                                  R, self.offsets, E, q2, self.dprobs, stream)),
            ("gemm_dgrad_down", lambda: mgq.grouped_gemm_dgrad(*d2, sc, self.offsets, E, R, H, F, self.dh,
                                                               mgq.OUT_BF16, stream)),
            ("gemm_wgrad_down", lambda: mgq.grouped_gemm_wgrad(*w2, sc, self.offsets, E, R, H, F, self.dw2, 0.0,
                                                               mgq.OUT_F32, stream)),
            ("dswiglu_quant", lambda: mgq.dswiglu_quantize(self.dh, self.gu, R, F, self.offsets, E, q1,
                                                           self.dgu_bf16, stream)),
            ("gemm_dgrad_gateup", lambda: mgq.grouped_gemm_dgrad(*d1, sc, self.offsets, E, R, 2 * F, H, self.dxp,
                                                                 mgq.OUT_BF16, stream)),
            ("gemm_wgrad_gateup", lambda: mgq.grouped_gemm_wgrad(*w1, sc, self.offsets, E, R, 2 * F, H, self.dw1,
                                                                 0.0, mgq.OUT_F32, stream)),
            ("permute_bwd", lambda: mgq.moe_permute_bwd(self.dxp, self.row_id_map, self.dx, stream)),
        ]

    def update_ops(self, stream=None):
        return [("scaling_update", lambda: self.update_scaling(stream))] if self.delayed else []

    def step_ops(self, w1, w2, x, topk_idx, probs, dout=None, stream=None):
        """One whole step: weights, forward, and (training) backward + scaling."""
        ops = self.weight_ops(w1, w2, stream) + self.fwd_ops(x, topk_idx, probs, stream)
        if self.train:
            ops += self.bwd_ops(dout, probs, stream) + self.update_ops(stream)
        return ops

    # ---- convenience wrappers ---------------------------------------------------------
    def quantize_weights(self, w1, w2, stream=None):
        for _, op in self.weight_ops(w1, w2, stream):
            op()

    def forward(self, x, topk_idx, probs, stream=None):
        for _, op in self.fwd_ops(x, topk_idx, probs, stream):
            op()
        return self.out

    def backward(self, dout, probs, stream=None):
        for _, op in self.bwd_ops(dout, probs, stream):
            op()
        return self.dx

    def update_scaling(self, stream=None):
        """Delayed scaling: push this step's amaxes into the histories and
        derive the scales of the next step (nothing to do for MX scaling)."""
        if not self.delayed:
            return
        mgq.amax_history_update(self.fwd_hist, self.heads[0:1], self.fwd_amax, self.fwd_scale,
                                mgq.FMAX[mgq.E4M3], stream)
        mgq.amax_history_update(self.bwd_hist, self.heads[1:2], self.bwd_amax, self.bwd_scale,
                                mgq.FMAX[mgq.E5M2], stream)

    def _n_images(self) -> int:
        names = ("w1img", "w2img", "w1cimg", "w2cimg", "xcimg", "hcimg")
        return sum(getattr(self, n, None) is not None for n in names)

    def gpu_launches_per_step(self) -> int:
        """Kernels this object launches per forward (+ backward) step."""
        E = self.w.E
        n_route = 3 if self.w.T * self.w.k > 0 else 1   # count + rank, scan, finalize
        fwd = n_route + 1 + 1 + 1 + 1 + 1               # route, permute-quant, gemm1, swiglu, gemm2, unpermute
        if self.fused_swiglu:
            fwd -= 1                                    # SwiGLU in the gate/up GEMM epilogue
        if self.nv and self.train:
            # permute: x amax + one row/column tile pass; the gate/up GEMM's
            # second pass writes both copies of h; weights: 2 x (amax + 16x16
            # pass); backward: dY amax + token rows + column gather, dgrad,
            # wgrad, dSwiGLU (dGU + amax, then rows and columns), dgrad, wgrad,
            # permute_bwd; the scale images (both weights, both weight column
            # copies, the column copies of x and h) where they are used
            return fwd + 2 + 4 + (3 + 1 + 1 + 2 + 1 + 1 + 1) + self._n_images()
        if self.nv:
            # + amax passes (x, h); weights: 2 x (amax + rows); the permute's
            # row-major scales re-tiled in a second pass when a 128-row group's
            # scales fit a CTA's shared memory
            H = self.w.H
            retile = 1 if H % 256 == 0 and 128 * (H // 64 + 1) * 4 <= 200 * 1024 else 0
            return fwd + 2 + 4 + retile + self._n_images()   # + the weights' scale images
        if not self.train:
            return fwd + 2                              # weight quantisation (row)
        wq = 2                                          # weights: rows (+ columns) in one pass each
        bwd = 1 + 2 + 1 + 2 + 1                         # unpermute_bwd, dgrad/wgrad, dswiglu (fused
                                                        # columns), dgrad/wgrad, permute_bwd
        if self.fused_swiglu and self.delayed:
            bwd -= 1                                    # dSwiGLU in the down dgrad epilogue
        if not self.mn:
            if self.delayed:
                fwd += 1                                # column copy of x (MX: fused into the permute;
                                                        # h's is fused into SwiGLU)
            bwd += 1                                    # column copy of dY2
        return fwd + wq + bwd + (2 if self.delayed else 0)

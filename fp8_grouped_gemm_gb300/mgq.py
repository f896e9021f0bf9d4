"""Thin Python binding of libmgq (include/mgq.h), by ctypes.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Tensors are PyTorch tensors (device memory and streams come from
PyTorch); each function passes their data pointers and the current CUDA stream
to the C entry point of the same name and raises MGQError on a non-OK status.

Loading fails loudly (ImportError) when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmgq.so")

# enums of mgq.h
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_INDEX = range(6)
E4M3, E5M2, E2M1 = 0, 1, 2
MX32_E8M0, NV16_UE4M3, BLK_1x128_F32, BLK_128x128_F32, TENSOR_F32, NV16x16_UE4M3 = range(6)
RCEIL, FLOOR = 0, 1
OUT_BF16, OUT_F32 = 0, 1
LAYOUT_K, LAYOUT_MN = 0, 1
(GEMM_OPT_FORCE_1CTA, GEMM_OPT_MX_PAIR, GEMM_OPT_NV_PAIR, GEMM_OPT_DIRECT_STORE, GEMM_OPT_DEBUG_STALL,
 GEMM_OPT_WAIT_MS) = range(6)

FMAX = {E4M3: 448.0, E5M2: 57344.0}

# every symbol include/mgq.h declares
INTERFACE_VERSION = 2   # mgq_version() of the library these struct mirrors match

EXPORTS = (
    "mgq_status_string", "mgq_version", "mgq_get_error", "mgq_permute_workspace_size",
    "mgq_moe_permute", "mgq_moe_route", "mgq_moe_permute_routed", "mgq_moe_permute_noalloc", "mgq_block_quantize", "mgq_grouped_quantize", "mgq_grouped_gemm_fwd", "mgq_grouped_gemm_dgrad",
    "mgq_grouped_gemm_wgrad", "mgq_grouped_gemm_fwd_swiglu",
    "mgq_grouped_gemm_dgrad_dswiglu", "mgq_swiglu_quantize", "mgq_dswiglu_quantize", "mgq_moe_unpermute",
    "mgq_moe_unpermute_bwd", "mgq_moe_permute_bwd", "mgq_amax_history_update", "mgq_set_gemm_option",
    "mgq_get_gemm_option", "mgq_nv_scale_image",
)


class MGQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class QBuf(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class QDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("scaling", ctypes.c_int), ("e8m0_mode", ctypes.c_int),
                ("row", QBuf), ("col", QBuf), ("tensor_scale", ctypes.c_void_p),
                ("amax_out", ctypes.c_void_p)]


class Operand(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("ld", ctypes.c_int64),
                ("dtype", ctypes.c_int), ("global_scale", ctypes.c_void_p), ("layout", ctypes.c_int),
                ("scale_image", ctypes.c_void_p)]


_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmgq.so not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        P = ctypes.POINTER
        lib.mgq_status_string.restype = ctypes.c_char_p
        lib.mgq_status_string.argtypes = [i32]
        lib.mgq_version.restype = i32
        lib.mgq_get_error.argtypes = [vp, P(i32)]
        lib.mgq_permute_workspace_size.restype = sz
        lib.mgq_permute_workspace_size.argtypes = [i32, i32, i32]
        lib.mgq_moe_permute.argtypes = [vp, i32, i32, vp, i32, i32, i32, P(QDesc), vp, i64,
                                        vp, vp, vp, vp, vp, sz, vp]
        lib.mgq_moe_route.argtypes = [vp, i32, i32, i32, i32, i64, vp, vp, vp, vp, vp, sz, vp]
        lib.mgq_moe_permute_routed.argtypes = [vp, i32, i32, i32, i32, P(QDesc), vp, i64, vp, vp, vp, vp, vp]
        lib.mgq_moe_permute_noalloc.argtypes = [vp, i32, i32, vp, i32, i32, i32, P(QDesc), vp, i64,
                                                vp, vp, vp, vp, vp]
        lib.mgq_block_quantize.argtypes = [vp, i64, i64, i64, P(QDesc), vp]
        lib.mgq_grouped_quantize.argtypes = [vp, i64, i64, vp, i32, P(QDesc), vp]
        gemm = [P(Operand), P(Operand), i32, vp, i32, i64, i64, i64]
        lib.mgq_grouped_gemm_fwd.argtypes = gemm + [vp, i32, vp]
        lib.mgq_grouped_gemm_dgrad.argtypes = gemm + [vp, i32, vp]
        lib.mgq_grouped_gemm_wgrad.argtypes = gemm + [ctypes.c_float, vp, i32, vp]
        lib.mgq_nv_scale_image.argtypes = [vp, i64, i64, vp, vp]
        lib.mgq_grouped_gemm_fwd_swiglu.argtypes = gemm + [P(QDesc), vp, vp, vp]
        lib.mgq_grouped_gemm_dgrad_dswiglu.argtypes = gemm + [vp, P(QDesc), vp, vp, vp]
        lib.mgq_swiglu_quantize.argtypes = [vp, i64, i32, vp, i32, P(QDesc), vp, vp]
        lib.mgq_dswiglu_quantize.argtypes = [vp, vp, i64, i32, vp, i32, P(QDesc), vp, vp]
        lib.mgq_moe_unpermute.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
        lib.mgq_moe_unpermute_bwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, vp, i32,
                                              P(QDesc), vp, vp]
        lib.mgq_moe_permute_bwd.argtypes = [vp, vp, i32, i32, i32, vp, vp]
        lib.mgq_amax_history_update.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.c_float, vp]
        lib.mgq_set_gemm_option.argtypes = [i32, i64]
        lib.mgq_get_gemm_option.argtypes = [i32, P(i64)]
        for name in EXPORTS:
            if name not in ("mgq_status_string", "mgq_permute_workspace_size"):
                getattr(lib, name).restype = i32
        if lib.mgq_version() != INTERFACE_VERSION:   # the struct layouts below are this version's
            raise RuntimeError(f"{LIB_PATH}: interface version {lib.mgq_version()}, expected {INTERFACE_VERSION}")
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().mgq_status_string(status).decode()


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != OK:
        raise MGQError(rc, where)


def qdesc(dtype, scaling, row_data, row_scale=None, col_data=None, col_scale=None,
          tensor_scale=None, amax_out=None, e8m0_mode=RCEIL) -> QDesc:
    return QDesc(dtype, scaling, e8m0_mode, QBuf(_p(row_data), _p(row_scale)),
                 QBuf(_p(col_data), _p(col_scale)), _p(tensor_scale), _p(amax_out))


def operand(data, scale, ld, dtype, global_scale=None, layout=0, scale_image=None) -> Operand:
    return Operand(_p(data), _p(scale), int(ld), int(dtype), _p(global_scale), int(layout), _p(scale_image))


# ---- sizes of the caller-owned buffers (host arithmetic only) ----------------

def r_cap(T: int, k: int, E: int, align: int) -> int:
    """Rows the permuted buffers need: T*k + E*(align-1), rounded up to 128."""
    n = T * k + E * (align - 1)
    return (n + 127) // 128 * 128


def mx_scale_bytes(rows: int, ld: int) -> int:
    """Bytes of the 128x4-tiled E8M0 scales of a [rows, ld] matrix."""
    return (rows + 127) // 128 * 128 * (ld // 32)


def nv_scale_bytes(rows: int, ld: int) -> int:
    """Bytes of the 128x4-tiled ue4m3 scales (one per 16 elements) of a [rows, ld] matrix."""
    return (rows + 127) // 128 * 128 * (ld // 16)


def permute_workspace_size(T: int, k: int, E: int) -> int:
    return int(load().mgq_permute_workspace_size(T, k, E))


# ---- entry points --------------------------------------------------------------

def get_error(stream=None) -> int:
    st = ctypes.c_int(0)
    _check(load().mgq_get_error(_s(stream), ctypes.byref(st)), "mgq_get_error")
    return st.value


def set_gemm_option(option: int, value: int) -> None:
    _check(load().mgq_set_gemm_option(int(option), int(value)), "mgq_set_gemm_option")


def get_gemm_option(option: int) -> int:
    v = ctypes.c_int64(0)
    _check(load().mgq_get_gemm_option(int(option), ctypes.byref(v)), "mgq_get_gemm_option")
    return v.value


def moe_permute(x, topk_idx, E, align, q: QDesc | None, R_cap, row_id_map, src_row, offsets,
                counts, workspace, out_bf16=None, stream=None):
    T, H = (x.shape[0], x.shape[1]) if x is not None else (0, 0)
    k = topk_idx.shape[1]
    rc = load().mgq_moe_permute(_p(x), T, H, _p(topk_idx), k, E, align,
                                ctypes.byref(q) if q is not None else None, _p(out_bf16), R_cap,
                                _p(row_id_map), _p(src_row), _p(offsets), _p(counts), _p(workspace),
                                workspace.numel() * workspace.element_size(), _s(stream))
    _check(rc, "mgq_moe_permute")


def moe_route(topk_idx, E, align, R_cap, row_id_map, src_row, offsets, counts, workspace, stream=None):
    """Routing alone (row_id_map, src_row, offsets, counts as mgq_moe_permute)."""
    T, k = topk_idx.shape
    _check(load().mgq_moe_route(_p(topk_idx), T, k, E, align, R_cap, _p(row_id_map), _p(src_row), _p(offsets),
                                _p(counts), _p(workspace), workspace.numel() * workspace.element_size(),
                                _s(stream)), "mgq_moe_route")


def moe_permute_routed(x, k, E, q: QDesc, R_cap, row_id_map, src_row, offsets, counts, out_bf16=None,
                       stream=None):
    """Permute + quantise on final routing arrays from moe_route."""
    T, H = x.shape
    _check(load().mgq_moe_permute_routed(_p(x), T, H, k, E, ctypes.byref(q), _p(out_bf16), R_cap, _p(row_id_map),
                                         _p(src_row), _p(offsets), _p(counts), _s(stream)),
           "mgq_moe_permute_routed")


def moe_permute_noalloc(x, topk_idx, E, align, q: QDesc | None, R_cap, row_id_map, src_row, offsets,
                        counts, out_bf16=None, stream=None):
    """mgq_moe_permute without a workspace: the routing scratch is the
    library's fixed 1 MiB device array (for callers that cannot allocate)."""
    T, H = (x.shape[0], x.shape[1]) if x is not None else (0, 0)
    k = topk_idx.shape[1]
    rc = load().mgq_moe_permute_noalloc(_p(x), T, H, _p(topk_idx), k, E, align,
                                        ctypes.byref(q) if q is not None else None, _p(out_bf16), R_cap,
                                        _p(row_id_map), _p(src_row), _p(offsets), _p(counts), _s(stream))
    _check(rc, "mgq_moe_permute_noalloc")


def block_quantize(x, q: QDesc, stream=None):
    """x: [G, M, K] (or [M, K]) bf16."""
    shp = tuple(x.shape)
    G, M, K = shp if len(shp) == 3 else (1,) + shp
    _check(load().mgq_block_quantize(_p(x), G, M, K, ctypes.byref(q), _s(stream)), "mgq_block_quantize")


def grouped_quantize(x, offsets, E, q: QDesc, stream=None):
    """x: [R_cap, C] bf16; rows [0, offsets[E]) in ragged groups."""
    R_cap, C = x.shape
    _check(load().mgq_grouped_quantize(_p(x), R_cap, C, _p(offsets), E, ctypes.byref(q), _s(stream)),
           "mgq_grouped_quantize")


def grouped_gemm_fwd(A: Operand, W: Operand, scaling, offsets, E, R_cap, N, K, Y, out_dtype=OUT_BF16,
                     stream=None):
    _check(load().mgq_grouped_gemm_fwd(ctypes.byref(A), ctypes.byref(W), scaling, _p(offsets), E, R_cap,
                                       N, K, _p(Y), out_dtype, _s(stream)), "mgq_grouped_gemm_fwd")


def grouped_gemm_dgrad(dY: Operand, Wcol: Operand, scaling, offsets, E, R_cap, N, K, dA,
                       out_dtype=OUT_BF16, stream=None):
    _check(load().mgq_grouped_gemm_dgrad(ctypes.byref(dY), ctypes.byref(Wcol), scaling, _p(offsets), E,
                                         R_cap, N, K, _p(dA), out_dtype, _s(stream)),
           "mgq_grouped_gemm_dgrad")


def grouped_gemm_wgrad(dYcol: Operand, Acol: Operand, scaling, offsets, E, R_cap, N, K, dW, beta=0.0,
                       out_dtype=OUT_F32, stream=None):
    _check(load().mgq_grouped_gemm_wgrad(ctypes.byref(dYcol), ctypes.byref(Acol), scaling, _p(offsets), E,
                                         R_cap, N, K, ctypes.c_float(beta), _p(dW), out_dtype, _s(stream)),
           "mgq_grouped_gemm_wgrad")


def nv_scale_image(scale, rows, ld, image, stream=None):
    """The GEMM scale image of an NVFP4 operand's scales (rows * ld / 4 bytes)."""
    _check(load().mgq_nv_scale_image(_p(scale), rows, ld, _p(image), _s(stream)), "mgq_nv_scale_image")


def nv_scale_image_bytes(rows, ld):
    return rows * ld // 4


def grouped_gemm_fwd_swiglu(A: Operand, W1: Operand, scaling, offsets, E, R_cap, F, K, qh: QDesc, gu=None, h=None,
                            stream=None):
    """Gate/up GEMM with SwiGLU + row-wise quantisation of h in its epilogue
    (MX: also the column-wise copy when qh has one; gu [R_cap, 2F] and h
    [R_cap, F] bf16 written only when given)."""
    _check(load().mgq_grouped_gemm_fwd_swiglu(ctypes.byref(A), ctypes.byref(W1), scaling, _p(offsets), E, R_cap,
                                              F, K, ctypes.byref(qh), _p(gu), _p(h), _s(stream)),
           "mgq_grouped_gemm_fwd_swiglu")


def grouped_gemm_dgrad_dswiglu(dY: Operand, W2: Operand, scaling, offsets, E, R_cap, H, F, gu, q: QDesc, dh=None,
                               dgu=None, stream=None):
    """Down-projection dgrad with dSwiGLU + row-wise quantisation of [dG | dU]
    in its epilogue, per tensor or MX (MX: also the column-wise copy when q has
    one; dh [R_cap, F] and dgu [R_cap, 2F] bf16 only when given)."""
    _check(load().mgq_grouped_gemm_dgrad_dswiglu(ctypes.byref(dY), ctypes.byref(W2), scaling, _p(offsets), E,
                                                 R_cap, H, F, _p(gu), ctypes.byref(q), _p(dh), _p(dgu), _s(stream)),
           "mgq_grouped_gemm_dgrad_dswiglu")


def swiglu_quantize(gu, R_cap, F, offsets, E, q: QDesc, h_out=None, stream=None):
    _check(load().mgq_swiglu_quantize(_p(gu), R_cap, F, _p(offsets), E, ctypes.byref(q), _p(h_out),
                                      _s(stream)), "mgq_swiglu_quantize")


def dswiglu_quantize(dh, gu, R_cap, F, offsets, E, q: QDesc, dgu_out=None, stream=None):
    _check(load().mgq_dswiglu_quantize(_p(dh), _p(gu), R_cap, F, _p(offsets), E, ctypes.byref(q),
                                       _p(dgu_out), _s(stream)), "mgq_dswiglu_quantize")


def moe_unpermute(y, row_id_map, probs, out, stream=None):
    T, k = row_id_map.shape
    H = out.shape[1]
    _check(load().mgq_moe_unpermute(_p(y), _p(row_id_map), _p(probs), T, k, H, _p(out), _s(stream)),
           "mgq_moe_unpermute")


def moe_unpermute_bwd(dout, y, row_id_map, src_row, probs, R_cap, offsets, E, q: QDesc, dprobs,
                      stream=None):
    T, k = row_id_map.shape
    H = dout.shape[1]
    _check(load().mgq_moe_unpermute_bwd(_p(dout), _p(y), _p(row_id_map), _p(src_row), _p(probs), T, k,
                                        H, R_cap, _p(offsets), E, ctypes.byref(q), _p(dprobs),
                                        _s(stream)), "mgq_moe_unpermute_bwd")


def moe_permute_bwd(da, row_id_map, dx, stream=None):
    T, k = row_id_map.shape
    H = dx.shape[1]
    _check(load().mgq_moe_permute_bwd(_p(da), _p(row_id_map), T, k, H, _p(dx), _s(stream)),
           "mgq_moe_permute_bwd")


def amax_history_update(history, head, amax, scale, fmax, stream=None):
    n, L = history.shape
    _check(load().mgq_amax_history_update(_p(history), _p(head), _p(amax), _p(scale), n, L,
                                          ctypes.c_float(fmax), _s(stream)), "mgq_amax_history_update")

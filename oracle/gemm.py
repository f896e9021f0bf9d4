"""Grouped GEMMs of the oracle (TEST INFRASTRUCTURE ONLY).

A grouped GEMM multiplies each expert's rows by that expert's weight in one
call over variable per-expert row counts ("--moe-grouped-gemm", Megatron-LM
issue #1152; ``grouped_mm`` behind dynamic quantisation, pytorch/ao PR #2275,
description). Its exact result is the matmul of the dequantised operands, so
the oracle is that definition in float64, one expert at a time:

* forward: Y_e = A_e W_e^T           (A [R_pad, K], W [E, N, K], Y [R_pad, N])
* dgrad:   dA_e = dY_e W_e           (dY [R_pad, N], W [E, N, K], dA [R_pad, K])
* wgrad:   dW_e = dY_e^T A_e         (dW [E, N, K], contraction over the rows
                                      of expert e)

Rows of expert e are [offsets[e], offsets[e+1]). Rows outside every group (the
tail of the buffer) are left at zero in Y / dA. An empty group gives no rows
and, in wgrad, an all-zero dW_e (or the accumulator unchanged when beta = 1:
the "gradient accumulation fusion" column of the coverage matrix in
Megatron-LM PR #5487).
"""
from __future__ import annotations

import numpy as np


def grouped_gemm_fwd(a, w, offsets):
    a = np.asarray(a, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    E, N, K = w.shape
    out = np.zeros((a.shape[0], N), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            out[lo:hi] = a[lo:hi] @ w[e].T
    return out


def grouped_gemm_dgrad(dy, w, offsets):
    dy = np.asarray(dy, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    E, N, K = w.shape
    out = np.zeros((dy.shape[0], K), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            out[lo:hi] = dy[lo:hi] @ w[e]
    return out


def grouped_gemm_wgrad(dy, a, offsets, E, beta=0.0, dw_in=None):
    dy = np.asarray(dy, dtype=np.float64)
    a = np.asarray(a, dtype=np.float64)
    N, K = dy.shape[1], a.shape[1]
    out = np.zeros((E, N, K), dtype=np.float64)
    if beta and dw_in is not None:
        out += beta * np.asarray(dw_in, dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            out[e] += dy[lo:hi].T @ a[lo:hi]
    return out


def sqnr_db(ref, q):
    """10 log10(|ref|^2 / |ref - q|^2): the quantised-vs-bf16 comparison of
    pytorch/ao PR #2275 (testing)."""
    ref = np.asarray(ref, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    num = np.sum(ref * ref)
    den = np.sum((ref - q) ** 2)
    return float("inf") if den == 0 else float(10.0 * np.log10(num / den))


def rel_frobenius(ref, got):
    """|ref - got|_F / |ref|_F (Frobenius norms over every element): the
    relative error behind the GEMM tolerances."""
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    n = np.linalg.norm(ref)
    d = np.linalg.norm(ref - got)
    return 0.0 if n == 0 and d == 0 else float(d / n)

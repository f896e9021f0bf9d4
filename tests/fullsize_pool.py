"""Worker pool of the full-size parity tests (test infrastructure).

At the workloads' full sizes the oracle has to quantise every weight (about
1.4 G elements for the Mixtral shapes) and every activation row, which takes
minutes in one process. This module spreads those oracle calls over the host
cores: the arrays sit in shared memory, each job takes one slice (rows of one
expert's weight, or a chunk of activation rows), runs the oracle's own
functions on it unchanged, compares the result with the GPU's bytes for that
slice, and returns the slice's float64 GEMM partial products for the sampled
rows. Nothing here computes any step of the method itself.

The pool uses the "spawn" start method, so it is safe to create after CUDA has
been initialised in the parent.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

_POOL = None


def workers() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def pool():
    global _POOL
    if _POOL is None:
        _POOL = mp.get_context("spawn").Pool(workers())
    return _POOL


class Shared:
    """A numpy array in shared memory, passed to jobs by name."""

    def __init__(self, arr: np.ndarray):
        arr = np.ascontiguousarray(arr)
        self.shm = shared_memory.SharedMemory(create=True, size=max(1, arr.nbytes))
        self.desc = (self.shm.name, arr.shape, arr.dtype.str)
        np.ndarray(arr.shape, arr.dtype, buffer=self.shm.buf)[...] = arr

    def close(self):
        self.shm.close()
        self.shm.unlink()

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


def _attach(desc):
    name, shape, dt = desc
    shm = shared_memory.SharedMemory(name=name)
    return shm, np.ndarray(shape, np.dtype(dt), buffer=shm.buf)


def _as_f64(a):
    from oracle import formats as OF
    if a.dtype == np.uint16:                       # bf16 bit patterns
        return OF.bf16_bits_to_f64(a)
    return a.astype(np.float64)


def weight_job(job):
    """One slice W[e, n0:n1, :] of a weight [E, N, K] (bf16 bits in shared
    memory), quantised by the oracle with `job["recipe"]`:
      "mx"      MXFP8 e4m3 row-wise (and, with "col", the column-wise copy
                quantize_mx(W^T) with blocks along N; n0, n1 multiples of 32)
      "blk"     128x128 float32 tiles (n0, n1 multiples of 128; with "col",
                the column-wise copy quantize_block_128x128(W^T))
      "nv"      NVFP4 1x16 with the expert's s_g
      "nv2d"    NVFP4 16x16 with the expert's s_g (row and column copies)
      "tensor"  per-tensor e4m3 with the expert's scale
    Compares the codes and scales with the GPU's (shared arrays, natural
    scale layout) and returns mismatch counts plus, when given sampled rows,
    fwd = A @ Wdeq[n0:n1]^T ([S, n1-n0]) and dgrad = dY[:, n0:n1] @ Wcol_deq^T
    ([S, K]; Wcol the column-wise copy where one exists)."""
    from oracle import quant as OQ
    e, n0, n1, rec = job["e"], job["n0"], job["n1"], job["recipe"]
    shms, views = [], {}
    for key, desc in job["shared"].items():
        s, v = _attach(desc)
        shms.append(s)
        views[key] = v
    try:
        w = _as_f64(views["w"][e, n0:n1])
        K = w.shape[1]
        out = {"mismatch": {}}

        def cmp(key, idx, want):
            if key not in views:
                out["mismatch"][key] = -1
                return
            got = views[key][idx]
            if got.shape != want.shape:
                raise ValueError(f"{key}: GPU slice {got.shape} against oracle {want.shape}")
            out["mismatch"][key] = int(np.count_nonzero(got != want))

        col_deq = None
        if rec == "mx":
            c, s = OQ.quantize_mx(w)
            cmp("codes", (e, slice(n0, n1)), c)
            cmp("scales", (e, slice(n0, n1)), s)
            deq = OQ.dequantize_mx(c, s)
            if job.get("col"):
                cc, cs = OQ.quantize_mx(np.ascontiguousarray(w.T))           # [K, n]
                cmp("col_codes", (e, slice(None), slice(n0, n1)), cc)
                cmp("col_scales", (e, slice(None), slice(n0 // 32, n1 // 32)), cs)
                col_deq = OQ.dequantize_mx(cc, cs)                          # [K, n]
        elif rec == "blk":
            c, si = OQ.quantize_block_128x128(w)
            cmp("codes", (e, slice(n0, n1)), c)
            cmp("scales", (e, slice(n0 // 128, n1 // 128)), si)
            deq = OQ.dequantize_block_128x128(c, si)
            if job.get("col"):
                cc, cs = OQ.quantize_block_128x128(np.ascontiguousarray(w.T))   # [K, n]
                cmp("col_codes", (e, slice(None), slice(n0, n1)), cc)
                cmp("col_scales", (e, slice(None), slice(n0 // 128, n1 // 128)), cs)
                col_deq = OQ.dequantize_block_128x128(cc, cs)
        elif rec == "nv":
            sg = np.float32(job["s_g"])
            c, s = OQ.quantize_nvfp4(w, sg)
            cmp("codes", (e, slice(n0, n1)), c)
            cmp("scales", (e, slice(n0, n1)), s)
            deq = OQ.dequantize_nvfp4(c, s, sg, K)
        elif rec == "nv2d":
            sg = np.float32(job["s_g"])
            rc, rs, cc, cs = OQ.quantize_nvfp4_2d(w, sg)
            cmp("codes", (e, slice(n0, n1)), rc)
            cmp("scales", (e, slice(n0, n1)), rs)
            cmp("col_codes", (e, slice(None), slice(n0 // 2, n1 // 2)), cc)
            cmp("col_scales", (e, slice(None), slice(n0 // 16, n1 // 16)), cs)
            deq = OQ.dequantize_nvfp4(rc, rs, sg, K)
            col_deq = OQ.dequantize_nvfp4(cc, cs, sg, n1 - n0)                # [K, n]
        elif rec == "tensor":
            sc = np.float32(job["scale"])
            c, _ = OQ.quantize_tensor(w, sc)
            cmp("codes", (e, slice(n0, n1)), c)
            deq = OQ.dequantize_tensor(c, sc)
        else:
            raise ValueError(rec)
        if job.get("a") is not None:
            out["fwd"] = job["a"] @ deq.T
        if job.get("dy") is not None:
            wc = deq.T if col_deq is None else col_deq                       # [K, n]
            out["dgrad"] = job["dy"] @ wc.T
        return out
    finally:
        for s in shms:
            s.close()


def rows_job(job):
    """Rows r0:r1 of an activation [M, C] in shared memory (bf16 bits, or
    float32 values), quantised row-wise by the oracle with `job["recipe"]`
    ("mx", "mx_e5m2", "blk", "blk_e5m2", "nv" with s_g, "tensor" / "tensor_e5m2" with a
    scale). Returns (codes, scales or None)."""
    from oracle import quant as OQ
    s, v = _attach(job["x"])
    try:
        x = _as_f64(v[job["r0"]:job["r1"]])
        rec = job["recipe"]
        if rec in ("mx", "mx_e5m2"):
            return OQ.quantize_mx(x, "e5m2" if rec == "mx_e5m2" else "e4m3")
        if rec in ("blk", "blk_e5m2"):
            return OQ.quantize_block_1x128(x, "e5m2" if rec == "blk_e5m2" else "e4m3")
        if rec == "nv":
            return OQ.quantize_nvfp4(x, np.float32(job["s_g"]))
        if rec in ("tensor", "tensor_e5m2"):
            return OQ.quantize_tensor(x, np.float32(job["scale"]), "e5m2" if rec == "tensor_e5m2" else "e4m3")[0], None
        raise ValueError(rec)
    finally:
        s.close()


def quantize_rows(x: np.ndarray, recipe: str, chunk: int = 2048, **kw):
    """Row-wise oracle quantisation of a large activation, in parallel chunks.
    Returns (codes, scales or None) for all rows."""
    with Shared(x) as sh:
        jobs = [dict(x=sh.desc, r0=r0, r1=min(r0 + chunk, x.shape[0]), recipe=recipe, **kw)
                for r0 in range(0, x.shape[0], chunk)]
        res = pool().map(rows_job, jobs)
    codes = np.concatenate([r[0] for r in res]) if res else np.zeros((0,), np.uint8)
    scales = None if (not res or res[0][1] is None) else np.concatenate([r[1] for r in res])
    return codes, scales


def weight_sweep(w_bits: np.ndarray, recipe: str, *, gpu: dict | None = None, a_rows: dict | None = None,
                 dy_rows: dict | None = None, chunk: int = 2048, col: bool = False, per_expert: dict | None = None):
    """Runs weight_job over every expert and every `chunk` rows of N.

    w_bits   [E, N, K] uint16 bf16 bits
    gpu      GPU bytes to compare: "codes" [E, N, K(/2)], "scales" natural
             layout, "col_codes" [E, K, N(/2)], "col_scales" [E, K, N/b]
    a_rows   {e: [S_e, K] float64} sampled forward rows (dequantised)
    dy_rows  {e: [S_e, N] float64} sampled dgrad rows (dequantised)
    per_expert {"s_g": [E]} or {"scale": [E]}
    Returns (mismatch totals per key, {e: fwd [S_e, N]}, {e: dgrad [S_e, K]})."""
    E, N, K = w_bits.shape
    shared = {"w": Shared(w_bits)}
    for key, arr in (gpu or {}).items():
        shared[key] = Shared(arr)
    try:
        descs = {k: s.desc for k, s in shared.items()}
        jobs = []
        for e in range(E):
            for n0 in range(0, N, chunk):
                n1 = min(n0 + chunk, N)
                j = dict(e=e, n0=n0, n1=n1, recipe=recipe, shared=descs, col=col)
                if a_rows is not None and e in a_rows and len(a_rows[e]):
                    j["a"] = a_rows[e]
                if dy_rows is not None and e in dy_rows and len(dy_rows[e]):
                    j["dy"] = dy_rows[e][:, n0:n1]
                for key, vals in (per_expert or {}).items():
                    j[key] = float(vals[e])
                jobs.append(j)
        res = pool().map(weight_job, jobs)
    finally:
        for s in shared.values():
            s.close()
    totals, fwd, dgrad = {}, {}, {}
    for j, r in zip(jobs, res):
        for key, n in r["mismatch"].items():
            if n >= 0:
                totals[key] = totals.get(key, 0) + n
        e = j["e"]
        if "fwd" in r:
            fwd.setdefault(e, np.zeros((r["fwd"].shape[0], N)))[:, j["n0"]:j["n1"]] = r["fwd"]
        if "dgrad" in r:
            dgrad[e] = dgrad.get(e, 0) + r["dgrad"]
    return totals, fwd, dgrad

"""Benchmark of the low-precision MoE expert layer (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: quantisation of the
grouped weights, the forward (permute + quantise, gate/up grouped GEMM,
SwiGLU + quantise, down grouped GEMM, unpermute) and, for the training
workload, the backward (unpermute backward + quantise, dgrad and wgrad of both
GEMMs, dSwiGLU + quantise, permute backward) and the delayed-scaling update.
The default workload is the Mixtral-8x7B-shaped layer, forward + backward
(8 experts, top-2, 16384 tokens, hidden 4096, ffn 14336, hybrid e4m3/e5m2,
delayed scaling with a 1024-long amax history).

metric: grouped-GEMM TFLOP/s of the step (algorithmic GEMM FLOPs of the
unpadded rows / step time). The GEMM kernel's own roofline fraction, the
memory-bound kernels' GB/s, an end-to-end figure through host buffers and the
CPU oracle on a bounded sample are reported beside it.

--impl reference times the CPU oracle (the only reference implementation of
this method) on the host cores, on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own replica of the layer (the path
has no exchange step on one node); value = work of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

# Fallback peaks of this GPU pool (earlier GB300 measurement) when the measured
# file is absent; FP8 dense = bf16 x 2 (nominal 4.5 / 2.25 PFLOP/s).
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0
FP4_OVER_BF16 = 6.0   # nominal dense 13.5 / 2.25 PFLOP/s


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        src = "measured"
        out = {}
        for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            v = d.get(key)
            if isinstance(v, dict):
                v = v.get("value")
            out[key] = float(v) if v else FALLBACK[key]
        return out, src
    return dict(FALLBACK), "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = f"/tmp/mgq_clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- the layer step

class Step:
    """Inputs resident on the device + the layer; one call = one step."""

    def __init__(self, w, dev, time_kernels=False):
        from fp8_grouped_gemm_gb300 import layer as L
        from fp8_grouped_gemm_gb300 import workloads as W
        self.w = w
        self.dev = dev
        self.lay = L.ExpertLayer(w, dev)
        self.train = self.lay.train
        x = W.make_activations(w)
        idx, probs = W.make_routing(w)
        self.x = x.to(dev)
        self.idx = torch.from_numpy(idx).to(dev)
        self.probs = torch.from_numpy(probs).to(dev)
        # weights drawn on the device (same distribution, seeded) to keep start-up short
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed * 1000 + 4)
        self.w1 = (torch.randn(w.E, 2 * w.F, w.H, generator=g, device=dev, dtype=torch.float32) * 0.02).to(
            torch.bfloat16)
        self.w2 = (torch.randn(w.E, w.H, w.F, generator=g, device=dev, dtype=torch.float32) * 0.02).to(
            torch.bfloat16)
        self.dout = W.make_dout(w).to(dev) if self.train else None
        self.time_kernels = time_kernels
        self.events = []
        self.ops = None

    def __call__(self):
        if self.ops is None:
            self.ops = self.lay.step_ops(self.w1, self.w2, self.x, self.idx, self.probs, self.dout)
        if not self.time_kernels:
            for _, op in self.ops:
                op()
            return
        # the same sequence, with events around every launch group
        ev = {}
        for name, op in self.ops:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            op()
            b.record()
            ev.setdefault(name, []).append((a, b))
        self.events.append(ev)


def algorithmic_bytes(w, R_pad, cols):
    if w.recipe == "nvfp4":
        return algorithmic_bytes_nvfp4(w)
    return algorithmic_bytes_fp8(w, R_pad, cols)


def algorithmic_bytes_nvfp4(w):
    """NVFP4: codes are 0.5 byte per element plus one scale byte per 16; the
    tensor amax passes re-read their input once, and the two-pass casts
    (SwiGLU, dSwiGLU) write their bf16 result and read it back. Training adds
    the column-wise copies."""
    T, k, H, F, E = w.T, w.k, w.H, w.F, w.E
    R = T * k
    q = 0.5 + 1.0 / 16
    c = 1 if w.backward else 0
    b = {"permute_quant": T * H * 2 * 2 + (1 + c) * R * H * q,
         "swiglu_quant": R * 2 * F * 2 + R * F * 2 * 2 + (1 + c) * R * F * q,
         "unpermute": R * H * 2 + T * H * 2,
         "weight_quant": E * 3 * F * H * 2 * 2 + (1 + c) * E * 3 * F * H * q}
    if w.backward:
        b["unpermute_bwd_quant"] = T * H * 2 * 2 + R * H * 2 + (1 + c) * R * H * q
        b["dswiglu_quant"] = R * F * 2 + R * 2 * F * 2 + R * 2 * F * 2 * 2 + (1 + c) * R * 2 * F * q
        b["permute_bwd"] = R * H * 2 + T * H * 2
    return b


def algorithmic_bytes_fp8(w, R_pad, cols):
    """Compulsory HBM bytes of the memory-bound steps: each input read once,
    each output written once (a row quantised once per token is written k
    times). A quantised output is one byte per element plus, with MX scaling,
    one E8M0 byte per 32 (blockwise: a float32 per 128); `cols` adds the column-wise copies (MX training;
    per-tensor scaling reads the row-wise codes MN-major and writes none)."""
    T, k, H, F, E = w.T, w.k, w.H, w.F, w.E
    R = T * k
    # MX: one E8M0 byte per 32; blockwise: one float32 per 128 (activations)
    # or per 128x128 tile (weights)
    q = 1 + 1 / 32 if w.recipe in ("mxfp8", "blockwise") else 1
    qw = 1 + 4 / (128 * 128) if w.recipe == "blockwise" else q
    c = 1 if cols else 0
    b = {}
    b["permute_quant"] = T * H * 2 + (1 + c) * R * H * q
    b["swiglu_quant"] = R * 2 * F * 2 + (1 + c) * R * F * q
    b["unpermute"] = R * H * 2 + T * H * 2
    b["weight_quant"] = E * 3 * F * H * 2 + (1 + c) * E * 3 * F * H * qw
    if w.backward:
        b["unpermute_bwd_quant"] = T * H * 2 + R * H * 2 + (1 + c) * R * H * q
        b["dswiglu_quant"] = R * F * 2 + R * 2 * F * 2 + (1 + c) * R * 2 * F * q
        b["permute_bwd"] = R * H * 2 + T * H * 2
    return b


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_sample(w, rows=512, f_slice=1024):
    """Times the CPU oracle on a bounded sample of the workload: one expert,
    `rows` routed rows, the full hidden size, an `f_slice`-wide slice of the
    FFN; the same chain of steps as the GPU step. Returns (seconds, GEMM FLOPs
    of the sample)."""
    from oracle import gemm as OG
    from oracle import layer as OL
    from oracle import quant as OQ
    from oracle import routing as OR
    rng = np.random.default_rng(w.seed)
    H, Fs = w.H, f_slice
    x = rng.standard_normal((rows, H))
    if w.outlier_frac:
        x[:, :max(1, int(round(w.outlier_frac * H)))] *= w.outlier_mult
    from oracle.formats import round_to_bf16
    x = round_to_bf16(x)
    w1 = round_to_bf16(rng.standard_normal((1, 2 * Fs, H)) * 0.02)
    w2 = round_to_bf16(rng.standard_normal((1, H, Fs)) * 0.02)
    dout = round_to_bf16(rng.standard_normal((rows, H)) * w.dout_std)
    off = np.array([0, rows])
    idx = np.zeros((rows, 1), dtype=np.int32)
    probs = np.ones((rows, 1), dtype=np.float32)
    t0 = time.perf_counter()
    rim, src, o2, cnt = OR.permute_indices(idx, 1, 128)
    s = np.float32(1.0)

    def q_nv(a):
        s_g = OQ.nvfp4_global_scale(float(np.max(np.abs(a))))
        c, sc = OQ.quantize_nvfp4(a, s_g)
        return OQ.dequantize_nvfp4(c, sc, s_g, a.shape[1])

    def q_act(a):
        if w.recipe == "nvfp4":
            return q_nv(a)
        if w.recipe == "mxfp8":
            c, sc = OQ.quantize_mx(a)
            return OQ.dequantize_mx(c, sc)
        if w.recipe == "blockwise":
            c, sc = OQ.quantize_block_1x128(a)
            return OQ.dequantize_block_1x128(c, sc)
        c, _ = OQ.quantize_tensor(a, s)
        return OQ.dequantize_tensor(c, s)

    def q_w(b):
        if w.recipe == "blockwise":
            c, sc = OQ.quantize_block_128x128(b)
            return OQ.dequantize_block_128x128(c, sc)
        if w.recipe == "nvfp4" and w.backward:        # 16x16 weight blocks
            s_g = OQ.nvfp4_global_scale(float(np.max(np.abs(b))))
            rc, rs, _, _ = OQ.quantize_nvfp4_2d(b, s_g)
            return OQ.dequantize_nvfp4(rc, rs, s_g, b.shape[1])
        return q_act(b)

    xd, w1d, w2d = q_act(x), q_w(w1[0])[None], q_w(w2[0])[None]
    gu = round_to_bf16(OG.grouped_gemm_fwd(xd, w1d, off))
    h = round_to_bf16(OL.swiglu(gu, Fs))
    hd = q_act(h)
    y = round_to_bf16(OG.grouped_gemm_fwd(hd, w2d, off))
    OR.unpermute(y, rim, probs)
    flops = 2.0 * rows * H * 2 * Fs + 2.0 * rows * Fs * H
    if w.backward:
        def q_grad(a):
            if w.recipe == "nvfp4":          # row-wise copy for dgrad, column-wise for wgrad
                return q_nv(a), q_nv(np.ascontiguousarray(a.T)).T
            if w.recipe == "mxfp8":          # row-wise copy for dgrad, column-wise for wgrad
                c, sc = OQ.quantize_mx(a, "e5m2")
                ct, st = OQ.quantize_mx(a.T, "e5m2")
                return OQ.dequantize_mx(c, sc, "e5m2"), OQ.dequantize_mx(ct, st, "e5m2").T
            c, _ = OQ.quantize_tensor(a, s, "e5m2")
            d = OQ.dequantize_tensor(c, s, "e5m2")
            return d, d

        dy32, _ = OR.unpermute_bwd(dout, y, rim, probs, rows)
        dy_r, dy_c = q_grad(dy32.astype(np.float64))
        dh = round_to_bf16(OG.grouped_gemm_dgrad(dy_r, w2d, off))
        OG.grouped_gemm_wgrad(dy_c, hd, off, 1)
        dgu = round_to_bf16(OL.dswiglu(dh, gu, Fs))
        d1_r, d1_c = q_grad(dgu)
        dxp = round_to_bf16(OG.grouped_gemm_dgrad(d1_r, w1d, off))
        OG.grouped_gemm_wgrad(d1_c, xd, off, 1)
        OR.permute_bwd(dxp, rim)
        flops *= 3
    return time.perf_counter() - t0, flops


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- main

GEMM_SOURCES = ("fp8_grouped_gemm_gb300/csrc/gemm.cu", "fp8_grouped_gemm_gb300/csrc/ptx_sm100.cuh",
                "fp8_grouped_gemm_gb300/csrc/device_common.cuh", "fp8_grouped_gemm_gb300/csrc/mgq_internal.h")


def measured_gemm_traffic(workload: str):
    """Mean DRAM bytes per grouped-GEMM launch from the committed ncu summary of
    this workload, if the GEMM sources are still the ones it measured; else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"grouped_gemm_dram_traffic_{workload}.md")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            if line.startswith("traffic_record:"):
                rec = dict(kv.split("=", 1) for kv in line.split()[1:])
    h = hashlib.sha256()
    for src in GEMM_SOURCES:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if rec.get("sources_sha256") != h.hexdigest():
        return None
    return {"bytes_per_launch": int(rec["bytes_per_launch"]),
            "algorithmic_bytes_per_launch": int(rec["algorithmic_bytes_per_launch"]),
            "source": f"stored ncu capture (profiles/{os.path.basename(path)}; {rec.get('case', 'see file')}), "
                      "valid for the current GEMM sources; not measured in this run"}


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (x itself without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_rank_step: float, world: int, ms_step: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica of the step (weak
    scaling), so the job does world x the work in the slowest rank's time."""
    return flops_per_rank_step * world / (ms_step * 1e-3) / 1e12


def run_reference(args, w, rank, world):
    """The CPU oracle, timed on the host cores, one bounded sample per step."""
    if rank != 0:
        return
    ncores = cpu_threads()
    for _ in range(args.warmup):
        oracle_sample(w, rows=128, f_slice=256)
    times, flops = [], 0.0
    for _ in range(args.steps):
        dt, flops = oracle_sample(w, *REF_SAMPLE)
        times.append(dt)
    tot = sum(times)
    value = flops * args.steps / tot / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(w),
        "data": "synthetic", "config": config_of(w, args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": ncores, "kind": "oracle",
                         "sample": sample_desc(*REF_SAMPLE)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "grouped FP8 GEMM fwd+bwd TFLOP/s (Mixtral-shaped expert layer step)"
DTYPE = {"mxfp8": "e4m3 fwd / e5m2 grads (MXFP8: E8M0 per 32, f32 accumulate)", "delayed": "e4m3/e5m2 (per-tensor delayed, f32 accumulate)",
         "blockwise": "e4m3 (1x128 / 128x128 float32 block scales, f32 accumulate)",
         "nvfp4": "e2m1 (NVFP4: 16-element ue4m3 scales + float32 global scale, f32 accumulate)"}
def dtype_of(w):
    if w.recipe == "mxfp8" and not w.backward:
        return "e4m3 (MXFP8: E8M0 per 32, f32 accumulate)"
    if w.recipe == "blockwise" and w.backward:
        return ("e4m3 fwd / e5m2 grads (blockwise float32 scales: 1x128 rows, 128x1 columns, 128x128 weight "
                "tiles; f32 accumulate)")
    if w.recipe == "nvfp4" and w.backward:
        return ("e2m1 fwd and grads (NVFP4: 16-element ue4m3 scales + float32 global scale, weights in 16x16 "
                "blocks, f32 accumulate)")
    return DTYPE[w.recipe]


def sample_desc(rows, f_slice):
    return (f"CPU oracle (numpy, float64 GEMMs) on one expert, {rows} routed rows, full hidden size, "
            f"a {f_slice}-wide FFN slice; same step chain as the GPU step; TFLOP/s = sample GEMM FLOPs / wall time")


REF_SAMPLE = (512, 1024)        # per --impl reference step (about a second on 16 cores)
CPU_BASELINE_SAMPLE = (2048, 2048)  # the cpu_baseline of our own line (about 10 s)


def config_of(w, args):
    return {"workload": f"{w.name}: E={w.E} top-{w.k} T={w.T} H={w.H} F={w.F} SwiGLU, recipe={w.recipe}"
                        + (", fwd+bwd" if w.backward else ", fwd"),
            "experts": w.E, "topk": w.k, "tokens": w.T, "hidden": w.H, "ffn": w.F,
            "parallelism": f"replicas x{args.gpus}",
            "l2": "inputs larger than L2 (bf16 weights 2.8 GB resident, re-quantised every step)"}


def gemm_roofline(w, gemm_ms, pk, pk_src):
    """Algorithmic GEMM FLOP/s of the step's grouped-GEMM launches against the
    burst tensor peak (the kernels run in a loop well under a second long),
    with the sustained fraction beside it."""
    flops = w.gemm_flops()
    achieved = flops / (gemm_ms * 1e-3) / 1e12
    ratio = FP4_OVER_BF16 if w.recipe == "nvfp4" else FP8_OVER_BF16
    kind = "fp4" if w.recipe == "nvfp4" else "fp8"
    peak = pk["bf16_tflops"] * ratio
    peak_sus = pk["bf16_tflops_sustained"] * ratio
    return {"bound": "tensor", "kernel": "grouped GEMM (all grouped GEMM launches of the step)",
            "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "frac_of_sustained": achieved / peak_sus,
            "peak_source": f"{pk_src}: bf16 burst {pk['bf16_tflops']} TFLOP/s x {ratio:g} ({kind}/bf16 nominal); "
                           f"frac_of_sustained uses bf16 sustained {pk['bf16_tflops_sustained']} x {ratio:g}",
            "gemm_ms_per_step": gemm_ms}


def hbm_table(w, per, lay, pk):
    R_pad = int(lay.offsets[-1].item())
    ab = algorithmic_bytes(w, R_pad, cols=lay.train and not lay.mn)
    return {k: {"ms": per[k], "GB/s": ab[k] / (per[k] * 1e-3) / 1e9,
                "frac": ab[k] / (per[k] * 1e-3) / 1e9 / pk["hbm_gbs"], "bytes": ab[k]} for k in ab if k in per}


def kernel_times(step, steps):
    """ms per step of every named op, from CUDA events around each launch
    group (on the launching stream) over `steps` further steps."""
    kstep = Step.__new__(Step)
    kstep.__dict__.update(step.__dict__)
    kstep.time_kernels = True
    kstep.events = []
    for _ in range(steps):
        kstep()
    torch.cuda.synchronize()
    per = {}
    for ev in kstep.events:
        for name, pairs in ev.items():
            per.setdefault(name, 0.0)
            per[name] += sum(a.elapsed_time(b) for a, b in pairs)
    return {k: v / steps for k, v in per.items()}


def e2e_run(step, flops, world, steps, barrier):
    """End to end through host buffers: every step copies its inputs from
    pinned host memory and reads its results back: the forward output, and
    for training also dX and dprobs (the weight gradients stay on the device,
    where an optimizer would consume them). The copies run on a second
    stream, pipelined with the compute: step i computes on input set i % 2
    while the copy stream reads back step i - 1's results and fills the other
    set for step i + 1. A step starts once its inputs have landed; the first
    op that rewrites a result (the unpermute) waits until the previous results
    have been read out. All copies of the timed steps lie inside the timed
    region (the first starts after its opening event, and the closing event
    waits for the last read-back)."""
    lay = step.lay
    hx = step.x.cpu().pin_memory()
    hidx = step.idx.cpu().pin_memory()
    hp = step.probs.cpu().pin_memory()
    hd = step.dout.cpu().pin_memory() if step.train else None
    res_dev = [lay.out] + ([lay.dx, lay.dprobs] if step.train else [])
    hres = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in res_dev]
    h2d = hx.numel() * 2 + hidx.numel() * 4 + hp.numel() * 4 + (hd.numel() * 2 if hd is not None else 0)
    d2h = sum(r.numel() * r.element_size() for r in hres)
    sets = [(step.x, step.idx, step.probs, step.dout),
            tuple(None if t is None else torch.empty_like(t) for t in (step.x, step.idx, step.probs, step.dout))]
    ops = [step.ops, step.lay.step_ops(step.w1, step.w2, *sets[1])]
    wr = [n for n, _ in ops[0]].index("unpermute")
    cur, cs = torch.cuda.current_stream(), torch.cuda.Stream()
    landed = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    read_out = torch.cuda.Event()

    def h2d_into(si):                       # on the copy stream
        x_, i_, p_, d_ = sets[si]
        x_.copy_(hx, non_blocking=True)
        i_.copy_(hidx, non_blocking=True)
        p_.copy_(hp, non_blocking=True)
        if d_ is not None:
            d_.copy_(hd, non_blocking=True)
        landed[si].record(cs)

    def run(n):
        """n pipelined steps on `cur` (the copy stream starts after `cur`'s current point)."""
        start = torch.cuda.Event()
        start.record(cur)
        cs.wait_event(start)
        with torch.cuda.stream(cs):
            h2d_into(0)
            if n > 1:
                h2d_into(1)
        for i in range(n):
            si = i % 2
            cur.wait_event(landed[si])
            for j, (_, op) in enumerate(ops[si]):
                if j == wr and i > 0:
                    cur.wait_event(read_out)
                op()
            done[si].record(cur)
            cs.wait_event(done[si])
            with torch.cuda.stream(cs):
                for h, r in zip(hres, res_dev):
                    h.copy_(r, non_blocking=True)
                read_out.record(cs)
                if i + 2 < n:
                    h2d_into(si)
        cur.wait_event(read_out)

    run(2)
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    run(steps)
    b.record()
    barrier()
    ems = a.elapsed_time(b) / steps
    return {"value": flops * world / (ems * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ems, "copies": "pipelined on a second stream",
            "read_back": "out" + (", dX, dprobs (dW stays on the device)" if step.train else "")}


def measure(w, dev, world, steps, warmup, barrier, local, with_e2e=False):
    """One workload: `warmup` untimed steps, then `steps` timed steps between
    barriers, clocks sampled meanwhile; then the per-kernel event timing and,
    if asked, the end-to-end run. Returns the record and the Step."""
    from fp8_grouped_gemm_gb300 import mgq
    step = Step(w, dev)
    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    if mgq.get_error() != mgq.OK:
        raise RuntimeError(f"{w.name}: device error in the warm-up steps")
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        step()
    t1.record()
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), dev if world > 1 else None)
    ms_step = ms / steps
    flops = w.gemm_flops()
    per = kernel_times(step, steps)
    pk, pk_src = peaks()
    gemm_ms = sum(v for k, v in per.items() if k.startswith("gemm"))
    rec = {"ms_per_step": ms_step, "value": job_value(flops, world, ms_step), "unit": "TFLOP/s",
           "steps": steps, "warmup": max(3, warmup), "dtype": dtype_of(w), "config": None,
           "roofline": gemm_roofline(w, gemm_ms, pk, pk_src), "hbm_kernels": hbm_table(w, per, step.lay, pk),
           "hbm_peak": {"GB/s": pk["hbm_gbs"], "source": pk_src}, "kernel_ms_per_step": per,
           "gpu_launches": step.lay.gpu_launches_per_step() * steps, "clocks": clk}
    if with_e2e:
        rec["e2e"] = e2e_run(step, flops, world, steps, barrier)
    if mgq.get_error() != mgq.OK:
        raise RuntimeError(f"{w.name}: device error in the timed steps")
    return rec, step


# the other configurations, each measured briefly in the same run beside the
# headline (same timing rules; no end-to-end or CPU legs)
OTHER_WORKLOADS = ("tiny", "mixtral_fwd", "scout_fwd", "finegrained_fwd", "mixtral_fwdbwd_mx",
                   "mixtral_fwdbwd_nvfp4", "scout_fwdbwd")
OTHER_STEPS = 20


def oracle_memory_steps(w, x, idx, probs):
    """The oracle's memory-bound steps timed on the host cores, as algorithmic
    GB/s by the byte counts the GPU kernels are measured with: permute +
    quantise and the unpermute at the workload's full token count (its own X
    and routing), the weight quantisation on 2048 rows of one expert's W1."""
    from oracle import quant as OQ
    from oracle import routing as OR
    from oracle.formats import round_to_bf16
    x64 = x.float().numpy().astype(np.float64)
    T, H = x64.shape
    k, E = w.k, w.E

    def quant(a):
        if w.recipe == "mxfp8":
            return OQ.quantize_mx(a)
        if w.recipe == "blockwise":
            return OQ.quantize_block_1x128(a)
        if w.recipe == "nvfp4":
            return OQ.quantize_nvfp4(a, OQ.nvfp4_global_scale(float(np.max(np.abs(a)))))
        return OQ.quantize_tensor(a, np.float32(1.0))

    q = 1.0 if w.recipe == "delayed" else (0.5 + 1 / 16 if w.recipe == "nvfp4" else 1 + 1 / 32)
    out = {}
    t = time.perf_counter()
    rim, src, off, cnt = OR.permute_indices(idx, E, 128)
    Rp = int(off[-1])
    codes = quant(x64)[0]
    OR.permute_rows(codes, rim, Rp)
    dt = time.perf_counter() - t
    out["permute_quant"] = {"GB/s": (T * H * 2 + T * k * H * q) / dt / 1e9, "seconds": dt,
                            "sample": f"full size: {T} tokens x {H}, top-{k} of {E}"}
    y = OR.permute_rows(x64, rim, Rp)
    t = time.perf_counter()
    OR.unpermute(y, rim, probs)
    dt = time.perf_counter() - t
    out["unpermute"] = {"GB/s": (T * k * H * 2 + T * H * 2) / dt / 1e9, "seconds": dt,
                        "sample": f"full size: {T} tokens x {H}, top-{k}"}
    rng = np.random.default_rng(w.seed)
    wslice = round_to_bf16(rng.standard_normal((2048, H)) * 0.02)
    t = time.perf_counter()
    if w.recipe == "blockwise":
        OQ.quantize_block_128x128(wslice)
    else:
        quant(wslice)
    dt = time.perf_counter() - t
    out["weight_quant"] = {"GB/s": 2048 * H * (2 + q) / dt / 1e9, "seconds": dt,
                           "sample": f"2048 x {H} rows of one expert's W1"}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="mixtral_fwdbwd")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the token count (small cases for profiler captures)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the expert count (small cases for profiler captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="measure only the named workload (no `workloads` entries)")
    args = ap.parse_args()
    from fp8_grouped_gemm_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    small = {}
    if args.tokens:
        small["T"] = args.tokens
    if args.experts:
        small["E"] = args.experts
    if small:
        w = w.scaled(**small)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from fp8_grouped_gemm_gb300 import mgq
    mgq.load()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    rec, step = measure(w, dev, world, args.steps, args.warmup, barrier, local, with_e2e=not args.no_e2e)
    # the headline's own inputs, for the oracle's memory steps (CPU leg below)
    oracle_inputs = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        oracle_inputs = (step.x.cpu(), step.idx.cpu().numpy(), step.probs.cpu().numpy())
    roofline = rec["roofline"]
    tr = measured_gemm_traffic(w.name) if not small else None
    roofline["traffic"] = tr["bytes_per_launch"] if tr else None
    if tr:
        roofline["algorithmic_bytes_per_launch"] = tr["algorithmic_bytes_per_launch"]
        roofline["traffic_source"] = tr["source"]
    del step
    torch.cuda.empty_cache()

    others = {}
    if not args.no_others and not small:
        for name in OTHER_WORKLOADS:
            if name == w.name:
                continue
            ow = WORKLOADS[name]
            orec, ostep = measure(ow, dev, world, min(args.steps, OTHER_STEPS), args.warmup, barrier, local)
            orec["config"] = config_of(ow, args)
            orec["metric"] = ("grouped GEMM TFLOP/s of the step (" + ("fwd+bwd" if ow.backward else "fwd")
                              + ", algorithmic FLOPs of the unpadded rows)")
            others[name] = orec
            del ostep
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, f = oracle_sample(w, *CPU_BASELINE_SAMPLE)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": sample_desc(*CPU_BASELINE_SAMPLE), "seconds": dt,
               # the whole step's GEMMs at the sample's rate: extrapolated, not run
               "gemm_full_step_seconds_extrapolated": w.gemm_flops() / (f / dt),
               "memory_steps": oracle_memory_steps(w, *oracle_inputs)}
        for k_, v in cpu["memory_steps"].items():
            if k_ in rec["hbm_kernels"]:
                v["gpu_GB/s"] = rec["hbm_kernels"][k_]["GB/s"]
    if rank == 0:
        line = {
            "metric": METRIC, "value": rec["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(w),
            "data": "synthetic (seeded; shapes of the workload)",
            "config": config_of(w, args), "roofline": roofline, "hbm_kernels": rec["hbm_kernels"],
            "kernel_ms_per_step": rec["kernel_ms_per_step"], "cpu_baseline": cpu, "e2e": rec.get("e2e"),
            "gpu_launches": rec["gpu_launches"], "clocks": rec["clocks"], "workloads": others,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Seeded synthetic inputs of the expert-layer workloads.

This module only draws inputs: it holds none of the layer's arithmetic
(no quantisation, permutation, GEMM or activation). Both the CUDA path's
callers (tests, bench) and the CPU oracle's callers take their inputs from
here, so that both sides see identical data.

Workloads (shapes of the routed-expert layers the source pages discuss:
Mixtral 8x7B in Megatron-LM issue #1152, Llama4 in pytorch/ao PR #2275):

======================  ==  =  =====  ====  =====  =========  ===========
name                    E   k  T      H     F      routing    recipe
======================  ==  =  =====  ====  =====  =========  ===========
tiny                    4   2  1024   256   512    top-k      MXFP8 e4m3
mixtral_fwd             8   2  16384  4096  14336  top-k      MXFP8 e4m3
scout_fwd               16  1  16384  5120  8192   Zipf(1.2)  blockwise
finegrained_fwd         128 8  32768  2048  768    uniform    NVFP4
mixtral_fwdbwd          8   2  16384  4096  14336  top-k      delayed
mixtral_fwdbwd_mx       8   2  16384  4096  14336  top-k      MXFP8 (train)
mixtral_fwdbwd_nvfp4    8   2  16384  4096  14336  top-k      NVFP4 (train)
======================  ==  =  =====  ====  =====  =========  ===========

Draws: activations bf16(N(0,1)) (Mixtral shapes: 0.1% of the hidden channels,
chosen by a seeded permutation, multiplied by 50 before the bf16 rounding),
weights bf16(N(0,0.02)), router logits N(0,1) float32, output gradients
bf16(N(0,1e-3)). Top-k routing takes the k largest logits (ties to the lower
expert id) and softmax over the selected logits as probabilities. Zipf(1.2)
routing spreads T tokens over 14 of 16 experts with counts proportional to
rank^-1.2 (largest remainder), leaving 2 experts empty, probabilities 1.
Uniform routing gives each token k distinct experts uniformly at random and
softmax probabilities of N(0,1) logits at those experts.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cid: int
    E: int
    k: int
    T: int
    H: int
    F: int
    routing: str          # "topk" | "zipf" | "uniform"
    recipe: str           # "mxfp8" | "blockwise" | "nvfp4" | "delayed"
    backward: bool = False
    outlier_frac: float = 0.0
    outlier_mult: float = 50.0
    dout_std: float = 1e-3
    zipf_s: float = 1.2
    n_empty: int = 0
    history: int = 1024

    @property
    def seed(self) -> int:
        return 1234 + self.cid

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def R(self) -> int:
        return self.T * self.k

    def gemm_flops(self) -> float:
        """Algorithmic FLOPs of the grouped GEMMs of one step (unpadded rows):
        gate/up (H -> 2F) and down (F -> H), times 3 with backward."""
        fwd = 2.0 * self.R * self.H * (2 * self.F) + 2.0 * self.R * self.F * self.H
        return fwd * (3 if self.backward else 1)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 2, 1024, 256, 512, "topk", "mxfp8"),
    "mixtral_fwd": Workload("mixtral_fwd", 2, 8, 2, 16384, 4096, 14336, "topk", "mxfp8",
                            outlier_frac=0.001),
    "scout_fwd": Workload("scout_fwd", 3, 16, 1, 16384, 5120, 8192, "zipf", "blockwise",
                          n_empty=2),
    "finegrained_fwd": Workload("finegrained_fwd", 4, 128, 8, 32768, 2048, 768, "uniform",
                                "nvfp4"),
    "mixtral_fwdbwd": Workload("mixtral_fwdbwd", 5, 8, 2, 16384, 4096, 14336, "topk",
                               "delayed", backward=True, outlier_frac=0.001),
    # the same layer trained with MXFP8 block scales in both passes (e4m3
    # forward, e5m2 gradients; column-wise 32x1 requantisation for wgrad)
    "mixtral_fwdbwd_mx": Workload("mixtral_fwdbwd_mx", 5, 8, 2, 16384, 4096, 14336, "topk",
                                  "mxfp8", backward=True, outlier_frac=0.001),
    # and with NVFP4 in both passes (e2m1 with 16-element ue4m3 scales and a
    # float32 global scale per tensor; weights with 16x16 blocks, one
    # quantisation giving both copies; column-wise 16x1 blocks along tokens)
    "mixtral_fwdbwd_nvfp4": Workload("mixtral_fwdbwd_nvfp4", 5, 8, 2, 16384, 4096, 14336, "topk",
                                     "nvfp4", backward=True, outlier_frac=0.001),
    # the Scout-shaped experts trained with blockwise FP8 (e4m3 forward, e5m2
    # gradients; 1x128 row-wise and 128x1 column-wise activation / gradient
    # blocks, 128x128 weight tiles)
    "scout_fwdbwd": Workload("scout_fwdbwd", 3, 16, 1, 16384, 5120, 8192, "zipf", "blockwise",
                             backward=True, n_empty=2),
}


def _gen(seed: int, stream: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed * 1000 + stream)
    return g


def zipf_counts(T: int, n: int, s: float) -> np.ndarray:
    """Counts proportional to rank^-s over n ranks, summing to T (largest
    remainder, ties to the lower rank)."""
    p = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    raw = p * T
    c = np.floor(raw).astype(np.int64)
    rem = T - int(c.sum())
    order = np.argsort(-(raw - c), kind="stable")
    c[order[:rem]] += 1
    return c


def make_routing(w: Workload):
    """Returns (topk_idx int32 [T, k], probs float32 [T, k]) as numpy arrays."""
    rng = np.random.default_rng(w.seed)
    T, E, k = w.T, w.E, w.k
    if w.routing == "topk":
        logits = torch.randn(T, E, generator=_gen(w.seed, 1), dtype=torch.float32).numpy()
        idx = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        sel = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
        ex = np.exp(sel - sel.max(axis=1, keepdims=True))
        probs = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    elif w.routing == "zipf":
        assert k == 1
        n = E - w.n_empty
        counts = zipf_counts(T, n, w.zipf_s)
        experts = rng.permutation(E)[:n]           # rank r -> expert id
        assign = np.repeat(experts, counts)
        rng.shuffle(assign)
        idx = assign.reshape(T, 1)
        probs = np.ones((T, 1), dtype=np.float32)
    elif w.routing == "uniform":
        keys = rng.random((T, E))
        idx = np.argsort(keys, axis=1)[:, :k]
        logits = torch.randn(T, k, generator=_gen(w.seed, 1), dtype=torch.float32).numpy()
        ex = np.exp(logits.astype(np.float64) - logits.max(axis=1, keepdims=True))
        probs = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    else:
        raise ValueError(w.routing)
    return np.ascontiguousarray(idx.astype(np.int32)), np.ascontiguousarray(probs)


def make_activations(w: Workload) -> torch.Tensor:
    """X bf16 [T, H] on the CPU."""
    x = torch.randn(w.T, w.H, generator=_gen(w.seed, 2), dtype=torch.float32)
    if w.outlier_frac > 0:
        n = max(1, int(round(w.outlier_frac * w.H)))
        ch = torch.randperm(w.H, generator=_gen(w.seed, 3))[:n]
        x[:, ch] *= w.outlier_mult
    return x.to(torch.bfloat16)


def make_weights(w: Workload):
    """W1 bf16 [E, 2F, H] (gate rows then up rows) and W2 bf16 [E, H, F]."""
    w1 = torch.empty(w.E, 2 * w.F, w.H, dtype=torch.float32)
    w1.normal_(0.0, 0.02, generator=_gen(w.seed, 4))
    w2 = torch.empty(w.E, w.H, w.F, dtype=torch.float32)
    w2.normal_(0.0, 0.02, generator=_gen(w.seed, 5))
    return w1.to(torch.bfloat16), w2.to(torch.bfloat16)


def make_dout(w: Workload) -> torch.Tensor:
    d = torch.empty(w.T, w.H, dtype=torch.float32)
    d.normal_(0.0, w.dout_std, generator=_gen(w.seed, 6))
    return d.to(torch.bfloat16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a bf16 tensor (for the oracle's callers)."""
    return t.detach().to("cpu").float().numpy().astype(np.float64)


def randn_bf16(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    g = _gen(seed, 7)
    x = torch.empty(*shape, dtype=torch.float32)
    x.normal_(0.0, std, generator=g)
    return x.to(torch.bfloat16)

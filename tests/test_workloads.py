"""The seeded synthetic inputs follow their stated recipe (CPU only): Zipf(1.2)
expert loads by largest remainder with two empty experts for the Scout shape,
top-k routing with k distinct experts and renormalised probabilities, uniform
fine-grained routing, 0.1% outlier channels scaled by 50, and determinism."""
import numpy as np
import torch

from fp8_grouped_gemm_gb300 import workloads as W


def test_zipf_counts_largest_remainder():
    # 16384 tokens over 14 non-empty experts, p_r proportional to r^-1.2
    c = W.zipf_counts(16384, 14, 1.2)
    assert list(c) == [6153, 2678, 1646, 1166, 892, 717, 596, 507, 441, 388, 346, 312, 283, 259]
    assert c.sum() == 16384
    # the remainder goes to the largest fractional parts, one each
    p = np.arange(1, 15, dtype=np.float64) ** -1.2
    raw = p / p.sum() * 16384
    assert np.all(np.abs(c - raw) < 1.0)


def test_scout_routing_loads():
    w = W.WORKLOADS["scout_fwd"]
    idx, probs = W.make_routing(w)
    assert idx.shape == (w.T, 1) and np.all(probs == 1.0)
    loads = np.bincount(idx[:, 0], minlength=w.E)
    assert (loads == 0).sum() == 2
    assert sorted(loads[loads > 0], reverse=True) == list(W.zipf_counts(w.T, w.E - 2, 1.2))


def test_topk_routing_invariants():
    w = W.WORKLOADS["mixtral_fwd"].scaled(T=2048)
    idx, probs = W.make_routing(w)
    assert idx.shape == (2048, 2) and idx.dtype == np.int32
    assert np.all(idx[:, 0] != idx[:, 1]) and idx.min() >= 0 and idx.max() < w.E
    assert np.all(probs > 0) and np.allclose(probs.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(probs[:, 0] >= probs[:, 1])          # top-k by logit, descending
    # every expert gets a share near 1/E of the entries
    share = np.bincount(idx.ravel(), minlength=w.E) / idx.size
    assert np.all(np.abs(share - 1.0 / w.E) < 0.05)


def test_uniform_finegrained_routing():
    w = W.WORKLOADS["finegrained_fwd"].scaled(T=1024)
    idx, probs = W.make_routing(w)
    assert idx.shape == (1024, 8)
    assert all(len(set(row)) == 8 for row in idx.tolist())
    assert np.allclose(probs.sum(axis=1), 1.0, atol=1e-6)


def test_outlier_channels():
    w = W.WORKLOADS["mixtral_fwd"].scaled(T=256)
    x = W.make_activations(w).float()
    std = x.std(dim=0)
    n = int(round(0.001 * w.H))
    assert n == 4
    big = torch.nonzero(std > 10).flatten()
    assert big.numel() == n
    assert torch.all((std[big] > 35) & (std[big] < 65))
    assert torch.all(std[std <= 10] < 1.5)


def test_inputs_are_deterministic():
    w = W.WORKLOADS["tiny"]
    a1, p1 = W.make_routing(w)
    a2, p2 = W.make_routing(w)
    assert np.array_equal(a1, a2) and np.array_equal(p1, p2)
    assert torch.equal(W.make_activations(w), W.make_activations(w))
    w1, w2 = W.make_weights(w)
    v1, v2 = W.make_weights(w)
    assert torch.equal(w1, v1) and torch.equal(w2, v2)
    assert abs(w1.float().std().item() - 0.02) < 0.002

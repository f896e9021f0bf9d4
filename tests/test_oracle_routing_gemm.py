"""Pins of the oracle's permutation, grouped GEMMs and elementwise steps
(CPU only): brute force on tiny inputs, invariants, adjoint identities,
finite differences and exact small-integer GEMMs."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats as F
from oracle import gemm as G
from oracle import layer as L
from oracle import quant as Q
from oracle import routing as R


def _rand_topk(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("seed", range(12))
def test_permute_matches_bruteforce(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(0, 9))
    E = int(rng.integers(1, 6))
    k = int(rng.integers(1, E + 1))
    align = int(rng.choice([1, 2, 4, 32]))
    idx = _rand_topk(rng, T, E, k).reshape(T, k)
    a = R.permute_indices(idx, E, align)
    b = R.permute_indices_bruteforce(idx.tolist(), E, align)
    np.testing.assert_array_equal(a[0], np.array(b[0], dtype=np.int32).reshape(T, k))
    np.testing.assert_array_equal(a[1], np.array(b[1], dtype=np.int32))
    np.testing.assert_array_equal(a[2], np.array(b[2], dtype=np.int32))
    np.testing.assert_array_equal(a[3], np.array(b[3], dtype=np.int32))


def test_permute_invariants_with_empty_groups():
    rng = np.random.default_rng(1)
    T, E, k, align = 500, 9, 2, 32
    idx = _rand_topk(rng, T, 7, k)          # experts 7 and 8 stay empty
    rim, src, off, cnt = R.permute_indices(idx, E, align)
    assert cnt.sum() == T * k
    assert cnt[7] == 0 and cnt[8] == 0 and off[7] == off[8] == off[9]
    assert np.all(off % align == 0) and np.all(np.diff(off) >= cnt)
    assert np.all(src[rim.reshape(-1)] == np.arange(T * k))
    assert np.sum(src >= 0) == T * k
    # rows inside each group are in token order
    for e in range(E):
        rows = src[off[e]:off[e] + cnt[e]] // k
        assert np.all(np.diff(rows) > 0)
        assert np.all(src[off[e] + cnt[e]:off[e + 1]] == -1)


def test_permute_then_unpermute_is_identity():
    rng = np.random.default_rng(2)
    T, E, k, H = 64, 6, 3, 16
    idx = _rand_topk(rng, T, E, k)
    rim, src, off, cnt = R.permute_indices(idx, E, 8)
    x = rng.standard_normal((T, H))
    xp = R.permute_rows(x, rim, int(off[-1]))
    out = R.unpermute(xp, rim, np.full((T, k), 1.0 / k))
    np.testing.assert_allclose(out, x, rtol=1e-14, atol=1e-14)


def test_unpermute_bwd_is_the_gradient():
    """dY and dprobs against finite differences of the combine."""
    rng = np.random.default_rng(3)
    T, E, k, H = 6, 4, 2, 5
    idx = _rand_topk(rng, T, E, k)
    rim, src, off, cnt = R.permute_indices(idx, E, 2)
    Rp = int(off[-1])
    y = rng.standard_normal((Rp, H))
    probs = rng.random((T, k)).astype(np.float32).astype(np.float64)
    dout = rng.standard_normal((T, H)).astype(np.float32).astype(np.float64)
    dy32, dprobs = R.unpermute_bwd(dout, y, rim, probs, Rp)
    loss = lambda yy, pp: np.sum(dout * R.unpermute(yy, rim, pp))
    h = 1e-6
    for t in range(T):
        for j in range(k):
            pp = probs.copy(); pp[t, j] += h
            pm = probs.copy(); pm[t, j] -= h
            fd = (loss(y, pp) - loss(y, pm)) / (2 * h)
            assert abs(fd - dprobs[t, j]) < 1e-6
    for r in range(Rp):
        for c in range(H):
            yp = y.copy(); yp[r, c] += h
            ym = y.copy(); ym[r, c] -= h
            fd = (loss(yp, probs) - loss(ym, probs)) / (2 * h)
            assert abs(fd - dy32[r, c]) < 1e-5


def test_permute_bwd_is_adjoint():
    rng = np.random.default_rng(4)
    T, E, k, H = 40, 5, 2, 8
    idx = _rand_topk(rng, T, E, k)
    rim, src, off, cnt = R.permute_indices(idx, E, 4)
    Rp = int(off[-1])
    x = rng.standard_normal((T, H))
    g = rng.standard_normal((Rp, H))
    g[src < 0] = 0.0
    lhs = np.sum(R.permute_rows(x, rim, Rp) * g)
    rhs = np.sum(x * R.permute_bwd(g, rim))
    assert abs(lhs - rhs) < 1e-10


def _brute_matmul(a, b):
    """Exact sum of products with fractions (a [M,K] @ b [K,N])."""
    M, K = a.shape
    N = b.shape[1]
    out = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for kk in range(K):
                s += Fraction(float(a[i, kk])) * Fraction(float(b[kk, j]))
            out[i, j] = float(s)
    return out


def test_grouped_gemms_bruteforce():
    rng = np.random.default_rng(5)
    E, N, K = 3, 5, 7
    off = np.array([0, 4, 4, 9])                  # group 1 is empty
    a = F.decode(rng.integers(0, 0x7F, (9, K)), F.E4M3)
    w = F.decode(rng.integers(0, 0x7F, (E, N, K)), F.E4M3)
    dy = F.decode(rng.integers(0, 0x7B, (9, N)), F.E5M2)
    y = G.grouped_gemm_fwd(a, w, off)
    da = G.grouped_gemm_dgrad(dy, w, off)
    dw = G.grouped_gemm_wgrad(dy, a, off, E)
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if hi > lo:
            np.testing.assert_array_equal(y[lo:hi], _brute_matmul(a[lo:hi], w[e].T))
            np.testing.assert_array_equal(da[lo:hi], _brute_matmul(dy[lo:hi], w[e]))
            np.testing.assert_array_equal(dw[e], _brute_matmul(dy[lo:hi].T, a[lo:hi]))
        else:
            assert np.all(dw[e] == 0)
    # beta = 1 accumulates into the previous dW (empty group: unchanged)
    prev = rng.standard_normal((E, N, K))
    dw1 = G.grouped_gemm_wgrad(dy, a, off, E, beta=1.0, dw_in=prev)
    np.testing.assert_allclose(dw1, prev + dw, rtol=1e-13)
    np.testing.assert_array_equal(dw1[1], prev[1])


def test_grouped_equals_per_group_and_single_expert():
    rng = np.random.default_rng(6)
    E, N, K = 4, 8, 16
    off = np.array([0, 3, 3, 10, 12])
    a = rng.standard_normal((12, K))
    w = rng.standard_normal((E, N, K))
    y = G.grouped_gemm_fwd(a, w, off)
    for e in range(E):
        one = G.grouped_gemm_fwd(a[off[e]:off[e + 1]], w[e:e + 1], np.array([0, off[e + 1] - off[e]]))
        np.testing.assert_array_equal(y[off[e]:off[e + 1]], one)
    # all rows in one expert
    y1 = G.grouped_gemm_fwd(a, w, np.array([0, 0, 12, 12, 12]))
    np.testing.assert_allclose(y1, a @ w[1].T, rtol=1e-14)


def test_quantised_gemm_sqnr():
    """MXFP8 e4m3 x e4m3 forward on N(0,1) x N(0,0.02): the SQNR of pytorch/ao
    PR #2275's quantised-vs-bf16 check lands near 28-29 dB."""
    rng = np.random.default_rng(7)
    a = F.round_to_bf16(rng.standard_normal((256, 2048)))
    w = F.round_to_bf16(rng.standard_normal((1, 256, 2048)) * 0.02)
    ca, sa = Q.quantize_mx(a)
    cw, sw = Q.quantize_mx(w[0])
    ref = G.grouped_gemm_fwd(a, w, np.array([0, 256]))
    q = G.grouped_gemm_fwd(Q.dequantize_mx(ca, sa), Q.dequantize_mx(cw, sw)[None], np.array([0, 256]))
    s = G.sqnr_db(ref, q)
    assert 27.5 < s < 30.5, s


def test_swiglu_derivative_by_finite_differences():
    rng = np.random.default_rng(8)
    Fd = 6
    gu = rng.standard_normal((5, 2 * Fd)) * 3
    dh = rng.standard_normal((5, Fd))
    d = L.dswiglu(dh, gu, Fd)
    h = 1e-6
    for r in range(5):
        for c in range(2 * Fd):
            p = gu.copy(); p[r, c] += h
            m = gu.copy(); m[r, c] -= h
            fd = np.sum(dh * (L.swiglu(p, Fd) - L.swiglu(m, Fd))) / (2 * h)
            assert abs(fd - d[r, c]) < 1e-6 * max(1, abs(fd))


def test_silu_special_values():
    assert L.silu(np.array([0.0]))[0] == 0.0
    assert L.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)
    assert abs(L.silu(np.array([-40.0]))[0]) < 1e-15
    assert L.silu(np.array([1.0]))[0] == pytest.approx(1.0 / (1.0 + np.exp(-1.0)))


def test_delayed_scaling_window():
    ds = L.DelayedScaling("e4m3", length=4)
    assert ds.scale == 1.0
    ds.update(0.0)
    assert ds.scale == 1.0                 # max 0 keeps the scale
    ds.update(2.0)
    assert ds.scale == np.float32(224.0)   # 448 / 2
    for a in (1.0, 0.5, 0.25):
        ds.update(a)
    assert ds.scale == np.float32(224.0)   # 2.0 still in the last 4
    ds.update(0.125)
    assert ds.scale == np.float32(448.0)   # 2.0 dropped: max is 1.0
    ds5 = L.DelayedScaling("e5m2", length=1024)
    ds5.update(7.0)
    assert ds5.scale == np.float32(57344.0) / np.float32(7.0)


def test_zipf_counts_of_scout_workload():
    from fp8_grouped_gemm_gb300.workloads import WORKLOADS, make_routing, zipf_counts
    c = zipf_counts(16384, 14, 1.2)
    assert list(c) == [6153, 2678, 1646, 1166, 892, 717, 596, 507, 441, 388, 346, 312, 283, 259]
    w = WORKLOADS["scout_fwd"].scaled(T=2048)
    idx, probs = make_routing(w)
    cnt = np.bincount(idx[:, 0], minlength=16)
    assert np.sum(cnt == 0) == 2 and cnt.sum() == 2048 and np.all(probs == 1)


def test_rel_frobenius_closed_forms():
    """Relative Frobenius error |ref - got|_F / |ref|_F on hand-computed
    cases: a vector (0.3 / 2 = 0.15; without the square roots it would read
    0.0225) and a matrix whose spectral and Frobenius norms differ
    (0.5 / 5 = 0.1; the spectral norm would give 0.125)."""
    assert G.rel_frobenius(np.ones(4), np.ones(4) + np.array([0.3, 0, 0, 0])) == pytest.approx(0.15, rel=1e-15)
    ref = np.array([[3.0, 0.0], [0.0, 4.0]])
    got = ref + np.array([[0.0, 0.0], [0.0, 0.5]])
    assert G.rel_frobenius(ref, got) == pytest.approx(0.1, rel=1e-15)
    assert G.rel_frobenius(ref, ref) == 0.0
    assert G.rel_frobenius(np.zeros(3), np.zeros(3)) == 0.0


def test_sqnr_closed_forms():
    """SQNR = 10 log10(|ref|^2 / |ref - q|^2) (pytorch/ao PR #2275, testing):
    a uniform 10% error is 20 dB (a 20 log10 slip would give 40 dB), a 1%
    error 40 dB, and an exact result is infinite."""
    ref = np.linspace(-3.0, 5.0, 100)
    assert G.sqnr_db(ref, 1.1 * ref) == pytest.approx(20.0, abs=1e-12)
    assert G.sqnr_db(ref, 0.99 * ref) == pytest.approx(40.0, abs=1e-12)
    assert G.sqnr_db(ref, ref) == float("inf")

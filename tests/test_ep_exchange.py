"""Expert-parallel dispatch and combine in FP8 (CPU, two gloo ranks).

Each rank routes and quantises its own tokens (here with the oracle: the
permutation of "[BUG] Loss difference when training with FP8 vs. BF16 MoE",
Megatron-LM issue #1152, groups padded to 128 rows, and MX e4m3 codes with
E8M0 scales in their 128x4 tiles), then the exchange moves the quantised
rows to the ranks that own their experts. Checked on every rank against the
oracle's own per-rank buffers (every rank can rebuild every rank's seeded
inputs):
* received codes and scale tiles bit-exact, expert-major, source ranks in
  order, with the local group offsets;
* combine returns every expert output to the row it came from;
* the whole layer with expert parallelism (dispatch, each rank's experts on
  the received rows, combine, unpermute) equals the same layer on one rank.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import formats as OF
from oracle import quant as OQ
from oracle import routing as OR
from tests.layer_check import tile_mx_scales

E, K, H, WORLD = 8, 2, 256, 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_inputs(r):
    """Rank r's tokens, routing and probabilities (seeded by the rank);
    rank 1 routes nothing to expert 5 (an empty group)."""
    rng = np.random.default_rng(100 + r)
    T = 300 + 70 * r
    allowed = np.array([e for e in range(E) if not (r == 1 and e == 5)])
    idx = np.stack([rng.choice(allowed, size=K, replace=False) for _ in range(T)]).astype(np.int32)
    probs = rng.random((T, K)).astype(np.float32)
    x = OF.round_to_bf16(rng.standard_normal((T, H)))
    return x, idx, probs


def _rank_buffers(r):
    """Rank r's permuted MX codes [Rp, H], tiled scales, and routing."""
    x, idx, probs = _rank_inputs(r)
    rim, src, off, cnt = OR.permute_indices(idx, E, 128)
    Rp = int(off[-1])
    c, s = OQ.quantize_mx(x)
    codes = OR.permute_rows(c, rim, Rp)
    scales = tile_mx_scales(OR.permute_rows(s, rim, Rp))
    return codes, scales, off, rim, probs, x


def _expert_fn(e, v):
    """A stand-in for expert e's computation on dequantised rows: exact in
    float64 and in bf16 (a power-of-two scale per expert)."""
    return v * 2.0 ** (e - 4)


def _worker(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        from fp8_grouped_gemm_gb300 import ep
        codes, scales, off, rim, probs, x = _rank_buffers(rank)
        sizes = ep.exchange_sizes(torch.from_numpy(off))
        bufs = [_rank_buffers(s) for s in range(WORLD)]
        assert np.array_equal(sizes, np.stack([np.diff(b[2]) for b in bufs]))
        ex = ep.EPExchange(sizes, rank)
        tile_bytes = H // 32 * 128
        rc = torch.zeros((ex.R_recv, H), dtype=torch.uint8)
        rs = torch.zeros(ex.R_recv // 128 * tile_bytes, dtype=torch.uint8)
        ep.dispatch(ex, torch.from_numpy(codes), torch.from_numpy(scales), rc, rs, tile_bytes)
        # expected: for each local expert, every source's padded group in rank order
        want_c, want_s, want_off = [], [], [0]
        for j in range(ex.El):
            e = rank * ex.El + j
            n = 0
            for s in range(WORLD):
                sc, ss, so = bufs[s][0], bufs[s][1], bufs[s][2]
                a, b = int(so[e]), int(so[e + 1])
                want_c.append(sc[a:b])
                want_s.append(ss[a // 128 * tile_bytes:b // 128 * tile_bytes])
                n += b - a
            want_off.append(want_off[-1] + n)
        assert np.array_equal(rc.numpy(), np.concatenate(want_c))
        assert np.array_equal(rs.numpy(), np.concatenate(want_s))
        assert np.array_equal(ex.recv_offsets, np.array(want_off, dtype=np.int32))
        # each rank's experts on the received rows (dequantised), then combine
        from tests.layer_check import untile_mx_scales
        deq = OQ.dequantize_mx(rc.numpy(), untile_mx_scales(rs.numpy(), ex.R_recv, H))
        y_recv = np.zeros_like(deq)
        for j in range(ex.El):
            lo, hi = int(ex.recv_offsets[j]), int(ex.recv_offsets[j + 1])
            y_recv[lo:hi] = _expert_fn(rank * ex.El + j, deq[lo:hi])
        y_local = torch.zeros((ex.R_send, H), dtype=torch.float64)
        ep.combine(ex, torch.from_numpy(y_recv), y_local)
        # every row came back to where it was routed from
        mine = OQ.dequantize_mx(codes, untile_mx_scales(scales, ex.R_send, H))
        want = np.zeros_like(mine)
        for e in range(E):
            want[off[e]:off[e + 1]] = _expert_fn(e, mine[off[e]:off[e + 1]])
        assert np.array_equal(y_local.numpy(), want)
        # the layer output equals the one-rank layer on this rank's tokens
        out_ep = OR.unpermute(y_local.numpy(), rim, probs)
        cx, sx = OQ.quantize_mx(x)
        xq = OQ.dequantize_mx(cx, sx)
        ref = np.zeros_like(xq)
        idx = _rank_inputs(rank)[1]
        for j in range(K):
            ref += probs[:, j:j + 1].astype(np.float64) * np.stack(
                [_expert_fn(int(e), xq[t]) for t, e in enumerate(idx[:, j])])
        assert np.allclose(out_ep, ref, rtol=1e-12, atol=1e-12)
        q.put((rank, "ok", int(ex.R_recv)))
    except Exception as exc:          # report, then leave the group like the others
        q.put((rank, repr(exc), 0))
    finally:
        dist.destroy_process_group()


def test_ep_dispatch_and_combine_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
    assert all(r[1] == "ok" for r in res), res
    assert all(p.exitcode == 0 for p in procs)
    # both ranks received rows (the experts are split evenly)
    assert all(r[2] > 0 for r in res)


def test_ep_exchange_bookkeeping():
    """Receive layout from the padded group sizes: local expert major, source
    rank minor; sizes must be multiples of 128 and experts divide the ranks."""
    from fp8_grouped_gemm_gb300 import ep
    sizes = np.array([[128, 256, 0, 128], [384, 0, 128, 128]])
    ex = ep.EPExchange(sizes, 1)
    assert (ex.El, ex.R_send, ex.R_recv) == (2, 640, 384)
    assert ex.send_range(0, 1) == (384, 384) and ex.send_range(1, 0) == (384, 512)
    assert ex.recv_range(0, 0) == (0, 0) and ex.recv_range(0, 1) == (0, 128)
    assert ex.recv_range(1, 0) == (128, 256) and ex.recv_range(1, 1) == (256, 384)
    assert list(ex.recv_offsets) == [0, 128, 384]
    with pytest.raises(ValueError):
        ep.EPExchange(np.array([[100, 28], [128, 0]]), 0)
    with pytest.raises(ValueError):
        ep.EPExchange(np.zeros((2, 3), np.int64), 0)

"""mgq_moe_permute_noalloc, the permute + quantise call for callers that
cannot allocate device memory (for example a plugin whose host framework owns
every device allocation, or a runtime that forbids allocating while it runs).
It takes its routing scratch from a fixed device array inside the library, so
its results must equal those of mgq_moe_permute with a caller workspace.

This file is collected last on purpose (a failure here leaves every other
test already run); it passes alone in a fresh process and after the others."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _inputs(seed, T, E, k, H):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    return x, idx


def _run(mgq, fn, x, idx, E, align, R, with_ws):
    dev = x.device
    T, k = idx.shape
    H = x.shape[1]
    out = dict(
        rim=torch.full((T, k), -3, dtype=torch.int32, device=dev),
        src=torch.full((R,), -3, dtype=torch.int32, device=dev),
        off=torch.full((E + 1,), -3, dtype=torch.int32, device=dev),
        cnt=torch.full((E,), -3, dtype=torch.int32, device=dev),
        codes=torch.full((R, H), 0x11, dtype=torch.uint8, device=dev),
        sc=torch.full((mgq.mx_scale_bytes(R, H),), 0x22, dtype=torch.uint8, device=dev),
    )
    q = mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, out["codes"], out["sc"])
    if with_ws:
        ws = torch.empty(mgq.permute_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
        fn(x, idx, E, align, q, R, out["rim"], out["src"], out["off"], out["cnt"], ws)
    else:
        fn(x, idx, E, align, q, R, out["rim"], out["src"], out["off"], out["cnt"])
    torch.cuda.synchronize()
    n = int(out["off"][E].item())
    res = {key: v.cpu().numpy() for key, v in out.items()}
    res["src"] = res["src"][:n]
    res["codes"] = res["codes"][:n]
    return res


def test_noalloc_matches_workspace_call_twice_in_a_row():
    from fp8_grouped_gemm_gb300 import mgq
    mgq.load()
    dev = torch.device("cuda:0")
    # two calls in a row with different inputs and routing: the second must
    # not see the first call's scratch contents
    for seed, (T, E, k, H) in ((1, (3000, 16, 4, 512)), (2, (777, 6, 2, 1024))):
        x, idx = _inputs(seed, T, E, k, H)
        xd, idxd = x.to(dev), torch.from_numpy(idx).to(dev)
        R = mgq.r_cap(T, k, E, 128)
        want = _run(mgq, mgq.moe_permute, xd, idxd, E, 128, R, True)
        got = _run(mgq, mgq.moe_permute_noalloc, xd, idxd, E, 128, R, False)
        for key in want:
            assert np.array_equal(want[key], got[key]), key
        assert mgq.get_error() == mgq.OK


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from fp8_grouped_gemm_gb300 import mgq
    lib = mgq.load()
    # 300000 * 8 entries -> 2344 chunks x 128 experts > 262144 scratch ints:
    # refused on the host before anything is launched
    rc = lib.mgq_moe_permute_noalloc(None, 300000, 128, None, 8, 128, 128, None, None, 1 << 22, None, None,
                                     None, None, None)
    assert rc == mgq.ERR_INVALID_ARG

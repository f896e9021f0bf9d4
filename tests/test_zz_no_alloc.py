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
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)   # k distinct experts per token
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    return x, idx


def _run(mgq, fn, x, idx, E, align, R, with_ws, col):
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
    if col:
        # the column-wise copy too: routing then finishes in its own kernel,
        # which reads the scratch as well, and one tile pass writes both copies
        out["ccodes"] = torch.full((H, R), 0x33, dtype=torch.uint8, device=dev)
        out["csc"] = torch.full((mgq.mx_scale_bytes(H, R),), 0x44, dtype=torch.uint8, device=dev)
        q = mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, out["codes"], out["sc"], out["ccodes"], out["csc"])
    else:
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
    if col:
        res["ccodes"] = res["ccodes"][:, :n]
    return res


# (T, E, k, H) of two calls in a row; the last case fills the scratch exactly:
# ceil(131072 * 8 / 1024) chunks x 256 experts = 262144 ints = 1 MiB
CASES = {
    "rows": [(1, (3000, 16, 4, 512)), (2, (777, 6, 2, 1024))],
    "rows_and_columns": [(3, (2500, 8, 2, 384)), (4, (640, 12, 3, 256))],
    "full_scratch": [(5, (131072, 256, 8, 128)), (6, (5000, 32, 2, 256))],
}


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_workspace_call_twice_in_a_row(case):
    from fp8_grouped_gemm_gb300 import mgq
    mgq.load()
    dev = torch.device("cuda:0")
    col = case != "rows"
    # two calls in a row with different inputs and routing: the second must
    # not see the first call's scratch contents
    for seed, (T, E, k, H) in CASES[case]:
        if case == "full_scratch" and seed == 5:
            assert mgq.permute_workspace_size(T, k, E) == 1 << 20
        x, idx = _inputs(seed, T, E, k, H)
        xd, idxd = x.to(dev), torch.from_numpy(idx).to(dev)
        R = mgq.r_cap(T, k, E, 128)
        want = _run(mgq, mgq.moe_permute, xd, idxd, E, 128, R, True, col)
        got = _run(mgq, mgq.moe_permute_noalloc, xd, idxd, E, 128, R, False, col)
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
    # one routed entry past a full scratch: 1025 chunks x 256 experts
    rc = lib.mgq_moe_permute_noalloc(None, 131073, 128, None, 8, 256, 128, None, None, 1 << 22, None, None,
                                     None, None, None)
    assert rc == mgq.ERR_INVALID_ARG

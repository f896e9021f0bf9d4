"""Failure detection without a GPU fault: a grouped GEMM whose pipeline never
receives data (the producer is told to issue no loads) must come back with
MGQ_ERR_TIMEOUT after its bounded waits, leave the output untouched, and leave
the CUDA context usable for the next call. The stall and the short wait limit
are the library's test hooks (mgq_set_gemm_option); the test runs in a
subprocess so that its options cannot leak into other tests."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import os, sys, time
    import numpy as np, torch
    sys.path.insert(0, {root!r})
    from fp8_grouped_gemm_gb300 import mgq
    from tests.layer_check import tile_mx_scales
    mgq.load()
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(0)
    E, N, K, R = 2, 256, 256, 512
    offs = torch.tensor([0, 256, 512], dtype=torch.int32, device=dev)
    a = torch.from_numpy(rng.integers(0, 0x7E, (R, K)).astype(np.uint8)).to(dev)
    w = torch.from_numpy(rng.integers(0, 0x7E, (E * N, K)).astype(np.uint8)).to(dev)
    sa = torch.tensor([1.0], device=dev)
    sw = torch.ones(E, device=dev)
    sca = torch.from_numpy(tile_mx_scales(np.full((R, K // 32), 127, np.uint8))).to(dev)
    scw = torch.from_numpy(tile_mx_scales(np.full((E * N, K // 32), 127, np.uint8))).to(dev)
    kinds = [("tensor", mgq.TENSOR_F32, (a, sa), (w, sw)), ("mx", mgq.MX32_E8M0, (a, sca), (w, scw))]
    for name, sc, (ad, asc), (wd, wsc) in kinds:
        A = mgq.operand(ad, asc, K, mgq.E4M3)
        W = mgq.operand(wd, wsc, K, mgq.E4M3)
        y = torch.full((R, N), 7.0, dtype=torch.bfloat16, device=dev)
        mgq.set_gemm_option(mgq.GEMM_OPT_DEBUG_STALL, 1)
        mgq.set_gemm_option(mgq.GEMM_OPT_WAIT_MS, 50)
        t0 = time.time()
        mgq.grouped_gemm_fwd(A, W, sc, offs, E, R, N, K, y)
        torch.cuda.synchronize()
        dt = time.time() - t0
        st = mgq.get_error()
        assert st == mgq.ERR_TIMEOUT, (name, st)
        assert bool(torch.all(y == 7.0)), name            # nothing stored
        assert dt < 10.0, (name, dt)
        mgq.set_gemm_option(mgq.GEMM_OPT_DEBUG_STALL, 0)
        mgq.set_gemm_option(mgq.GEMM_OPT_WAIT_MS, 0)
        # the context is still usable: the same call without the stall is correct
        mgq.grouped_gemm_fwd(A, W, sc, offs, E, R, N, K, y)
        torch.cuda.synchronize()
        assert mgq.get_error() == mgq.OK
        assert not bool(torch.all(y == 7.0)), name
        print(name, "timeout reported in", round(dt, 3), "s; context usable")
    print("OK")
""")


def test_gemm_pipeline_timeout_is_reported_and_context_survives():
    code = SCRIPT.format(root=ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "OK" in r.stdout

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running oracle test")


def pytest_sessionstart(session):
    # test_gpu_gemm_1cta.py reruns the GEMM parity tests in a subprocess with
    # one kernel-selection option of the library set for the whole session
    opt = os.environ.get("MGQ_TEST_GEMM_OPTION")
    if opt:
        from fp8_grouped_gemm_gb300 import mgq
        mgq.set_gemm_option(getattr(mgq, opt), 1)
        assert mgq.get_gemm_option(getattr(mgq, opt)) == 1


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped, not failed, when no GPU is present and the run
    # did not select them explicitly; the driver runs them with -m gpu.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)

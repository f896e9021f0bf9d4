"""The grouped GEMM parity tests again under the other kernel selections:
the library option MGQ_GEMM_OPT_FORCE_1CTA puts every call on the 1-CTA
kernel (per-tensor calls otherwise go to the 2-CTA pair kernel),
MGQ_GEMM_OPT_MX_PAIR puts MX calls and MGQ_GEMM_OPT_NV_PAIR NVFP4 calls on the
pair kernel (otherwise 1-CTA). Each selection runs the parity tests in a
subprocess whose conftest sets the option named by MGQ_TEST_GEMM_OPTION
before any test, so the option cannot leak into other tests."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("opt,sel", [("GEMM_OPT_FORCE_1CTA", "gemm and not mn_major"),
                                     ("GEMM_OPT_MX_PAIR", "gemm and not mn_major"),
                                     ("GEMM_OPT_NV_PAIR", "nvfp4")])
def test_gemm_parity_under_other_kernel_selection(opt, sel):
    env = dict(os.environ, MGQ_TEST_GEMM_OPTION=opt)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        os.path.join(ROOT, "tests", "test_gpu_kernels.py"), "-k", sel],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout

"""The grouped GEMM parity tests again under the other kernel selections:
MGQ_GEMM_1CTA=1 puts every call on the 1-CTA kernel (per-tensor calls
otherwise go to the 2-CTA pair kernel), MGQ_GEMM_MX_PAIR=1 puts MX calls and
MGQ_GEMM_NV_PAIR=1 NVFP4 calls on the pair kernel (otherwise 1-CTA). They are
read once per process, hence the subprocesses."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("var,sel", [("MGQ_GEMM_1CTA", "gemm and not mn_major"),
                                     ("MGQ_GEMM_MX_PAIR", "gemm and not mn_major"),
                                     ("MGQ_GEMM_NV_PAIR", "nvfp4")])
def test_gemm_parity_under_other_kernel_selection(var, sel):
    env = dict(os.environ, **{var: "1"})
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        os.path.join(ROOT, "tests", "test_gpu_kernels.py"), "-k", sel],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout

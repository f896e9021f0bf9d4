"""The grouped GEMM parity tests again, with every call on the 1-CTA kernel
(MGQ_GEMM_1CTA=1): by default per-tensor and MX calls go to the 2-CTA pair
kernel, so this keeps the 1-CTA MX and per-tensor paths under the same
oracle checks. The variable is read once per process, hence the subprocess."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gemm_parity_on_the_1cta_kernel():
    env = dict(os.environ, MGQ_GEMM_1CTA="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        os.path.join(ROOT, "tests", "test_gpu_kernels.py"), "-k", "gemm and not mn_major"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout

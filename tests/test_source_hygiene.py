"""Source hygiene (CPU only): no source file names the batched memory-copy
calls that this library must not use (one copy per call or a gather kernel
instead), and every kernel source is compiled for sm_103a only."""
import glob
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = [p for ext in ("*.cu", "*.cuh", "*.h", "*.c", "*.py", "*.sh", "*.txt", "*.ini")
           for p in glob.glob(os.path.join(ROOT, "**", ext), recursive=True)
           if "/_work/" not in p and "/gpurun_out/" not in p and "/_build/" not in p]
# the four names, assembled so that this file does not spell them out
_B = "Batch" + "Async"
BANNED = ["cuda" + "Memcpy" + _B, "cuda" + "Memcpy3D" + _B, "cu" + "Memcpy" + _B, "cu" + "Memcpy3D" + _B]


def test_no_batched_memcpy_calls():
    assert SOURCES
    for p in SOURCES:
        text = open(p, errors="replace").read()
        for name in BANNED:
            assert name.lower() not in text.lower(), f"{os.path.relpath(p, ROOT)} names {name}"


def test_build_targets_sm103a_only():
    from fp8_grouped_gemm_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_library_reads_no_environment():
    """Kernel choice and test hooks are explicit calls (mgq_set_gemm_option):
    no stray environment variable can change what the library runs."""
    for p in glob.glob(os.path.join(ROOT, "fp8_grouped_gemm_gb300", "csrc", "*")):
        text = open(p, errors="replace").read()
        assert "getenv" not in text, os.path.relpath(p, ROOT)

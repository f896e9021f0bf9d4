"""The C-ABI library loads and exports every symbol include/mgq.h declares;
host-side argument validation answers before anything is launched (CPU only:
no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mgq.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mgq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from fp8_grouped_gemm_gb300 import _build, mgq
    if not os.path.exists(mgq.LIB_PATH):
        _build.build()
    return mgq.load()


def test_every_declared_symbol_is_exported(lib):
    from fp8_grouped_gemm_gb300 import mgq
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(mgq.EXPORTS) | {n for n in names if n.startswith("mgq_")}
    assert set(mgq.EXPORTS) <= set(names)


def test_status_strings(lib):
    from fp8_grouped_gemm_gb300 import mgq
    assert mgq.status_string(mgq.OK) == "ok"
    assert "invalid" in mgq.status_string(mgq.ERR_INVALID_ARG)
    assert lib.mgq_version() == 2          # the operand struct with scale_image


def test_workspace_size(lib):
    from fp8_grouped_gemm_gb300 import mgq
    assert mgq.permute_workspace_size(16384, 2, 8) == 32 * 8 * 4
    assert mgq.permute_workspace_size(-1, 2, 8) == 0


def test_host_validation_rejects_bad_arguments(lib):
    """Each call returns MGQ_ERR_INVALID_ARG (or UNSUPPORTED) before touching
    the GPU when its arguments are wrong."""
    from fp8_grouped_gemm_gb300 import mgq
    INV = mgq.ERR_INVALID_ARG
    # negative token count, misaligned H, k > 8, missing outputs
    assert lib.mgq_moe_permute(None, -1, 128, None, 2, 8, 128, None, None, 1024, None, None, None, None,
                               None, 0, None) == INV
    assert lib.mgq_moe_permute(None, 4, 100, None, 2, 8, 128, None, None, 1024, None, None, None, None,
                               None, 0, None) == INV
    assert lib.mgq_moe_permute(None, 4, 128, None, 9, 16, 128, None, None, 1024, None, None, None, None,
                               None, 0, None) == INV
    # GEMM: null operands, then an unsupported format
    a = mgq.Operand(None, None, 128, mgq.E4M3)
    assert lib.mgq_grouped_gemm_fwd(ctypes.byref(a), ctypes.byref(a), mgq.MX32_E8M0, None, 4, 128, 256, 128,
                                    None, 0, None) == INV
    b = mgq.Operand(16, 16, 128, 7)
    assert lib.mgq_grouped_gemm_fwd(ctypes.byref(b), ctypes.byref(b), mgq.MX32_E8M0, None, 4, 128, 256, 128,
                                    None, 0, None) == mgq.ERR_UNSUPPORTED
    # GEMM shapes: N not a multiple of 256 / K not of 128 / misaligned output
    c = mgq.Operand(16, 16, 128, mgq.E4M3)
    assert lib.mgq_grouped_gemm_fwd(ctypes.byref(c), ctypes.byref(c), mgq.MX32_E8M0, 16, 4, 128, 200, 128,
                                    32, 0, None) == INV
    assert lib.mgq_grouped_gemm_fwd(ctypes.byref(c), ctypes.byref(c), mgq.MX32_E8M0, 16, 4, 128, 256, 100,
                                    32, 0, None) == INV
    assert lib.mgq_grouped_gemm_fwd(ctypes.byref(c), ctypes.byref(c), mgq.MX32_E8M0, 16, 4, 128, 256, 128,
                                    33, 0, None) == INV
    # beta != 0 only for float32 wgrad
    assert lib.mgq_grouped_gemm_wgrad(ctypes.byref(c), ctypes.byref(c), mgq.MX32_E8M0, 16, 4, 128, 128, 256,
                                      ctypes.c_float(1.0), 32, mgq.OUT_BF16, None) == INV
    # quantiser: K not a multiple of 128; unsupported scaling
    q = mgq.qdesc(mgq.E4M3, mgq.MX32_E8M0, 16, 16)
    assert lib.mgq_block_quantize(16, 1, 128, 100, ctypes.byref(q), None) == INV
    q2 = mgq.qdesc(mgq.E4M3, 9, 16, 16)
    assert lib.mgq_block_quantize(16, 1, 128, 128, ctypes.byref(q2), None) == mgq.ERR_UNSUPPORTED
    # ragged-group quantiser: C not a multiple of 128, missing offsets, blockwise scaling
    assert lib.mgq_grouped_quantize(16, 256, 100, 16, 4, ctypes.byref(q), None) == INV
    assert lib.mgq_grouped_quantize(16, 256, 128, None, 4, ctypes.byref(q), None) == INV
    # 128x128 tiles are a weight layout, not one over ragged groups
    q3 = mgq.qdesc(mgq.E4M3, mgq.BLK_128x128_F32, 16, 16)
    assert lib.mgq_grouped_quantize(16, 256, 128, 16, 4, ctypes.byref(q3), None) == mgq.ERR_UNSUPPORTED
    # blockwise column copies need their scale_inv buffer, and the permute's
    # groups padded to the 128-row column block
    q4 = mgq.qdesc(mgq.E4M3, mgq.BLK_1x128_F32, 16, 16, 32, None)
    assert lib.mgq_grouped_quantize(16, 256, 128, 16, 4, ctypes.byref(q4), None) == mgq.ERR_INVALID_ARG
    assert lib.mgq_block_quantize(16, 1, 128, 128, ctypes.byref(q4), None) == mgq.ERR_INVALID_ARG
    q5 = mgq.qdesc(mgq.E4M3, mgq.BLK_1x128_F32, 16, 16, 32, 48)
    assert lib.mgq_moe_permute(16, 4, 128, 16, 2, 8, 32, ctypes.byref(q5), None, 1024, 16, 16, 16, 16, 16,
                               1 << 20, None) == mgq.ERR_INVALID_ARG
    assert lib.mgq_amax_history_update(None, None, None, None, 1, 1, ctypes.c_float(448.0), None) == INV
    assert lib.mgq_get_error(None, None) == INV
    # NVFP4 scale image: rows a multiple of 128, ld of 256, aligned pointers
    assert lib.mgq_nv_scale_image(16, 100, 256, 16, None) == INV
    assert lib.mgq_nv_scale_image(16, 128, 200, 16, None) == INV
    assert lib.mgq_nv_scale_image(16, 128, 256, 8, None) == INV
    assert lib.mgq_nv_scale_image(None, 128, 256, 16, None) == INV


def test_operand_layout_validation(lib):
    """MN-major operands: per-tensor scaling in dgrad (B) and wgrad (A, B)
    only; anything else is refused on the host."""
    from fp8_grouped_gemm_gb300 import mgq
    UNS, INV = mgq.ERR_UNSUPPORTED, mgq.ERR_INVALID_ARG
    k = mgq.Operand(16, 16, 256, mgq.E4M3)
    mn = mgq.Operand(16, 16, 256, mgq.E4M3, None, mgq.LAYOUT_MN)
    bad = mgq.Operand(16, 16, 256, mgq.E4M3, None, 5)
    args = (16, 4, 256, 256, 256)
    # MX block scales run along the contraction: no MN-major reading
    assert lib.mgq_grouped_gemm_dgrad(ctypes.byref(k), ctypes.byref(mn), mgq.MX32_E8M0, *args, 32, 0,
                                      None) == UNS
    # the forward activations (and dgrad's dY) are K-major
    assert lib.mgq_grouped_gemm_fwd(ctypes.byref(mn), ctypes.byref(k), mgq.TENSOR_F32, *args, 32, 0,
                                    None) == UNS
    assert lib.mgq_grouped_gemm_fwd(ctypes.byref(bad), ctypes.byref(k), mgq.TENSOR_F32, *args, 32, 0,
                                    None) == INV


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes mirrors of mgq_operand / mgq_qdesc have the C layout (sizes
    and field offsets from a program compiled against include/mgq.h)."""
    import shutil
    import subprocess
    from fp8_grouped_gemm_gb300 import mgq
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "probe.c"
    src.write_text(
        "#include <stdio.h>\n#include <stddef.h>\n#include \"mgq.h\"\n"
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(mgq_operand),"
        " offsetof(mgq_operand, ld), offsetof(mgq_operand, dtype), offsetof(mgq_operand, global_scale),"
        " offsetof(mgq_operand, layout), sizeof(mgq_qdesc), offsetof(mgq_qdesc, amax_out));"
        "printf(\"%zu\\n\", offsetof(mgq_operand, scale_image));return 0;}\n")
    exe = tmp_path / "probe"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    O, Q = mgq.Operand, mgq.QDesc
    assert got == [ctypes.sizeof(O), O.ld.offset, O.dtype.offset, O.global_scale.offset, O.layout.offset,
                   ctypes.sizeof(Q), Q.amax_out.offset, O.scale_image.offset]


def test_gemm_options_round_trip_and_validation(lib):
    """The GEMM options are host state only: set, read back, reset; values
    outside their range and unknown options are refused."""
    from fp8_grouped_gemm_gb300 import mgq
    for opt in (mgq.GEMM_OPT_FORCE_1CTA, mgq.GEMM_OPT_MX_PAIR, mgq.GEMM_OPT_NV_PAIR, mgq.GEMM_OPT_DIRECT_STORE,
                mgq.GEMM_OPT_DEBUG_STALL):
        assert mgq.get_gemm_option(opt) == 0
        mgq.set_gemm_option(opt, 1)
        assert mgq.get_gemm_option(opt) == 1
        mgq.set_gemm_option(opt, 0)
        assert lib.mgq_set_gemm_option(opt, 2) == mgq.ERR_INVALID_ARG
        assert lib.mgq_set_gemm_option(opt, -1) == mgq.ERR_INVALID_ARG
    mgq.set_gemm_option(mgq.GEMM_OPT_WAIT_MS, 50)
    assert mgq.get_gemm_option(mgq.GEMM_OPT_WAIT_MS) == 50
    mgq.set_gemm_option(mgq.GEMM_OPT_WAIT_MS, 0)
    assert lib.mgq_set_gemm_option(mgq.GEMM_OPT_WAIT_MS, 600001) == mgq.ERR_INVALID_ARG
    assert lib.mgq_set_gemm_option(6, 0) == mgq.ERR_INVALID_ARG
    assert lib.mgq_set_gemm_option(-1, 0) == mgq.ERR_INVALID_ARG
    assert lib.mgq_get_gemm_option(0, None) == mgq.ERR_INVALID_ARG

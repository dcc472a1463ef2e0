"""The C-ABI library builds, loads and exports every symbol include/rfp2.h
declares; host-side checks that need no GPU behave as documented."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rfp2.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b((?:rfp2|hfp4)_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import gemm_rocmfp2_mul_gb300 as g
    g.build()
    return g.lib()


def test_header_declares_the_hot_path_calls():
    names = _declared_functions()
    for required in ["rfp2_quantize_act", "rfp2_gemv", "rfp2_moe_gemv", "rfp2_gemm", "hfp4_gemv"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    import gemm_rocmfp2_mul_gb300 as g
    assert g.status_str(0) == "RFP2_OK"
    assert g.status_str(7) == "RFP2_EBADID"
    assert g.status_str(8) == "RFP2_ETIMEOUT"
    assert g.status_str(99) == "RFP2_UNKNOWN"
    assert lib.rfp2_version() >= 100


def test_workspace_sizes(lib):
    import gemm_rocmfp2_mul_gb300 as g
    up = lambda v: (v + 255) // 256 * 256
    # q int8 [N, K] rounded up to 256 bytes, then d fp32 [N, K/32]
    assert g.rfp2_gemv_workspace_bytes(1, 4096) == 4096 + 128 * 4
    # every batch 1..8 runs the int8 path: only q and d
    assert g.rfp2_gemv_workspace_bytes(3, 256) == up(768) + 24 * 4
    assert g.rfp2_gemv_workspace_bytes(8, 4096) == 8 * 4096 + 8 * 128 * 4
    # the verify-batch entry point keeps its own layout: q, d, the two f16
    # activation pieces of a 32-token tile and the exponents
    assert g.rfp2_gemv_batched_workspace_bytes(16, 256, 3) == up(768) + up(24 * 4) + up(2 * 32 * 256 * 2) + up(3 * 4)
    assert g.rfp2_gemv_workspace_bytes(0, 256) == 0


def test_null_pointers_are_rejected_before_any_cuda_call(lib):
    EINVAL = 1
    assert lib.rfp2_gemv_q8(None, 16, 256, None, None, 1, None, None, None) == EINVAL
    assert lib.rfp2_gemv(None, 16, 256, None, 1, None, None, 0, None, None) == EINVAL
    assert lib.rfp2_quantize_act(None, 1, 32, None, None, None) == EINVAL
    assert lib.rfp2_pack_weights(None, 2, 32, None, None) == EINVAL
    assert lib.rfp2_validate_weights(None, 4, None, None, None) == EINVAL
    # K not a multiple of 32 is a shape error for the quantizer and packers
    assert lib.rfp2_quantize_act(None, 1, 40, None, None, None) == 2
    assert lib.rfp2_pack_weights(None, 2, 40, None, None) == 2


def test_binding_refuses_to_run_without_the_library(monkeypatch, tmp_path):
    import gemm_rocmfp2_mul_gb300 as g
    from gemm_rocmfp2_mul_gb300 import buildlib as b
    monkeypatch.setattr(b, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(g, "_lib", None)
    with pytest.raises(RuntimeError):
        g.lib()


def test_product_package_never_touches_the_oracle():
    """The product path never imports, includes, links or runs the oracle."""
    pkg = os.path.join(ROOT, "gemm_rocmfp2_mul_gb300")
    bad = re.compile(r"(import\s+oracle|from\s+oracle|oracle/|liboracle|rfp2_oracle|orc_)")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f)).read()
                assert not bad.search(text), f

"""The C ABI: the library builds, loads without a GPU, exports every function
include/iq.h declares, and its host-side checks and size helpers behave as
documented (none of these calls touches a device)."""

import os
import re
import subprocess

import pytest

from fp4_fp8_quant_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "iq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(iq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    from fp4_fp8_quant_gb300 import iq
    return iq.lib()


def test_header_declarations_match_binding(lib):
    from fp4_fp8_quant_gb300 import iq
    assert _declared_functions() == sorted(iq.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(iq_[a-z0-9_]+)$", out, flags=re.M))
    missing = [f for f in _declared_functions() if f not in exported]
    assert not missing, missing
    for f in _declared_functions():
        assert getattr(lib, f) is not None


def test_size_helpers(lib):
    assert lib.iq_fp8_scale_words(4632, 7168) == 14 * 4632
    assert lib.iq_fp8_scale_words(5, 1536) == 3 * 8
    assert lib.iq_fp8_scale_words(5, 640) == 2 * 8
    assert lib.iq_fp8_scale_words(0, 1536) == 0
    # FP8 latent, scale words at the next 256-byte boundary, then the fused
    # quantizer's flags (an epoch word and 512 progress words) at the next one
    assert lib.iq_prepare_q_workspace(4632) == 7170560 + 513 * 8
    assert (4632 * 1536 + 3 * 4632 * 4 + 255) // 256 * 256 == 7170560
    assert lib.iq_prepare_q_workspace(5) == (7680 + 3 * 8 * 4 + 255) // 256 * 256 + 513 * 8
    assert lib.iq_prepare_q_workspace(0) == 0


def test_host_side_argument_checks_need_no_device(lib):
    # shape and argument errors are returned before any CUDA call
    assert lib.iq_fp8_quant_1x128_ue8m0(16, 4, 200, 256, 16, 256, 16, None) == -3
    assert lib.iq_fp8_quant_1x128_ue8m0(16, 4, 0, 256, 16, 256, 16, None) == -3
    assert lib.iq_fp8_quant_1x128_ue8m0(16, -1, 128, 256, 16, 256, 16, None) == -1
    assert lib.iq_fp8_quant_1x128_ue8m0(16, 0, 128, 256, 16, 256, 16, None) == 0
    assert lib.iq_fp8_quant_1x128_ue8m0(None, 4, 128, 256, 16, 256, 16, None) == -1
    assert lib.iq_fp8_quant_1x128_ue8m0(18, 4, 128, 256, 16, 256, 16, None) == -2
    assert lib.iq_fp8_quant_1x128_ue8m0(16, 4, 128, 100, 16, 256, 16, None) == -1
    assert lib.iq_prepare_q(16, 0, 16, 16, 16, 16, 16, None, 0, None) == 0
    assert lib.iq_prepare_q(16, -3, 16, 16, 16, 16, 16, None, 0, None) == -1
    assert lib.iq_prepare_q(16, 4, 16, 16, 16, 16, 16, None, 0, None) == -1
    assert lib.iq_prepare_q(16, 4, 16, 16, 16, 16, 16, 256, 10, None) == -6
    assert lib.iq_prepare_q(16, 4, 17, 16, 16, 16, 16, 256, 1 << 20, None) == -2
    assert lib.iq_prepare_q_debug(16, 4, 16, 16, 16, 16, 16, None, 256, 1 << 20, None) == -1
    assert lib.iq_gemm_rope_hadamard_fp4(16, None, 4, 16, 16, 16, 16, 16, None, None) == -1


def test_status_strings(lib):
    for code in range(0, -8, -1):
        s = lib.iq_status_str(code).decode()
        assert s.startswith("IQ_")


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from fp4_fp8_quant_gb300 import iq
    monkeypatch.setattr(iq, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(iq, "_lib", None)
    with pytest.raises(ImportError):
        iq.lib()


def test_small_m_threshold_is_clamped_and_restored(lib):
    """The token-count route switch is host state only: no device needed."""
    old = lib.iq_small_m_threshold()
    assert old == 128
    try:
        assert lib.iq_set_small_m_threshold(8) == 128
        assert lib.iq_small_m_threshold() == 8
        lib.iq_set_small_m_threshold(1000)
        assert lib.iq_small_m_threshold() == 128
        lib.iq_set_small_m_threshold(-5)
        assert lib.iq_small_m_threshold() == 0
    finally:
        lib.iq_set_small_m_threshold(old)
    assert lib.iq_small_m_threshold() == old


def test_fp4_format_helpers_and_checks(lib):
    assert lib.iq_fp4_scale_bytes(0) == 256 and lib.iq_fp4_scale_bytes(1) == 256
    assert lib.iq_fp4_scale_bytes(2) == 512 and lib.iq_fp4_scale_bytes(3) == 0
    # unknown format, before anything else
    assert lib.iq_prepare_q_ex(16, 4, 16, 16, 16, 7, 16, 16, None, 256, 1 << 20, None) == -1
    # NVFP4 scales need 8-byte alignment
    assert lib.iq_prepare_q_ex(16, 4, 16, 16, 16, 2, 16, 20, None, 256, 1 << 20, None) == -2
    assert lib.iq_prepare_q_ex(16, 0, 16, 16, 16, 2, 16, 20, None, None, 0, None) == 0


def test_host_entry_sizes_settings_and_checks(lib):
    """iq_prepare_q_host: workspace size, chunk-row setting, and the argument
    checks that come before any CUDA call."""
    # codes + scales + positions + FP8 latent + packed scales, each 256-aligned
    assert lib.iq_prepare_q_host_workspace(4632, 0) == 4632 * 4096 + 4632 * 256 + 18688 + 4632 * 1536 + 3 * 4632 * 4
    assert lib.iq_prepare_q_host_workspace(4632, 2) == 4632 * 4096 + 4632 * 512 + 18688 + 4632 * 1536 + 3 * 4632 * 4
    assert lib.iq_prepare_q_host_workspace(5, 0) == 20480 + 1280 + 256 + 7680 + 3 * 8 * 4
    assert lib.iq_prepare_q_host_workspace(0, 0) == 0
    assert lib.iq_prepare_q_host_workspace(16, 9) == 0
    old = lib.iq_host_chunk_rows()
    try:
        assert lib.iq_set_host_chunk_rows(300) == old
        assert lib.iq_host_chunk_rows() == 512
        lib.iq_set_host_chunk_rows(1)
        assert lib.iq_host_chunk_rows() == 256
        lib.iq_set_host_chunk_rows(1 << 30)
        assert lib.iq_host_chunk_rows() == 1 << 20
    finally:
        lib.iq_set_host_chunk_rows(old)
    assert lib.iq_host_chunk_rows() == old
    need = lib.iq_prepare_q_host_workspace(4, 0)
    assert lib.iq_prepare_q_host(16, 0, 16, 16, 16, 0, 16, 16, None, 0, None) == 0       # M == 0
    assert lib.iq_prepare_q_host(16, -1, 16, 16, 16, 0, 16, 16, 256, need, None) == -1   # M < 0
    assert lib.iq_prepare_q_host(16, 4, 16, 16, 16, 5, 16, 16, 256, need, None) == -1    # unknown format
    assert lib.iq_prepare_q_host(16, 4, 16, 16, 16, 0, 16, 16, None, need, None) == -1   # no workspace
    assert lib.iq_prepare_q_host(16, 4, 16, 16, 16, 0, 16, 16, 128, need, None) == -2    # workspace alignment
    assert lib.iq_prepare_q_host(16, 4, 16, 16, 16, 0, 16, 16, 256, need - 1, None) == -6
    assert lib.iq_prepare_q_host(24, 4, 16, 16, 16, 0, 16, 16, 256, need, None) == -2    # latent alignment



def test_quant_fusion_switch_is_host_state(lib):
    old = lib.iq_set_quant_fusion(0)
    try:
        assert old == 0, "off by default"
        assert lib.iq_set_quant_fusion(5) == 0
        assert lib.iq_set_quant_fusion(0) == 1
        assert lib.iq_set_quant_fusion(1) == 0
    finally:
        lib.iq_set_quant_fusion(old)

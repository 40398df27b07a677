"""The C-ABI library builds, loads and exports every entry point that
include/moe.h declares (no GPU: no compute call is made)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib_path():
    from bit_moe_expert_top_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available to build libmoe.so")
        from bit_moe_expert_top_gb300 import build
        build.build()
    return _lib.LIB_PATH


def test_header_declares_the_path():
    names = _declared()
    for n in ["moe_route", "moe_permute", "moe_w2_mm", "moe_mxfp4_mm", "mxfp4_to_fp8_ws", "moe_combine"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    from bit_moe_expert_top_gb300 import _lib
    assert sorted(_lib.EXPORTS) == _declared()


def test_host_only_calls(lib_path):
    from bit_moe_expert_top_gb300 import _lib as L
    lib = L.lib()
    assert lib.moe_version() == 1
    assert lib.moe_permute_workspace_size(8, 2, 8) == 0
    a = lib.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, 64, 2048, 4096)
    b = lib.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, 128, 2048, 4096)
    assert 0 < a < b
    assert lib.moe_w2_mm_workspace_size(7, 64, 2048, 4096) == 0
    # K not a multiple of the table GEMV's 512-element slice: no workspace
    assert lib.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, 64, 256, 640) == 0
    assert lib.moe_w2_mm_workspace_size(L.STAGE_FC2, 64, 4096, 1152) == 0
    assert lib.moe_w2_mm_workspace_size(L.STAGE_FC2, 64, 4096, 1536) > 0
    # the bounded-wait limit is host state: set, read back, restore
    prev = lib.moe_set_wait_limit(777)
    assert lib.moe_set_wait_limit(prev) == 777


def test_noalloc_limit_matches_header(lib_path):
    """The binding's copy of MOE_W2_NOALLOC_SCRATCH_BYTES, and the row counts
    the header states for it (decode shapes H=4096, I=2048)."""
    from bit_moe_expert_top_gb300 import _lib as L
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    m = re.search(r"#define MOE_W2_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", src)
    assert m and int(m.group(1)) << int(m.group(2)) == L.W2_NOALLOC_SCRATCH_BYTES
    lib = L.lib()
    cap = L.W2_NOALLOC_SCRATCH_BYTES
    assert lib.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, 127, 2048, 4096) <= cap
    assert lib.moe_w2_mm_workspace_size(L.STAGE_FC1_SWIGLU, 128, 2048, 4096) > cap
    assert lib.moe_w2_mm_workspace_size(L.STAGE_FC2, 255, 4096, 2048) <= cap
    assert lib.moe_w2_mm_workspace_size(L.STAGE_FC2, 256, 4096, 2048) > cap


def test_side_sms_setting_rules(lib_path):
    """moe_set_side_sms (host only): returns the previous value, rejects
    counts outside [0, 1024] with -1 and leaves the setting unchanged."""
    from bit_moe_expert_top_gb300 import _lib as L
    lib = L.lib()
    prev = lib.moe_set_side_sms(12)
    assert lib.moe_set_side_sms(-1) == -1
    assert lib.moe_set_side_sms(1025) == -1
    assert lib.moe_set_side_sms(prev) == 12
    assert L.moe_set_side_sms(prev) == prev


def test_split_mode_constant_matches_header(lib_path):
    """The binding's mode numbers are the header's, MOE_MODE_SPLIT included."""
    from bit_moe_expert_top_gb300 import _lib as L
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    for name, val in (("AUTO", L.MODE_AUTO), ("GEMV", L.MODE_GEMV), ("GEMM", L.MODE_GEMM), ("SPLIT", L.MODE_SPLIT)):
        m = re.search(rf"#define MOE_MODE_{name} (\d+)", src)
        assert m and int(m.group(1)) == val


def test_decode_layer_host_rules(lib_path):
    """moe_w2_decode_layer (host-side checks, no launch): its workspace is the
    fused launch's for T*k rows, zero for no rows or a K the table GEMV does
    not take; shapes it cannot take are refused before any device call."""
    from bit_moe_expert_top_gb300 import _lib as L
    lib = L.lib()
    assert lib.moe_w2_decode_layer_workspace_size(8, 8, 4096, 2048) == lib.moe_w2_decode_fused_workspace_size(64, 4096, 2048) > 0
    assert lib.moe_w2_decode_layer_workspace_size(0, 8, 4096, 2048) == 0
    assert lib.moe_w2_decode_layer_workspace_size(8, 8, 640, 2048) == 0
    null = [None] * 24

    def call(T, E, k, out_fmt=L.FMT_BF16, offsets=None):
        a = list(null)
        a[2], a[3], a[4], a[9], a[10], a[13], a[19] = T, E, k, 512, 512, offsets, out_fmt
        a[21] = 0
        return lib.moe_w2_decode_layer(*a)

    assert call(-1, 8, 2) == L.MOE_ERR_ARG          # negative token count
    assert call(4, 8, 9) == L.MOE_ERR_ARG           # k > E
    assert call(4, 1025, 2) == L.MOE_ERR_ARG        # E above 1024
    assert call(4, 8, 2) == L.MOE_ERR_ARG           # offsets NULL
    # output format (checked before any pointer is read: the offsets address is never used)
    assert call(4, 8, 2, out_fmt=L.FMT_MXFP8, offsets=256) == L.MOE_ERR_ARG

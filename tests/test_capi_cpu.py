"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
entry point include/swin_wattn.h declares, and rejects bad arguments before any CUDA
call is made."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from swin_window_attention_gb300 import build, capi
    build.build()
    return capi


def _declared():
    txt = open(os.path.join(ROOT, "include", "swin_wattn.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(swin_wattn_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_documented_entry_points():
    names = _declared()
    for n in ("swin_wattn_plan", "swin_wattn_fwd", "swin_wattn_bwd", "swin_wattn_set_bias",
              "swin_wattn_debug_maps", "swin_wattn_destroy", "swin_wattn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = lib.load()
    for n in _declared():
        assert hasattr(so, n), n
    assert set(_declared()) == set(lib.SIGNATURES)


def test_debug_library_exports_its_header_and_the_library_does_not():
    """The fault-injection build exports every entry point of both headers; the default
    library exports nothing of include/swin_wattn_debug.h."""
    from swin_window_attention_gb300 import build, capi
    build.build(debug=True)
    txt = open(os.path.join(ROOT, "include", "swin_wattn_debug.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = sorted(set(re.findall(r"\b(swin_wattn_[a-z0-9_]+)\s*\(", txt)))
    assert names == sorted(capi.DEBUG_SIGNATURES)
    dbg = capi.load_debug()
    for n in _declared() + names:
        assert hasattr(dbg, n), n
    so = capi.load()
    for n in names:
        assert not hasattr(so, n), n
    # argument checks, host-side only
    assert dbg.swin_wattn_debug_set_fault(9, 1000000) == capi.ERR_INVALID_ARG
    assert dbg.swin_wattn_debug_set_fault(capi.FAULT_NONE, 10) == capi.ERR_INVALID_ARG
    assert dbg.swin_wattn_debug_set_fault(capi.FAULT_NONE, 1000000000) == capi.OK


def test_status_strings(lib):
    for code in range(7):
        assert lib.swin_wattn_status_string(code)
    assert lib.swin_wattn_status_string(99) == "unknown status"


@pytest.mark.parametrize("args,status", [
    # (B, H, W, C, nH, M, s, dtype)
    ((1, 8, 8, 64, 2, 5, 0, 0), 2),     # window size not supported
    ((1, 8, 8, 64, 2, 4, 4, 0), 1),     # shift >= M
    ((1, 8, 8, 64, 2, 4, -1, 0), 1),    # negative shift
    ((1, 10, 8, 64, 2, 4, 0, 0), 2),    # H not a multiple of M
    ((1, 8, 8, 96, 2, 4, 0, 0), 2),     # head width 48
    ((1, 8, 8, 64, 3, 4, 0, 0), 2),     # C not divisible by nH
    ((1, 8, 8, 64, 2, 4, 0, 7), 1),     # bad dtype code
    ((-1, 8, 8, 64, 2, 4, 0, 0), 1),    # negative batch
    ((1, 0, 8, 64, 2, 4, 0, 0), 1),     # empty grid
])
def test_plan_rejects_bad_shapes_before_touching_cuda(lib, args, status):
    rc, h = lib.swin_wattn_plan(*args, None, None)
    assert rc == status and h is None


def test_null_and_foreign_plan_handles(lib):
    assert lib.swin_wattn_fwd(None, None, None, None) == lib.ERR_BAD_PLAN
    assert lib.swin_wattn_bwd(12345678, None, None, None, None, None) == lib.ERR_BAD_PLAN
    assert lib.swin_wattn_set_bias(None, None, None) == lib.ERR_BAD_PLAN
    assert lib.swin_wattn_debug_maps(None, None, None, None, None, None) == lib.ERR_BAD_PLAN
    assert lib.swin_wattn_destroy(None) == lib.OK
    assert lib.swin_wattn_destroy(987654) == lib.ERR_BAD_PLAN


def test_null_out_handle(lib):
    so = lib.load()
    assert so.swin_wattn_plan(None, 1, 8, 8, 64, 2, 4, 0, 0, None, None) == lib.ERR_INVALID_ARG


def test_gemm_steps_reject_bad_arguments_before_touching_cuda(lib):
    # producer: workspace size query and shape checks
    assert lib.swin_wattn_qkv_workspace_bytes(80, 4) == 0           # C not a multiple of 32
    assert lib.swin_wattn_qkv_workspace_bytes(1568, 4) == 0         # C above 1536
    assert lib.swin_wattn_qkv_workspace_bytes(96, 4) >= 288 * 96 * 2 + 2 * 288 * 4 + 4 * 8
    assert lib.swin_wattn_qkv_proj(*([None] * 6), -1, 96, 1e-5, None, 0, None, None) == lib.ERR_INVALID_ARG
    assert lib.swin_wattn_qkv_proj(*([None] * 6), 4, 96, -1.0, None, 0, None, None) == lib.ERR_INVALID_ARG
    assert lib.swin_wattn_qkv_proj(*([None] * 6), 4, 80, 1e-5, None, 0, None, None) == lib.ERR_UNSUPPORTED
    assert lib.swin_wattn_qkv_proj(*([None] * 6), 0, 96, 1e-5, None, 0, None, None) == lib.OK
    # producer on prepared weights
    assert lib.swin_wattn_qkv_prepared_bytes(80) == 0
    assert lib.swin_wattn_qkv_prepared_bytes(96) >= 288 * 96 * 2 + 2 * 288 * 4
    assert lib.swin_wattn_qkv_stats_bytes(-1) == 0 and lib.swin_wattn_qkv_stats_bytes(5) >= 40
    assert lib.swin_wattn_qkv_prepare(*([None] * 4), 80, None, 0, None) == lib.ERR_UNSUPPORTED
    assert lib.swin_wattn_qkv_prepare(*([None] * 4), 96, None, 0, None) == lib.ERR_INVALID_ARG
    assert lib.swin_wattn_qkv_proj_prepared(None, None, None, -1, 96, 1e-5, None, 0, None, None) == lib.ERR_INVALID_ARG
    assert lib.swin_wattn_qkv_proj_prepared(None, None, None, 4, 80, 1e-5, None, 0, None, None) == lib.ERR_UNSUPPORTED
    assert lib.swin_wattn_qkv_proj_prepared(None, None, None, 0, 96, 1e-5, None, 0, None, None) == lib.OK
    # consumer
    assert lib.swin_wattn_proj_residual(*([None] * 5), -1, 96, None, None) == lib.ERR_INVALID_ARG
    assert lib.swin_wattn_proj_residual(*([None] * 5), 4, 48, None, None) == lib.ERR_UNSUPPORTED
    assert lib.swin_wattn_proj_residual(*([None] * 5), 4, 3072, None, None) == lib.ERR_UNSUPPORTED
    assert lib.swin_wattn_proj_residual(*([None] * 5), 0, 96, None, None) == lib.OK


def test_fp8_forward_rejects_a_bad_plan_before_touching_cuda(lib):
    assert lib.swin_wattn_fwd_fp8(None, None, 1.0, 1.0, 1.0, None, None) == lib.ERR_BAD_PLAN

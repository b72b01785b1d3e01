"""Error paths of the C ABI on a GPU machine. Every bad argument is refused on the host with
a status code before anything is launched; nothing here faults the GPU."""
import ctypes

import pytest
import torch

from swin_window_attention_gb300 import capi, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from swin_window_attention_gb300 import build
    build.build()
    capi.load()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _plan(B=1, H=14, W=14, M=7, s=3, nH=2, dtype=capi.BF16):
    table = inputs.trunc_normal(((2 * M - 1) ** 2, nH), 1).cuda()
    rc, h = capi.swin_wattn_plan(B, H, W, 32 * nH, nH, M, s, dtype, table.data_ptr(), _stream())
    assert rc == capi.OK, capi.swin_wattn_status_string(rc)
    return h, table


def test_host_pointers_are_refused():
    h, _ = _plan()
    host = torch.zeros(1, 14, 14, 192, dtype=torch.bfloat16)
    out = torch.zeros(1, 14, 14, 64, dtype=torch.bfloat16, device="cuda")
    assert capi.swin_wattn_fwd(h, host.data_ptr(), out.data_ptr(), _stream()) == capi.ERR_INVALID_ARG
    tab = inputs.trunc_normal((169, 2), 1)
    rc, h2 = capi.swin_wattn_plan(1, 14, 14, 64, 2, 7, 3, capi.BF16, tab.data_ptr(), _stream())
    assert rc == capi.ERR_INVALID_ARG and h2 is None
    assert capi.swin_wattn_destroy(h) == capi.OK


def test_misaligned_pointers_are_refused():
    h, _ = _plan()
    buf = torch.zeros(1 * 14 * 14 * 192 + 16, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 14, 14, 64, dtype=torch.bfloat16, device="cuda")
    assert capi.swin_wattn_fwd(h, buf.data_ptr() + 2, out.data_ptr(), _stream()) == capi.ERR_MISALIGNED
    assert capi.swin_wattn_fwd(h, buf.data_ptr(), out.data_ptr() + 8, _stream()) == capi.ERR_MISALIGNED
    assert capi.swin_wattn_destroy(h) == capi.OK


def test_null_tensor_pointers_are_refused():
    h, _ = _plan()
    out = torch.zeros(1, 14, 14, 64, dtype=torch.bfloat16, device="cuda")
    assert capi.swin_wattn_fwd(h, None, out.data_ptr(), _stream()) == capi.ERR_INVALID_ARG
    assert capi.swin_wattn_bwd(h, None, None, None, None, _stream()) == capi.ERR_INVALID_ARG
    assert capi.swin_wattn_set_bias(h, None, _stream()) == capi.ERR_INVALID_ARG
    assert capi.swin_wattn_destroy(h) == capi.OK


def test_destroyed_plan_is_refused():
    h, _ = _plan()
    assert capi.swin_wattn_destroy(h) == capi.OK
    out = torch.zeros(1, 14, 14, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(1, 14, 14, 192, dtype=torch.bfloat16, device="cuda")
    assert capi.swin_wattn_fwd(h, q.data_ptr(), out.data_ptr(), _stream()) == capi.ERR_BAD_PLAN
    assert capi.swin_wattn_destroy(h) == capi.ERR_BAD_PLAN


def test_empty_batch_is_a_no_op_and_zeroes_the_table_gradient():
    h, _ = _plan(B=0)
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    out = torch.full((16,), 7.0, dtype=torch.bfloat16, device="cuda")
    assert capi.swin_wattn_fwd(h, q.data_ptr(), out.data_ptr(), _stream()) == capi.OK
    dt = torch.full((169, 2), 3.0, device="cuda")
    assert capi.swin_wattn_bwd(h, q.data_ptr(), q.data_ptr(), out.data_ptr(), dt.data_ptr(),
                               _stream()) == capi.OK
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(dt == 0)
    assert capi.swin_wattn_destroy(h) == capi.OK


def test_backward_for_twelve_by_twelve_windows_is_unsupported():
    h, _ = _plan(B=1, H=24, W=24, M=12, s=6)
    q = torch.zeros(1, 24, 24, 192, dtype=torch.bfloat16, device="cuda")
    d = torch.zeros(1, 24, 24, 64, dtype=torch.bfloat16, device="cuda")
    dt = torch.zeros(529, 2, device="cuda")
    assert capi.swin_wattn_bwd(h, q.data_ptr(), d.data_ptr(), q.data_ptr(), dt.data_ptr(),
                               _stream()) == capi.ERR_UNSUPPORTED
    assert capi.swin_wattn_destroy(h) == capi.OK


def test_launch_count_tracks_calls():
    capi.swin_wattn_launch_count(reset=True)
    h, _ = _plan()
    q = torch.zeros(1, 14, 14, 192, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 14, 14, 64, dtype=torch.bfloat16, device="cuda")
    assert capi.swin_wattn_fwd(h, q.data_ptr(), out.data_ptr(), _stream()) == capi.OK
    # the bias tables (mma fragments, mask fragments, dense bias), the dense mask, forward
    # (the tcgen05 tables are built only before a tcgen05 forward)
    assert capi.swin_wattn_launch_count() == 3
    assert capi.swin_wattn_destroy(h) == capi.OK
    assert isinstance(ctypes.c_int(0).value, int)

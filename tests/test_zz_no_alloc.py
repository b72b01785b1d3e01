"""swin_wattn_bwd_noalloc: the backward for callers that cannot allocate device memory
when they run it (a runtime with a device memory plan fixed at start-up, or a framework
whose allocator must own every device byte), so they cannot create a plan. Called
through the C ABI twice in a row, it must give the same dqkv and bias-table gradient as
the plan-based swin_wattn_bwd, within the parity tolerances of the other GPU tests.

Kept in a file of its own that pytest collects last; it passes alone in a fresh process
and after the other tests."""
import pytest
import torch

from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import assert_close, plan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from swin_window_attention_gb300 import build
    build.build()
    capi.load()


@pytest.mark.parametrize("name", ["swin_b224_s2", "swin_b224_s4"])
def test_noalloc_backward_matches_plan_backward_twice(name):
    wl = inputs.BY_NAME[name].with_batch(16)
    qkv, table, dout = inputs.make_qkv(wl), inputs.make_table(wl), inputs.make_dout(wl)
    q, d, t = qkv.cuda(), dout.cuda(), table.cuda()
    att = plan(wl, t)
    ref_dq, ref_dt = att.bwd(q, d)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        dq = torch.full_like(q, float("nan"))
        dt = torch.full_like(t, float("nan"))
        rc = capi.swin_wattn_bwd_noalloc(q.data_ptr(), d.data_ptr(), dq.data_ptr(), dt.data_ptr(),
                                         t.data_ptr(), wl.B, wl.H, wl.W, wl.C, wl.nH, wl.M, wl.s,
                                         capi.BF16, stream)
        assert rc == capi.OK, capi.swin_wattn_last_error()
        torch.cuda.synchronize()
        assert_close("noalloc dqkv", dq, ref_dq.double().cpu().numpy())
        assert_close("noalloc dtable", dt, ref_dt.double().cpu().numpy())
    att.close()


def test_noalloc_refuses_shapes_beyond_its_working_memory():
    # 160 heads of 7x7 windows need more than the fixed working memory for bias fragments.
    nH, M = 160, 7
    t = torch.zeros((2 * M - 1) ** 2, nH, device="cuda")
    q = torch.zeros(1, 7, 7, 3 * 32 * nH, dtype=torch.bfloat16, device="cuda")
    d = torch.zeros(1, 7, 7, 32 * nH, dtype=torch.bfloat16, device="cuda")
    rc = capi.swin_wattn_bwd_noalloc(q.data_ptr(), d.data_ptr(), q.data_ptr(), t.data_ptr(),
                                     t.data_ptr(), 1, 7, 7, 32 * nH, nH, M, 0, capi.BF16,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == capi.ERR_UNSUPPORTED
    assert "working memory" in capi.swin_wattn_last_error()

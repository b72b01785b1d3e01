"""The forward's bounded waits: a window whose loads are withheld (a debug switch of the
library) makes its pipeline wait run out; the kernel records SWIN_WATTN_ERR_TIMEOUT and
returns instead of hanging, and the next call on the same context is correct again."""
import pytest
import torch

from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import assert_close, oracle_fwd, plan, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from swin_window_attention_gb300 import build
    build.build()
    capi.load()


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_withheld_window_times_out_and_context_recovers(dt):
    wl = workload(2, 14, 14, 64, 2, 7, 3, dt, seed=11)
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.cuda())
    q = qkv.cuda()
    stream = torch.cuda.current_stream().cuda_stream
    assert capi.swin_wattn_debug_withhold(att.handle, 5) == capi.OK
    att.fwd(q)
    assert capi.swin_wattn_sync(att.handle, stream) == capi.ERR_TIMEOUT
    assert capi.swin_wattn_debug_withhold(att.handle, -1) == capi.OK
    y = att.fwd(q)
    assert capi.swin_wattn_sync(att.handle, stream) == capi.OK
    assert_close("Y after recovery", y, oracle_fwd(qkv, table, wl))
    att.close()

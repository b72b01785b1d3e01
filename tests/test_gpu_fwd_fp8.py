"""The forward on 8-bit operands (OCP FP8 E4M3 q, k, v with per-tensor scales) against the
fp64 oracle applied to the decoded values: the same tolerance as the bf16 forward, on
shapes with 1 to 3 windows per CTA range, with and without the shift, wide C, a full-size
stage on every image, determinism, and the refusals."""
import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import Accum, assert_close, batch_chunks, plan, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from swin_window_attention_gb300 import build
    build.build()
    oracle.build()
    capi.load()


def _ref(q8, scales, table, wl, batches=None):
    d = inputs.fp8_decoded_f64(q8 if batches is None else q8[batches], scales, wl.C)
    return oracle.fwd(d, table.double().numpy(), wl.nH, wl.M, wl.s)


@pytest.mark.parametrize("B,H,W,C,nH,s", [(1, 7, 7, 64, 2, 3), (1, 14, 21, 64, 2, 3), (2, 14, 14, 96, 3, 3),
                                          (3, 21, 28, 64, 2, 3), (2, 14, 14, 96, 3, 0), (2, 7, 7, 64, 2, 6),
                                          (5, 7, 7, 1536, 48, 0), (4, 56, 56, 192, 6, 3)])
def test_fp8_forward_against_oracle(B, H, W, C, nH, s):
    wl = workload(B, H, W, C, nH, 7, s, "bf16", seed=13 * B + H + W + s)
    q8, scales = inputs.make_qkv_fp8(wl)
    table = inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    y = att.fwd_fp8(q8.to(DEV), scales)
    att.device_status()
    assert y.dtype == torch.bfloat16 and y.shape == (B, H, W, C)
    assert_close("Y", y, _ref(q8, scales, table, wl))
    att.close()


def test_fp8_forward_scales_enter_as_defined():
    """Scaling the decoded tensors by powers of two must give the same attention when the
    scales absorb it: (q8, 2 sq) with (k8, sk / 2) leaves q.k unchanged; v's scale scales
    the output."""
    wl = workload(2, 14, 14, 64, 2, 7, 3, "bf16", seed=77)
    q8, (sq, sk, sv) = inputs.make_qkv_fp8(wl)
    table = inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    q8d = q8.to(DEV)
    y1 = att.fwd_fp8(q8d, (sq, sk, sv)).float()
    y2 = att.fwd_fp8(q8d, (2 * sq, sk / 2, sv)).float()
    y3 = att.fwd_fp8(q8d, (sq, sk, 4 * sv)).float()
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert torch.equal(4 * y1, y3)
    assert_close("Y", y1, _ref(q8, (sq, sk, sv), table, wl))
    att.close()


def test_fp8_forward_full_size_stage_and_determinism():
    wl = inputs.BY_NAME["swin_l224_s1"]
    q8, scales = inputs.make_qkv_fp8(wl)
    table = inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    q8d = q8.to(DEV)
    y = att.fwd_fp8(q8d, scales)
    y2 = att.fwd_fp8(q8d, scales)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    yc = y.cpu()
    acc = Accum()
    for bs in batch_chunks(wl.B):
        acc.add(yc[bs], _ref(q8, scales, table, wl, slice(bs[0], bs[-1] + 1)))
    acc.check("Y")
    att.close()


def test_fp8_forward_refusals():
    s = torch.cuda.current_stream().cuda_stream
    q8 = torch.zeros(1, 8, 8, 192, dtype=torch.uint8, device=DEV)
    out = torch.zeros(1, 8, 8, 64, dtype=torch.bfloat16, device=DEV)
    wl4 = workload(1, 8, 8, 64, 2, 4, 2, "bf16", seed=1)
    att4 = plan(wl4, inputs.make_table(wl4).to(DEV))
    assert capi.swin_wattn_fwd_fp8(att4.handle, q8.data_ptr(), 1.0, 1.0, 1.0, out.data_ptr(), s) == capi.ERR_UNSUPPORTED
    att4.close()
    wl = workload(1, 7, 7, 64, 2, 7, 3, "bf16", seed=2)
    att = plan(wl, inputs.make_table(wl).to(DEV))
    q7 = torch.zeros(1, 7, 7, 192, dtype=torch.uint8, device=DEV)
    o7 = torch.full((1, 7, 7, 64), 3.0, dtype=torch.bfloat16, device=DEV)
    f = lambda sq, sk, sv, qp=q7.data_ptr(): capi.swin_wattn_fwd_fp8(att.handle, qp, sq, sk, sv, o7.data_ptr(), s)
    for bad in ((0.0, 1.0, 1.0), (1.0, -1.0, 1.0), (1.0, 1.0, float("inf")), (1.0, 1.0, float("nan")),
                (1e30, 1e30, 1.0), (1e-30, 1e-30, 1.0)):
        assert f(*bad) == capi.ERR_INVALID_ARG, bad
    assert f(1.0, 1.0, 1.0, q7.data_ptr() + 1) == capi.ERR_MISALIGNED
    torch.cuda.synchronize()
    assert torch.all(o7 == 3.0)  # nothing launched
    wl32 = workload(1, 7, 7, 64, 2, 7, 3, "fp32", seed=3)
    att32 = plan(wl32, inputs.make_table(wl32).to(DEV))
    assert capi.swin_wattn_fwd_fp8(att32.handle, q7.data_ptr(), 1.0, 1.0, 1.0, o7.data_ptr(), s) == capi.ERR_UNSUPPORTED
    att32.close()
    att.close()

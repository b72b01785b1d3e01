"""swin_wattn_bwd_noalloc: the backward for callers that cannot allocate device memory
when they run it (a runtime with a device memory plan fixed at start-up, or a framework
whose allocator must own every device byte), so they cannot create a plan.

It runs the plan backward's mma.sync kernels on fragments built by the plan's own
fragment kernel into a fixed array inside the library, so its dqkv and bias-table gradient
must equal the plan-based swin_wattn_bwd with that kernel bit for bit, call after call,
whatever ran before it on the shared array. One case is also compared with the fp64 oracle directly.

Kept in a file of its own that pytest collects last; it passes alone in a fresh process
and after the other tests."""
import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import assert_close, oracle_bwd, plan, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from swin_window_attention_gb300 import build
    build.build()
    oracle.build()
    capi.load()


def noalloc(wl, q, d, t):
    """dqkv, dtable from the entry point, into outputs pre-filled with NaN."""
    dq = torch.full_like(q, float("nan"))
    dt = torch.full_like(t, float("nan"))
    rc = capi.swin_wattn_bwd_noalloc(q.data_ptr(), d.data_ptr(), dq.data_ptr(), dt.data_ptr(),
                                     t.data_ptr(), wl.B, wl.H, wl.W, wl.C, wl.nH, wl.M, wl.s,
                                     capi.FP32 if wl.dtype == "fp32" else capi.BF16,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == capi.OK, capi.swin_wattn_last_error()
    return dq, dt


def plan_bwd(wl, q, d, t):
    att = plan(wl, t)
    att.set_bwd_kernel(capi.KERNEL_MMA_SYNC)
    dq, dt = att.bwd(q, d)
    torch.cuda.synchronize()
    att.close()
    return dq, dt


def inputs_of(wl):
    return (inputs.make_qkv(wl).cuda(), inputs.make_dout(wl).cuda(), inputs.make_table(wl).cuda())


@pytest.mark.parametrize("name", ["swin_b224_s2", "swin_b224_s4"])
def test_noalloc_backward_equals_plan_backward_twice(name):
    wl = inputs.BY_NAME[name].with_batch(16)
    q, d, t = inputs_of(wl)
    ref_dq, ref_dt = plan_bwd(wl, q, d, t)
    for _ in range(2):
        dq, dt = noalloc(wl, q, d, t)
        torch.cuda.synchronize()
        assert torch.equal(dq, ref_dq)
        assert torch.equal(dt, ref_dt)


SMALL = [
    # B, H, W, C, nH, M, s, dtype: window 4, fp32 I/O, and a few-head shape
    (1, 8, 8, 64, 2, 4, 2, "fp32"),
    (2, 8, 16, 32, 1, 4, 1, "bf16"),
    (1, 14, 14, 64, 2, 7, 3, "fp32"),
    (2, 14, 14, 96, 3, 7, 3, "bf16"),
]


@pytest.mark.parametrize("B,H,W,C,nH,M,s,dt", SMALL)
def test_noalloc_backward_equals_plan_backward_small(B, H, W, C, nH, M, s, dt):
    wl = workload(B, H, W, C, nH, M, s, dt, seed=5 * B + H + M + s)
    q, d, t = inputs_of(wl)
    ref_dq, ref_dt = plan_bwd(wl, q, d, t)
    for _ in range(2):
        dq, dtab = noalloc(wl, q, d, t)
        torch.cuda.synchronize()
        assert torch.equal(dq, ref_dq)
        assert torch.equal(dtab, ref_dt)


def test_noalloc_after_a_larger_shape_on_the_shared_array():
    """A many-head, many-CTA call leaves fragments and partials in the shared array; the
    few-head call after it must not see any of them."""
    big = inputs.BY_NAME["swin_b224_s4"].with_batch(8)          # 32 heads, every CTA busy
    small = workload(1, 14, 14, 64, 2, 7, 3, "bf16", seed=41)  # 2 heads, 4 windows
    qb, db, tb = inputs_of(big)
    qs, ds, ts = inputs_of(small)
    ref_dq, ref_dt = plan_bwd(small, qs, ds, ts)
    for _ in range(2):
        noalloc(big, qb, db, tb)
        dq, dt = noalloc(small, qs, ds, ts)
        torch.cuda.synchronize()
        assert torch.equal(dq, ref_dq)
        assert torch.equal(dt, ref_dt)


def test_noalloc_against_the_oracle():
    wl = workload(2, 14, 21, 96, 3, 7, 3, "bf16", seed=43)
    qkv, dout, table = inputs.make_qkv(wl), inputs.make_dout(wl), inputs.make_table(wl)
    dq, dt = noalloc(wl, qkv.cuda(), dout.cuda(), table.cuda())
    torch.cuda.synchronize()
    ref_dq, ref_dt = oracle_bwd(qkv, dout, table, wl)
    assert_close("noalloc dqkv", dq, ref_dq)
    assert_close("noalloc dtable", dt, ref_dt)


def test_noalloc_counts_its_launches():
    wl = workload(1, 14, 14, 64, 2, 7, 3, "bf16", seed=44)
    q, d, t = inputs_of(wl)
    torch.cuda.synchronize()
    capi.swin_wattn_launch_count(reset=True)
    noalloc(wl, q, d, t)
    assert capi.swin_wattn_launch_count() == 3
    torch.cuda.synchronize()


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

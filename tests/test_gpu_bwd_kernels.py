"""The two backward kernels (tcgen05 + tensor memory, and warp-level mma.sync) against the
fp64 oracle: small shapes compared in full, with one and two window pairs per CTA range,
an odd window count (a pair with one window), every wrap of a shifted layer and many
heads; the Swin-B 224 training stages at full size on every image; determinism; the
kernel choice itself."""
import numpy as np
import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import Accum, assert_close, batch_chunks, oracle_bwd, plan, workload

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


KERNELS = [capi.KERNEL_TCGEN05, capi.KERNEL_MMA_SYNC]

SMALL = [
    # B, H, W, C, nH, s
    (1, 7, 7, 64, 2, 3),      # one window: a pair with one window, right and bottom wrap
    (1, 14, 14, 64, 2, 3),    # two pairs: every window class
    (3, 21, 14, 64, 2, 3),    # odd window count per range
    (2, 14, 14, 96, 3, 0),    # no shift
    (2, 14, 28, 64, 2, 4),    # the bottom wrap as two row bands (7 - s even)
    (2, 7, 7, 64, 2, 6),
    (4, 7, 7, 1024, 32, 0),   # many heads, few windows
    (4, 56, 56, 128, 4, 3),   # several pairs per CTA range
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("B,H,W,C,nH,s", SMALL)
def test_bwd_kernel_against_oracle(kernel, B, H, W, C, nH, s):
    wl = workload(B, H, W, C, nH, 7, s, "bf16", seed=13 * B + H + W + s)
    qkv, table, dout = inputs.make_qkv(wl), inputs.make_table(wl), inputs.make_dout(wl)
    att = plan(wl, table.to(DEV))
    att.set_bwd_kernel(kernel)
    assert att.bwd_kernel == kernel
    dq, dt = att.bwd(qkv.to(DEV), dout.to(DEV))
    att.device_status()
    ref_dq, ref_dt = oracle_bwd(qkv, dout, table, wl)
    assert_close("dqkv", dq, ref_dq)
    assert_close("dtable", dt, ref_dt)
    att.close()


@pytest.mark.parametrize("name", [w.name for w in inputs.WORKLOADS if w.bwd])
def test_tcgen05_bwd_workload_every_image(name):
    wl = inputs.BY_NAME[name]
    qkv, table, dout = inputs.make_qkv(wl), inputs.make_table(wl), inputs.make_dout(wl)
    att = plan(wl, table.to(DEV))
    att.set_bwd_kernel(capi.KERNEL_TCGEN05)
    dqkv, dtab = att.bwd(qkv.to(DEV), dout.to(DEV))
    att.device_status()
    dqkv, dtab = dqkv.cpu(), dtab.cpu()
    att.close()
    acc = Accum()
    ref_dt = np.zeros(tuple(table.shape))
    for bs in batch_chunks(wl.B):
        ref_dq, dt_part = oracle_bwd(qkv, dout, table, wl, batches=bs)
        acc.add(dqkv[bs], ref_dq)
        ref_dt += dt_part
    acc.check(f"{name} dqkv tcgen05")
    assert_close(f"{name} dtable tcgen05", dtab, ref_dt)


def test_tcgen05_bwd_is_deterministic_and_follows_a_new_bias():
    wl = inputs.BY_NAME["swin_b224_s3"]
    qkv, table, dout = inputs.make_qkv(wl), inputs.make_table(wl), inputs.make_dout(wl)
    att = plan(wl, table.to(DEV))
    att.set_bwd_kernel(capi.KERNEL_TCGEN05)
    q, d = qkv.to(DEV), dout.to(DEV)
    a1, t1 = att.bwd(q, d)
    a2, t2 = att.bwd(q, d)
    torch.cuda.synchronize()
    assert torch.equal(a1, a2) and torch.equal(t1, t2)
    # a new table reaches the kernel's bias image (built lazily before the next backward)
    small = workload(2, 14, 14, 64, 2, 7, 3, "bf16", seed=71)
    qs, ts, ds = inputs.make_qkv(small), inputs.make_table(small), inputs.make_dout(small)
    t2 = inputs.trunc_normal(ts.shape, 4321) * 2.0
    att2 = plan(small, ts.to(DEV))
    att2.set_bwd_kernel(capi.KERNEL_TCGEN05)
    att2.bwd(qs.to(DEV), ds.to(DEV))
    att2.set_bias(t2.to(DEV))
    dq, dt = att2.bwd(qs.to(DEV), ds.to(DEV))
    att2.device_status()
    ref_dq, ref_dt = oracle_bwd(qs, ds, t2, small)
    assert_close("dqkv after set_bias", dq, ref_dq)
    assert_close("dtable after set_bias", dt, ref_dt)
    att.close()
    att2.close()


@pytest.mark.parametrize("M,dt", [(4, "bf16"), (7, "fp32"), (12, "bf16")])
def test_tcgen05_bwd_refused_where_it_does_not_apply(M, dt):
    wl = workload(1, 2 * M, 2 * M, 64, 2, M, 1, dt)
    att = plan(wl, inputs.make_table(wl).to(DEV))
    kern = att.bwd_kernel
    assert capi.swin_wattn_set_bwd_kernel(att.handle, capi.KERNEL_TCGEN05) == capi.ERR_UNSUPPORTED
    assert att.bwd_kernel == kern
    assert capi.swin_wattn_set_bwd_kernel(att.handle, 9) == capi.ERR_INVALID_ARG
    att.close()


def test_tcgen05_bwd_output_16_byte_aligned():
    """dqkv on a 16-byte (not 32-byte) boundary: the kernel stores in 16-byte pieces."""
    wl = workload(2, 14, 14, 64, 2, 7, 3, "bf16", seed=77)
    qkv, table, dout = inputs.make_qkv(wl), inputs.make_table(wl), inputs.make_dout(wl)
    att = plan(wl, table.to(DEV))
    att.set_bwd_kernel(capi.KERNEL_TCGEN05)
    buf = torch.full((qkv.numel() + 16,), float("nan"), dtype=qkv.dtype, device=DEV)
    dq = buf[8:8 + qkv.numel()].view(qkv.shape)
    assert dq.data_ptr() % 32 == 16
    _, dt = att.bwd(qkv.to(DEV), dout.to(DEV), dqkv=dq)
    att.device_status()
    ref_dq, ref_dt = oracle_bwd(qkv, dout, table, wl)
    assert_close("dqkv 16-byte aligned", dq, ref_dq)
    assert_close("dtable", dt, ref_dt)
    assert torch.isnan(buf[:8]).all() and torch.isnan(buf[8 + qkv.numel():]).all()
    att.close()


@pytest.mark.parametrize("B,H,W,C,nH,M,s,dt,expect", [
    (2, 56, 56, 128, 4, 7, 3, "bf16", capi.KERNEL_TCGEN05),   # 8 windows wide, shifted
    (2, 28, 28, 256, 8, 7, 3, "bf16", capi.KERNEL_TCGEN05),
    (2, 14, 14, 512, 16, 7, 3, "bf16", capi.KERNEL_MMA_SYNC),  # 2 windows wide, shifted
    (2, 14, 14, 512, 16, 7, 0, "bf16", capi.KERNEL_TCGEN05),   # not shifted
    (2, 7, 7, 1024, 32, 7, 0, "bf16", capi.KERNEL_TCGEN05),
    (2, 56, 56, 128, 4, 7, 3, "fp32", capi.KERNEL_MMA_SYNC),   # tcgen05 is bf16 only
    (2, 16, 16, 64, 2, 4, 2, "bf16", capi.KERNEL_MMA_SYNC),    # window 4
])
def test_auto_backward_kernel_choice(B, H, W, C, nH, M, s, dt, expect):
    wl = workload(B, H, W, C, nH, M, s, dt)
    att = plan(wl, inputs.make_table(wl).to(DEV))
    assert att.bwd_kernel == expect
    att.set_bwd_kernel(capi.KERNEL_MMA_SYNC)
    assert att.bwd_kernel == capi.KERNEL_MMA_SYNC
    att.set_bwd_kernel(capi.KERNEL_AUTO)
    assert att.bwd_kernel == expect
    att.close()

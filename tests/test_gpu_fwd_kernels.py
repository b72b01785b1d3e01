"""The two forward kernels (tcgen05 + tensor memory, and warp-level mma.sync) on the
same inputs: each against the fp64 oracle, the kernel choice itself, and the tcgen05
kernel's device status word after its bounded waits."""
import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import Accum, assert_close, batch_chunks, oracle_fwd, plan, workload

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

SMALL_M7 = [
    # B, H, W, C, nH, s: windows per CTA range over 1 (a pair with one window), 2 and 3
    (1, 7, 7, 64, 2, 3),
    (1, 14, 21, 64, 2, 3),
    (2, 14, 14, 96, 3, 3),
    (3, 21, 28, 64, 2, 3),
    (2, 14, 14, 96, 3, 0),
    (2, 7, 7, 64, 2, 6),
    (5, 7, 7, 1536, 48, 0),
    (4, 56, 56, 192, 6, 3),
    (3, 28, 35, 128, 4, 5),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("B,H,W,C,nH,s", SMALL_M7)
def test_fwd_kernel_against_oracle(kernel, B, H, W, C, nH, s):
    wl = workload(B, H, W, C, nH, 7, s, "bf16", seed=11 * B + H + W + s)
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    att.set_fwd_kernel(kernel)
    assert att.fwd_kernel == kernel
    y = att.fwd(qkv.to(DEV))
    att.device_status()
    assert_close("Y", y, oracle_fwd(qkv, table, wl))
    att.close()


@pytest.mark.parametrize("name", [w.name for w in inputs.WORKLOADS if w.M == 7 and w.dtype == "bf16"])
def test_fwd_kernels_agree_on_workloads(name):
    """Full-size workloads: both kernels against the oracle on every image."""
    wl = inputs.BY_NAME[name]
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    att.set_fwd_kernel(capi.KERNEL_TCGEN05)
    q = qkv.to(DEV)
    y_tc = att.fwd(q)
    att.device_status()
    att.set_fwd_kernel(capi.KERNEL_MMA_SYNC)
    y_mma = att.fwd(q)
    torch.cuda.synchronize()
    att.close()
    y_tc, y_mma = y_tc.cpu(), y_mma.cpu()
    acc_tc, acc_mma = Accum(), Accum()
    for bs in batch_chunks(wl.B):
        ref = oracle_fwd(qkv, table, wl, batches=bs)
        acc_tc.add(y_tc[bs], ref)
        acc_mma.add(y_mma[bs], ref)
    acc_tc.check(f"{name} Y tcgen05")
    acc_mma.check(f"{name} Y mma.sync")


SMALL_M12 = [
    # B, H, W, C, nH, s: one window; every window class of a shifted layer (interior, right
    # wrap, bottom wrap, corner); several windows per CTA range; many heads; odd shifts
    (1, 12, 12, 64, 2, 0),
    (1, 24, 24, 64, 2, 6),
    (2, 36, 24, 96, 3, 6),
    (1, 12, 12, 1536, 48, 0),
    (3, 24, 36, 64, 2, 6),
    (2, 24, 24, 64, 2, 5),
    (1, 24, 24, 64, 2, 1),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("B,H,W,C,nH,s", SMALL_M12)
def test_fwd12_kernel_against_oracle(kernel, B, H, W, C, nH, s):
    wl = workload(B, H, W, C, nH, 12, s, "bf16", seed=13 * B + H + W + s)
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    att.set_fwd_kernel(kernel)
    assert att.fwd_kernel == kernel
    y = att.fwd(qkv.to(DEV))
    att.device_status()
    assert_close("Y", y, oracle_fwd(qkv, table, wl))
    att.close()


@pytest.mark.parametrize("name", [w.name for w in inputs.WORKLOADS if w.M == 12 and w.dtype == "bf16"])
def test_fwd12_tcgen05_workload_every_image(name):
    """Full-size 12x12 workloads: the tcgen05 kernel against the oracle on every image, and
    bit-identical on a second call."""
    wl = inputs.BY_NAME[name]
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    att.set_fwd_kernel(capi.KERNEL_TCGEN05)
    q = qkv.to(DEV)
    y = att.fwd(q)
    y2 = att.fwd(q)
    att.device_status()
    assert torch.equal(y, y2)
    att.close()
    y = y.cpu()
    acc = Accum()
    for bs in batch_chunks(wl.B):
        acc.add(y[bs], oracle_fwd(qkv, table, wl, batches=bs))
    acc.check(f"{name} Y tcgen05")


@pytest.mark.parametrize("name,expect", [
    ("swin_l384_s1", capi.KERNEL_TCGEN05),
    ("swin_l384_s2", capi.KERNEL_TCGEN05),
    ("swin_l384_s3", capi.KERNEL_MMA_SYNC),
    ("swin_l384_s4", capi.KERNEL_MMA_SYNC),
    ("swin_l224_s1", capi.KERNEL_MMA_SYNC),
])
def test_auto_forward_kernel_choice(name, expect):
    """AUTO takes the tcgen05 kernel for 12x12 windows with at least 16 window-heads per SM
    (on this GPU's SM count), else the mma.sync kernel; choosing a kernel and going back to
    AUTO restores the choice."""
    wl = inputs.BY_NAME[name]
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    wh = wl.B * (wl.H // wl.M) * (wl.W // wl.M) * wl.nH
    if wl.M == 12 and (wh >= 16 * nsm) != (expect == capi.KERNEL_TCGEN05):
        pytest.skip(f"{nsm} SMs: the window-head count {wh} falls on the other side of the rule")
    att = plan(wl, inputs.make_table(wl).to(DEV))
    assert att.fwd_kernel == expect
    att.set_fwd_kernel(capi.KERNEL_MMA_SYNC)
    assert att.fwd_kernel == capi.KERNEL_MMA_SYNC
    att.set_fwd_kernel(capi.KERNEL_AUTO)
    assert att.fwd_kernel == expect
    att.close()


def test_tcgen05_kernel_is_deterministic():
    wl = inputs.BY_NAME["swin_l224_s2"]
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    att.set_fwd_kernel(capi.KERNEL_TCGEN05)
    q = qkv.to(DEV)
    a, b = att.fwd(q), att.fwd(q)
    att.device_status()
    assert torch.equal(a, b)
    att.close()


@pytest.mark.parametrize("M,dt", [(4, "bf16"), (12, "fp32"), (7, "fp32")])
def test_tcgen05_kernel_refused_where_it_does_not_apply(M, dt):
    wl = workload(1, 2 * M, 2 * M, 64, 2, M, 1, dt)
    table = inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    assert att.fwd_kernel == capi.KERNEL_MMA_SYNC
    rc = capi.swin_wattn_set_fwd_kernel(att.handle, capi.KERNEL_TCGEN05)
    assert rc == capi.ERR_UNSUPPORTED
    assert att.fwd_kernel == capi.KERNEL_MMA_SYNC
    assert capi.swin_wattn_set_fwd_kernel(att.handle, 7) == capi.ERR_INVALID_ARG
    att.close()


def test_new_bias_reaches_the_tcgen05_kernel_whenever_it_is_chosen():
    """set_bias rebuilds the mma fragments and the dense bias in one launch; the tcgen05
    kernel's tables follow before its next forward, whether the kernel was chosen before
    or after the new bias, and the dense bias dump matches the new table."""
    wl = workload(2, 14, 14, 64, 2, 7, 3, "bf16", seed=31)
    qkv, t1 = inputs.make_qkv(wl), inputs.make_table(wl)
    t2 = inputs.trunc_normal(t1.shape, 1234) * 8
    q = qkv.to(DEV)
    ref2 = oracle_fwd(qkv, t2, wl)
    # chosen after the new bias
    att = plan(wl, t1.to(DEV))
    att.set_bias(t2.to(DEV))
    att.set_fwd_kernel(capi.KERNEL_TCGEN05)
    assert_close("Y", att.fwd(q), ref2)
    att.device_status()
    att.close()
    # chosen before: a forward with the first table, then the new bias
    att = plan(wl, t1.to(DEV))
    att.set_fwd_kernel(capi.KERNEL_TCGEN05)
    assert_close("Y", att.fwd(q), oracle_fwd(qkv, t1, wl))
    att.set_bias(t2.to(DEV))
    assert_close("Y", att.fwd(q), ref2)
    # and back to the mma.sync kernel, which reads the fragments
    att.set_fwd_kernel(capi.KERNEL_MMA_SYNC)
    assert_close("Y", att.fwd(q), ref2)
    att.device_status()
    att.close()

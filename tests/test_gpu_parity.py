"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Index maps (gather, relative index, mask, dense bias) must match bit for bit; Y, dqkv
and the bias-table gradient must be within max-abs 1e-2 and relative-L2 5e-3 of the
oracle applied to the same bf16-rounded inputs. Small cases and the full-size workloads
(in the bench's launch configuration) are compared element by element on every image;
the oracle runs a few images at a time.
"""
import numpy as np
import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import (Accum, assert_close, assert_fwd_every_image, batch_chunks, oracle_bwd,
                            oracle_fwd, plan, workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from swin_window_attention_gb300 import build
    build.build()
    oracle.build()
    capi.load()


DEV = "cuda"

# ---------------------------------------------------------------------------------
# index maps, bit-exact
# ---------------------------------------------------------------------------------

MAP_CASES = [(8, 8, 4, 2), (56, 56, 7, 3), (28, 28, 7, 3), (14, 14, 7, 3), (7, 7, 7, 0),
             (7, 7, 7, 3), (96, 96, 12, 6), (12, 12, 12, 0), (12, 24, 12, 6), (14, 28, 7, 6),
             (56, 56, 7, 0)]


@pytest.mark.parametrize("H,W,M,s", MAP_CASES)
def test_index_maps_bit_exact(H, W, M, s):
    nH = 3
    table = inputs.trunc_normal(((2 * M - 1) ** 2, nH), 100 + M)
    att = capi.WindowAttention(1, H, W, 32 * nH, nH, M, s, table.to(DEV))
    gather, relidx, mask, dense = att.debug_maps()
    torch.cuda.synchronize()
    assert np.array_equal(gather.cpu().numpy(), oracle.gather(H, W, M, s))
    assert np.array_equal(relidx.cpu().numpy(), oracle.relidx(M))
    om = oracle.mask(H, W, M, s)
    assert np.array_equal(mask.cpu().numpy(), om.astype(np.float32))
    od = oracle.dense_bias(table.double().numpy(), nH, M).astype(np.float32)
    assert np.array_equal(dense.cpu().numpy(), od)
    att.close()


# ---------------------------------------------------------------------------------
# forward, small shapes compared in full
# ---------------------------------------------------------------------------------

FWD_SMALL = [
    # B, H, W, C, nH, M, s, dtype
    (1, 8, 8, 64, 2, 4, 2, "fp32"),     # the tiny workload's shape
    (1, 8, 8, 64, 2, 4, 2, "bf16"),
    (2, 16, 12, 32, 1, 4, 3, "bf16"),
    (2, 14, 14, 96, 3, 7, 3, "bf16"),   # 4 windows, mask classes 0..3
    (3, 21, 28, 64, 2, 7, 3, "bf16"),   # non-square, several CTAs per head
    (2, 14, 14, 96, 3, 7, 0, "bf16"),
    (2, 7, 7, 64, 2, 7, 3, "bf16"),     # one shifted window per image
    (1, 14, 14, 64, 2, 7, 6, "fp32"),
    (1, 24, 36, 64, 2, 12, 6, "bf16"),
    (2, 12, 12, 64, 2, 12, 5, "bf16"),  # one shifted 12x12 window
    (1, 24, 24, 64, 2, 12, 0, "fp32"),
    (5, 7, 7, 1536, 48, 7, 0, "bf16"),  # many heads, few windows
]


@pytest.mark.parametrize("B,H,W,C,nH,M,s,dt", FWD_SMALL)
def test_fwd_small_full(B, H, W, C, nH, M, s, dt):
    wl = workload(B, H, W, C, nH, M, s, dt, seed=B + H + M + s)
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    y = att.fwd(qkv.to(DEV))
    torch.cuda.synchronize()
    assert y.dtype == (torch.float32 if dt == "fp32" else torch.bfloat16)
    assert_close("Y", y, oracle_fwd(qkv, table, wl))
    att.close()


def test_fwd_extreme_logits_are_finite_and_match():
    """q and k scaled by 6 (logits with a spread of tens) and a bias scaled by 200: the
    max subtraction must keep the softmax finite and accurate."""
    wl = workload(2, 14, 14, 64, 2, 7, 3, seed=3)
    qkv = inputs.make_qkv(wl).float()
    qkv[..., :2 * wl.C] *= 6.0
    qkv = qkv.to(torch.bfloat16)
    table = inputs.make_table(wl) * 200.0
    att = plan(wl, table.to(DEV))
    y = att.fwd(qkv.to(DEV))
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    assert_close("Y", y, oracle_fwd(qkv, table, wl))
    att.close()


def test_set_bias_re_expands():
    wl = workload(1, 14, 14, 64, 2, 7, 3, seed=4)
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    t2 = inputs.trunc_normal(table.shape, 999) * 10
    att.set_bias(t2.to(DEV))
    y = att.fwd(qkv.to(DEV))
    torch.cuda.synchronize()
    assert_close("Y", y, oracle_fwd(qkv, t2, wl))
    att.close()


# ---------------------------------------------------------------------------------
# forward at full workload size, in the bench's launch configuration
# ---------------------------------------------------------------------------------

FWD_WORKLOADS = [w.name for w in inputs.WORKLOADS]


@pytest.mark.parametrize("name", FWD_WORKLOADS)
def test_fwd_workload(name):
    wl = inputs.BY_NAME[name]
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    y = att.fwd(qkv.to(DEV)).cpu()
    torch.cuda.synchronize()
    att.close()
    assert_fwd_every_image(f"{name} Y", y, qkv, table, wl)


# ---------------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------------

BWD_SMALL = [
    (1, 8, 8, 64, 2, 4, 2, "fp32"),
    (2, 8, 16, 32, 1, 4, 1, "bf16"),
    (2, 14, 14, 96, 3, 7, 3, "bf16"),
    (3, 21, 14, 64, 2, 7, 3, "bf16"),
    (2, 14, 14, 64, 2, 7, 0, "bf16"),
    (2, 7, 7, 64, 2, 7, 4, "bf16"),
    (1, 14, 14, 64, 2, 7, 3, "fp32"),
    (4, 7, 7, 1024, 32, 7, 0, "bf16"),
]


@pytest.mark.parametrize("B,H,W,C,nH,M,s,dt", BWD_SMALL)
def test_bwd_small_full(B, H, W, C, nH, M, s, dt):
    wl = workload(B, H, W, C, nH, M, s, dt, seed=2 * B + H + M + s)
    qkv, table, dout = inputs.make_qkv(wl), inputs.make_table(wl), inputs.make_dout(wl)
    att = plan(wl, table.to(DEV))
    dqkv, dtab = att.bwd(qkv.to(DEV), dout.to(DEV))
    torch.cuda.synchronize()
    ref_dq, ref_dt = oracle_bwd(qkv, dout, table, wl)
    assert_close("dqkv", dqkv, ref_dq)
    assert_close("dtable", dtab, ref_dt)
    att.close()


@pytest.mark.parametrize("name", [w.name for w in inputs.WORKLOADS if w.bwd])
def test_bwd_workload(name):
    wl = inputs.BY_NAME[name]
    qkv, table, dout = inputs.make_qkv(wl), inputs.make_table(wl), inputs.make_dout(wl)
    att = plan(wl, table.to(DEV))
    dqkv, dtab = att.bwd(qkv.to(DEV), dout.to(DEV))
    dqkv, dtab = dqkv.cpu(), dtab.cpu()
    att.close()
    # every image's dqkv; the table gradient sums over every image, so the oracle's
    # per-chunk gradients are accumulated
    acc = Accum()
    ref_dt = np.zeros(tuple(table.shape))
    for bs in batch_chunks(wl.B):
        ref_dq, dt_part = oracle_bwd(qkv, dout, table, wl, batches=bs)
        acc.add(dqkv[bs], ref_dq)
        ref_dt += dt_part
    acc.check(f"{name} dqkv")
    assert_close(f"{name} dtable", dtab, ref_dt)


def test_bwd_is_deterministic():
    wl = inputs.BY_NAME["swin_b224_s3"]
    qkv, table, dout = inputs.make_qkv(wl), inputs.make_table(wl), inputs.make_dout(wl)
    att = plan(wl, table.to(DEV))
    q, d = qkv.to(DEV), dout.to(DEV)
    a1, t1 = att.bwd(q, d)
    a2, t2 = att.bwd(q, d)
    torch.cuda.synchronize()
    assert torch.equal(a1, a2) and torch.equal(t1, t2)
    att.close()


def test_batch_shards_concatenate_exactly():
    """Data-parallel emulation on one GPU: two batch shards give bit-identical Y and
    dqkv slices, and their table gradients sum to the full batch's within tolerance."""
    wl = inputs.BY_NAME["swin_b224_s2"]
    qkv, table, dout = inputs.make_qkv(wl), inputs.make_table(wl), inputs.make_dout(wl)
    q, d, t = qkv.to(DEV), dout.to(DEV), table.to(DEV)
    full = plan(wl, t)
    y = full.fwd(q)
    dq, dt = full.bwd(q, d)
    half = wl.B // 2
    parts = []
    for lo, hi in ((0, half), (half, wl.B)):
        sh = plan(wl.with_batch(hi - lo), t)
        parts.append((sh.fwd(q[lo:hi].contiguous()),) + sh.bwd(q[lo:hi].contiguous(),
                                                              d[lo:hi].contiguous()))
        torch.cuda.synchronize()
        sh.close()
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([p[0] for p in parts]), y)
    assert torch.equal(torch.cat([p[1] for p in parts]), dq)
    assert_close("dtable shard sum", parts[0][2] + parts[1][2], dt.double().cpu().numpy())
    full.close()


@pytest.mark.parametrize("name,batch,kernel", [
    ("swin_t_s1_swmsa", 32, capi.KERNEL_AUTO),
    ("tiny", 1, capi.KERNEL_AUTO),
    ("swin_l224_s3", 3, capi.KERNEL_AUTO),
    ("swin_l224_s2", 5, capi.KERNEL_TCGEN05),
    ("swin_l384_s1", 16, capi.KERNEL_AUTO),
    ("swin_l384_s3", 3, capi.KERNEL_TCGEN05),
])
def test_fwd_host_buffers_match_device_path(name, batch, kernel):
    """swin_wattn_fwd_host (pinned host in/out, chunked copy/compute pipeline) gives the
    device path's output bit for bit, for each forward kernel (the batch chunks of the host
    path launch with their own window ranges)."""
    wl = inputs.BY_NAME[name].with_batch(batch)
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    att = plan(wl, table.to(DEV))
    att.set_fwd_kernel(kernel)
    if kernel == capi.KERNEL_AUTO and wl.M == 12:
        # AUTO's rule for 12x12 windows: tcgen05 from 16 window-heads per SM
        nsm = torch.cuda.get_device_properties(0).multi_processor_count
        wh = wl.B * (wl.H // wl.M) * (wl.W // wl.M) * wl.nH
        assert att.fwd_kernel == (capi.KERNEL_TCGEN05 if wh >= 16 * nsm else capi.KERNEL_MMA_SYNC)
    ref = att.fwd(qkv.to(DEV)).cpu()
    qh = qkv.pin_memory()
    oh = torch.empty(ref.shape, dtype=ref.dtype).pin_memory()
    dq = torch.empty(qkv.shape, dtype=qkv.dtype, device=DEV)
    do = torch.empty(ref.shape, dtype=ref.dtype, device=DEV)
    for _ in range(2):
        oh.zero_()
        att.fwd_host(qh, oh, dq, do)
        torch.cuda.synchronize()
        assert torch.equal(oh, ref)
    att.close()

"""Failure detection on the GPU without a fault: every device-side wait of the library's
kernels is bounded, and a wait that runs out must end in an error status, not a hang.

The fault-injection build (libswin_wattn_debug.so, include/swin_wattn_debug.h) withholds
one mbarrier arrival at an armed site and shortens the bound to a few milliseconds. For
each site the test checks that the launch returns within seconds, that the host sees
SWIN_WATTN_ERR_TIMEOUT (attention kernels) or bit 0 of the status word (GEMM steps),
and that the next normal call, on the same plan, is correct against the oracle, so the
CTAs that gave up released their tensor memory and let their copies land."""
import ctypes
import time

import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import assert_close, assert_close_rounded, oracle_fwd, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"
WAIT_NS = 5_000_000        # 5 ms per wait while a site is armed
DEFAULT_WAIT_NS = 1_000_000_000


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from swin_window_attention_gb300 import build
    build.build(debug=True)
    oracle.build()
    lib = capi.load_debug()
    yield lib
    lib.swin_wattn_debug_set_fault(capi.FAULT_NONE, DEFAULT_WAIT_NS)


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _plan(lib, wl, table):
    h = ctypes.c_void_p()
    rc = lib.swin_wattn_plan(ctypes.byref(h), wl.B, wl.H, wl.W, wl.C, wl.nH, wl.M, wl.s, capi.BF16,
                             table.data_ptr(), _stream())
    assert rc == capi.OK
    return h.value


def _armed_then_clean_forward(lib, kernel, site, M=7):
    # 2 x 2 shifted windows per image, half of them in the last window column (gathered
    # four rows at a time or by cp.async), the others through the copy engine: 228 images
    # of 7x7 windows, or 40 of 12x12 windows
    wl = workload(228, 14, 14, 64, 2, 7, 3, seed=61) if M == 7 else workload(40, 24, 24, 64, 2, 12, 5, seed=62)
    qkv, table = inputs.make_qkv(wl), inputs.make_table(wl)
    q, t = qkv.to(DEV), table.to(DEV)
    y = torch.empty(wl.B, wl.H, wl.W, wl.C, dtype=torch.bfloat16, device=DEV)
    h = _plan(lib, wl, t)
    try:
        assert lib.swin_wattn_set_fwd_kernel(h, kernel) == capi.OK
        assert lib.swin_wattn_device_status(h, _stream()) == capi.OK
        assert lib.swin_wattn_debug_set_fault(site, WAIT_NS) == capi.OK
        t0 = time.monotonic()
        assert lib.swin_wattn_fwd(h, q.data_ptr(), y.data_ptr(), _stream()) == capi.OK
        rc = lib.swin_wattn_device_status(h, _stream())  # synchronises the stream
        elapsed = time.monotonic() - t0
        assert lib.swin_wattn_debug_set_fault(capi.FAULT_NONE, DEFAULT_WAIT_NS) == capi.OK
        assert rc == capi.ERR_TIMEOUT
        assert elapsed < 10.0, f"the timed-out launch took {elapsed:.1f} s"
        # the status word was cleared by the read; a clean forward on the same plan
        y.fill_(float("nan"))
        assert lib.swin_wattn_fwd(h, q.data_ptr(), y.data_ptr(), _stream()) == capi.OK
        assert lib.swin_wattn_device_status(h, _stream()) == capi.OK
        assert_close("Y after a timed-out launch", y, oracle_fwd(qkv, table, wl))
    finally:
        lib.swin_wattn_debug_set_fault(capi.FAULT_NONE, DEFAULT_WAIT_NS)
        torch.cuda.synchronize()
        lib.swin_wattn_destroy(h)


def test_mma_sync_forward_stage_wait_runs_out(dbg):
    _armed_then_clean_forward(dbg, capi.KERNEL_MMA_SYNC, capi.FAULT_FWD_MMA_SYNC)


@pytest.mark.parametrize("M", [7, 12])
def test_tcgen05_forward_wait_runs_out_and_tensor_memory_is_released(dbg, M):
    _armed_then_clean_forward(dbg, capi.KERNEL_TCGEN05, capi.FAULT_FWD_TCGEN05, M)


def _f64(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("step,T,C", [
    ("consumer", 4096, 192),      # output projection + bias + residual
    ("producer", 300, 192),       # statistics from the prep pass
    ("producer", 80001, 96),      # statistics summed on chip by four extra warps
])
def test_gemm_epilogue_wait_runs_out_and_tensor_memory_is_released(dbg, step, T, C):
    wl = workload(1, 1, T, C, C // 32, 1, 0, seed=T + C)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if step == "consumer":
        o, wp, bp, r = inputs.make_consumer(wl)
        od, wd, bd, rd = (x.to(DEV) for x in (o, wp, bp, r))
        y = torch.empty_like(od)

        def call():
            return dbg.swin_wattn_proj_residual(od.data_ptr(), wd.data_ptr(), bd.data_ptr(), rd.data_ptr(),
                                                y.data_ptr(), T, C, status.data_ptr(), _stream())

        def ref():
            return oracle.proj_residual(_f64(o), _f64(wp), _f64(bp), _f64(r))
    else:
        x, g, be, w, b = inputs.make_producer(wl)
        xd, gd, bed, wd, bd = (v.to(DEV) for v in (x, g, be, w, b))
        y = torch.empty(1, 1, T, 3 * C, dtype=torch.bfloat16, device=DEV)
        ws = torch.empty(max(dbg.swin_wattn_qkv_workspace_bytes(C, T), 1), dtype=torch.uint8, device=DEV)

        def call():
            return dbg.swin_wattn_qkv_proj(xd.data_ptr(), gd.data_ptr(), bed.data_ptr(), wd.data_ptr(),
                                           bd.data_ptr(), y.data_ptr(), T, C, 1e-5, ws.data_ptr(), ws.numel(),
                                           status.data_ptr(), _stream())

        def ref():
            return oracle.qkv_proj(_f64(x), _f64(g), _f64(be), _f64(w), _f64(b))
    try:
        assert dbg.swin_wattn_debug_set_fault(capi.FAULT_GEMM, WAIT_NS) == capi.OK
        t0 = time.monotonic()
        assert call() == capi.OK
        torch.cuda.synchronize()
        elapsed = time.monotonic() - t0
        assert dbg.swin_wattn_debug_set_fault(capi.FAULT_NONE, DEFAULT_WAIT_NS) == capi.OK
        assert int(status.item()) & 1 == 1
        assert elapsed < 10.0, f"the timed-out launch took {elapsed:.1f} s"
        status.zero_()
        y.fill_(float("nan"))
        assert call() == capi.OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close_rounded(f"{step} after a timed-out launch", y, ref())
    finally:
        dbg.swin_wattn_debug_set_fault(capi.FAULT_NONE, DEFAULT_WAIT_NS)
        torch.cuda.synchronize()

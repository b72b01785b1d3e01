"""ctypes binding of libswin_wattn.so (declared in include/swin_wattn.h).

Argument marshalling only: every function forwards to the C entry point of the same
name and returns its status code; ``WindowAttention`` wraps a plan for torch CUDA
tensors. Every step of the computation runs in the library's CUDA kernels. If the
library has not been built (``python -m swin_window_attention_gb300.build``), ``load()``
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libswin_wattn.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_MISALIGNED = 3
ERR_BAD_PLAN = 4
ERR_CUDA = 5
ERR_TIMEOUT = 6
BF16 = 0
FP32 = 1
KERNEL_AUTO = 0
KERNEL_MMA_SYNC = 1
KERNEL_TCGEN05 = 2

# Every symbol include/swin_wattn.h declares, with (argtypes, restype).
_vp, _i, _cp = ctypes.c_void_p, ctypes.c_int, ctypes.c_char_p
SIGNATURES = {
    "swin_wattn_plan": ([ctypes.POINTER(_vp), _i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp], _i),
    "swin_wattn_set_bias": ([_vp, _vp, _vp], _i),
    "swin_wattn_fwd": ([_vp, _vp, _vp, _vp], _i),
    "swin_wattn_fwd_host": ([_vp, _vp, _vp, _vp, _vp, _vp], _i),
    "swin_wattn_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp], _i),
    "swin_wattn_debug_maps": ([_vp, _vp, _vp, _vp, _vp, _vp], _i),
    "swin_wattn_bwd_noalloc": ([_vp, _vp, _vp, _vp, _vp] + [_i] * 8 + [_vp], _i),
    "swin_wattn_qkv_workspace_bytes": ([_i, _i], ctypes.c_size_t),
    "swin_wattn_qkv_proj": ([_vp] * 6 + [_i, _i, ctypes.c_float, _vp, ctypes.c_size_t, _vp, _vp], _i),
    "swin_wattn_qkv_prepared_bytes": ([_i], ctypes.c_size_t),
    "swin_wattn_qkv_stats_bytes": ([_i], ctypes.c_size_t),
    "swin_wattn_qkv_prepare": ([_vp] * 4 + [_i, _vp, ctypes.c_size_t, _vp], _i),
    "swin_wattn_qkv_proj_prepared": ([_vp] * 3 + [_i, _i, ctypes.c_float, _vp, ctypes.c_size_t, _vp, _vp], _i),
    "swin_wattn_qkv_proj_prepared_fp8": ([_vp] * 3 + [_i, _i] + [ctypes.c_float] * 4 +
                                         [_vp, _vp, ctypes.c_size_t, _vp, _vp], _i),
    "swin_wattn_proj_residual": ([_vp] * 5 + [_i, _i, _vp, _vp], _i),
    "swin_wattn_fwd_fp8": ([_vp, _vp, ctypes.c_float, ctypes.c_float, ctypes.c_float, _vp, _vp], _i),
    "swin_wattn_set_fwd_kernel": ([_vp, _i], _i),
    "swin_wattn_fwd_kernel": ([_vp], _i),
    "swin_wattn_set_bwd_kernel": ([_vp, _i], _i),
    "swin_wattn_bwd_kernel": ([_vp], _i),
    "swin_wattn_device_status": ([_vp, _vp], _i),
    "swin_wattn_destroy": ([_vp], _i),
    "swin_wattn_status_string": ([_i], _cp),
    "swin_wattn_last_error": ([], _cp),
    "swin_wattn_launch_count": ([_i], ctypes.c_uint64),
}

# The fault-injection library (include/swin_wattn_debug.h) adds one entry point.
DEBUG_LIB_PATH = os.path.join(_HERE, "libswin_wattn_debug.so")
DEBUG_SIGNATURES = {"swin_wattn_debug_set_fault": ([_i, ctypes.c_int64], _i)}
FAULT_NONE = 0
FAULT_FWD_MMA_SYNC = 1
FAULT_FWD_TCGEN05 = 2
FAULT_GEMM = 3

_lib = None
_debug_lib = None


class SwinWAttnError(RuntimeError):
    def __init__(self, where: str, status: int):
        lib = load()
        msg = lib.swin_wattn_status_string(status).decode()
        if status == ERR_CUDA:
            msg += ": " + lib.swin_wattn_last_error().decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def load() -> ctypes.CDLL:
    """Load the library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m swin_window_attention_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def load_debug() -> ctypes.CDLL:
    """Load the fault-injection build (once), a separate library with the same entry
    points plus swin_wattn_debug_set_fault. Raises if it has not been built
    (``python -m swin_window_attention_gb300.build --debug``)."""
    global _debug_lib
    if _debug_lib is None:
        if not os.path.exists(DEBUG_LIB_PATH):
            raise RuntimeError(f"{DEBUG_LIB_PATH} is missing: build it with "
                               "`python -m swin_window_attention_gb300.build --debug`")
        lib = ctypes.CDLL(DEBUG_LIB_PATH)
        for name, (args, res) in list(SIGNATURES.items()) + list(DEBUG_SIGNATURES.items()):
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _debug_lib = lib
    return _debug_lib


# ---- same names as the C entry points --------------------------------------------------

def swin_wattn_plan(B, H, W, C, num_heads, window, shift, dtype, bias_table_ptr, stream):
    """Returns (status, plan handle or None)."""
    h = _vp()
    rc = load().swin_wattn_plan(ctypes.byref(h), B, H, W, C, num_heads, window, shift, dtype,
                                bias_table_ptr, stream)
    return rc, (h.value if rc == OK else None)


def swin_wattn_set_bias(plan, bias_table_ptr, stream):
    return load().swin_wattn_set_bias(plan, bias_table_ptr, stream)


def swin_wattn_fwd(plan, qkv_ptr, out_ptr, stream):
    return load().swin_wattn_fwd(plan, qkv_ptr, out_ptr, stream)


def swin_wattn_fwd_host(plan, qkv_host_ptr, out_host_ptr, dev_qkv_ptr, dev_out_ptr, stream):
    return load().swin_wattn_fwd_host(plan, qkv_host_ptr, out_host_ptr, dev_qkv_ptr,
                                      dev_out_ptr, stream)


def swin_wattn_bwd(plan, qkv_ptr, dout_ptr, dqkv_ptr, dtable_ptr, stream):
    return load().swin_wattn_bwd(plan, qkv_ptr, dout_ptr, dqkv_ptr, dtable_ptr, stream)


def swin_wattn_debug_maps(plan, gather_ptr, relidx_ptr, mask_ptr, dense_bias_ptr, stream):
    return load().swin_wattn_debug_maps(plan, gather_ptr, relidx_ptr, mask_ptr, dense_bias_ptr,
                                        stream)


def swin_wattn_bwd_noalloc(qkv_ptr, dout_ptr, dqkv_ptr, dtable_ptr, table_ptr, B, H, W, C,
                           num_heads, window, shift, dtype, stream):
    """Backward with no plan and no device allocation (fixed working memory in the
    library); see include/swin_wattn.h."""
    return load().swin_wattn_bwd_noalloc(qkv_ptr, dout_ptr, dqkv_ptr, dtable_ptr, table_ptr, B, H,
                                         W, C, num_heads, window, shift, dtype, stream)


def swin_wattn_qkv_workspace_bytes(C, tokens):
    return int(load().swin_wattn_qkv_workspace_bytes(C, tokens))


def swin_wattn_qkv_proj(x_ptr, gamma_ptr, beta_ptr, w_ptr, b_ptr, qkv_ptr, tokens, C, eps, workspace_ptr,
                        workspace_bytes, status_ptr, stream):
    return load().swin_wattn_qkv_proj(x_ptr, gamma_ptr, beta_ptr, w_ptr, b_ptr, qkv_ptr, tokens, C, eps,
                                      workspace_ptr, workspace_bytes, status_ptr, stream)


def qkv_proj(x, gamma, beta, w, b, qkv=None, eps=1e-5, status=None, workspace=None, stream=None):
    """LayerNorm over the last axis of the bf16 CUDA tensor x [..., C], then x W^T + b into
    a bf16 [..., 3C] tensor (allocated here when not given; so is the workspace)."""
    import torch
    C = x.shape[-1]
    if qkv is None:
        qkv = torch.empty(x.shape[:-1] + (3 * C,), dtype=torch.bfloat16, device=x.device)
    tokens = x.numel() // C
    if workspace is None:
        workspace = torch.empty(max(swin_wattn_qkv_workspace_bytes(C, tokens), 1), dtype=torch.uint8,
                                device=x.device)
    rc = swin_wattn_qkv_proj(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), w.data_ptr(), b.data_ptr(),
                             qkv.data_ptr(), tokens, C, eps, workspace.data_ptr(), workspace.numel(),
                             None if status is None else status.data_ptr(), _stream_handle(stream))
    if rc != OK:
        raise SwinWAttnError("swin_wattn_qkv_proj", rc)
    return qkv


def swin_wattn_qkv_prepared_bytes(C):
    return int(load().swin_wattn_qkv_prepared_bytes(C))


def swin_wattn_qkv_stats_bytes(tokens):
    return int(load().swin_wattn_qkv_stats_bytes(tokens))


def swin_wattn_qkv_prepare(gamma_ptr, beta_ptr, w_ptr, b_ptr, C, prepared_ptr, prepared_bytes, stream):
    return load().swin_wattn_qkv_prepare(gamma_ptr, beta_ptr, w_ptr, b_ptr, C, prepared_ptr, prepared_bytes, stream)


def swin_wattn_qkv_proj_prepared(x_ptr, prepared_ptr, qkv_ptr, tokens, C, eps, stats_ptr, stats_bytes, status_ptr,
                                 stream):
    return load().swin_wattn_qkv_proj_prepared(x_ptr, prepared_ptr, qkv_ptr, tokens, C, eps, stats_ptr,
                                               stats_bytes, status_ptr, stream)


class QkvProjection:
    """The producer step with its weights prepared once: LayerNorm over the last axis of a
    bf16 CUDA tensor x [..., C], then x W^T + b, for fixed gamma, beta, W [3C, C], b [3C]."""

    def __init__(self, gamma, beta, w, b, stream=None):
        import torch
        self.C = int(w.shape[1])
        self.prepared = torch.empty(max(swin_wattn_qkv_prepared_bytes(self.C), 1), dtype=torch.uint8,
                                    device=w.device)
        rc = swin_wattn_qkv_prepare(gamma.data_ptr(), beta.data_ptr(), w.data_ptr(), b.data_ptr(), self.C,
                                    self.prepared.data_ptr(), self.prepared.numel(), _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_qkv_prepare", rc)
        self.stats = None

    def __call__(self, x, qkv=None, eps=1e-5, status=None, stream=None):
        import torch
        C = self.C
        tokens = x.numel() // C
        if qkv is None:
            qkv = torch.empty(x.shape[:-1] + (3 * C,), dtype=torch.bfloat16, device=x.device)
        need = max(swin_wattn_qkv_stats_bytes(tokens), 16)
        if self.stats is None or self.stats.numel() < need:
            self.stats = torch.empty(need, dtype=torch.uint8, device=x.device)
        rc = swin_wattn_qkv_proj_prepared(x.data_ptr(), self.prepared.data_ptr(), qkv.data_ptr(), tokens, C, eps,
                                          self.stats.data_ptr(), self.stats.numel(),
                                          None if status is None else status.data_ptr(), _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_qkv_proj_prepared", rc)
        return qkv

    def fp8(self, x, scales, qkv8=None, amax=None, eps=1e-5, status=None, stream=None):
        """The same projection with OCP FP8 E4M3 output, qkv8 = E4M3(qkv / scale_t) for the
        tensor t (q, k, v) of each channel, as a uint8 [..., 3C] tensor (allocated here when
        not given); amax, an optional CUDA float tensor [3], receives max |qkv_t| (max-ed)."""
        import torch
        C = self.C
        tokens = x.numel() // C
        if qkv8 is None:
            qkv8 = torch.empty(x.shape[:-1] + (3 * C,), dtype=torch.uint8, device=x.device)
        need = max(swin_wattn_qkv_stats_bytes(tokens), 16)
        if self.stats is None or self.stats.numel() < need:
            self.stats = torch.empty(need, dtype=torch.uint8, device=x.device)
        sq, sk, sv = (float(v) for v in scales)
        rc = swin_wattn_qkv_proj_prepared_fp8(x.data_ptr(), self.prepared.data_ptr(), qkv8.data_ptr(), tokens, C,
                                              eps, sq, sk, sv, None if amax is None else amax.data_ptr(),
                                              self.stats.data_ptr(), self.stats.numel(),
                                              None if status is None else status.data_ptr(), _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_qkv_proj_prepared_fp8", rc)
        return qkv8


def swin_wattn_qkv_proj_prepared_fp8(x_ptr, prepared_ptr, qkv8_ptr, tokens, C, eps, scale_q, scale_k, scale_v,
                                     amax_ptr, stats_ptr, stats_bytes, status_ptr, stream):
    return load().swin_wattn_qkv_proj_prepared_fp8(x_ptr, prepared_ptr, qkv8_ptr, tokens, C, eps, scale_q, scale_k,
                                                   scale_v, amax_ptr, stats_ptr, stats_bytes, status_ptr, stream)


def swin_wattn_proj_residual(o_ptr, wp_ptr, bp_ptr, residual_ptr, y_ptr, tokens, C, status_ptr, stream):
    return load().swin_wattn_proj_residual(o_ptr, wp_ptr, bp_ptr, residual_ptr, y_ptr, tokens, C, status_ptr,
                                           stream)


def proj_residual(o, wp, bp, residual, y=None, status=None, stream=None):
    """residual + o Wp^T + bp over the last axis of the bf16 CUDA tensors o and residual
    [..., C] into a bf16 [..., C] tensor (allocated here when not given; it may be the
    residual itself)."""
    import torch
    C = o.shape[-1]
    if y is None:
        y = torch.empty(o.shape, dtype=torch.bfloat16, device=o.device)
    rc = swin_wattn_proj_residual(o.data_ptr(), wp.data_ptr(), bp.data_ptr(), residual.data_ptr(), y.data_ptr(),
                                  o.numel() // C, C, None if status is None else status.data_ptr(),
                                  _stream_handle(stream))
    if rc != OK:
        raise SwinWAttnError("swin_wattn_proj_residual", rc)
    return y


def swin_wattn_fwd_fp8(plan, qkv8_ptr, scale_q, scale_k, scale_v, out_ptr, stream):
    return load().swin_wattn_fwd_fp8(plan, qkv8_ptr, scale_q, scale_k, scale_v, out_ptr, stream)


def swin_wattn_set_fwd_kernel(plan, kernel):
    return load().swin_wattn_set_fwd_kernel(plan, kernel)


def swin_wattn_fwd_kernel(plan):
    return load().swin_wattn_fwd_kernel(plan)


def swin_wattn_set_bwd_kernel(plan, kernel):
    return load().swin_wattn_set_bwd_kernel(plan, kernel)


def swin_wattn_bwd_kernel(plan):
    return load().swin_wattn_bwd_kernel(plan)


def swin_wattn_device_status(plan, stream):
    return load().swin_wattn_device_status(plan, stream)


def swin_wattn_destroy(plan):
    return load().swin_wattn_destroy(plan)


def swin_wattn_status_string(status):
    return load().swin_wattn_status_string(status).decode()


def swin_wattn_last_error():
    return load().swin_wattn_last_error().decode()


def swin_wattn_launch_count(reset=False):
    return int(load().swin_wattn_launch_count(1 if reset else 0))


# ---- torch convenience wrapper ---------------------------------------------------------

def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class WindowAttention:
    """A plan for one layer shape, driven with torch CUDA tensors.

    ``table`` is the fp32 [(2M-1)^2, nH] bias table on the GPU. Activations are bf16 or
    fp32 [B,H,W,3C] tensors (contiguous); outputs are allocated by the caller or here.
    """

    def __init__(self, B, H, W, C, num_heads, window, shift, table, dtype="bf16", stream=None):
        import torch
        self.B, self.H, self.W, self.C = B, H, W, C
        self.nH, self.M, self.s = num_heads, window, shift
        self.dtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        code = BF16 if dtype == "bf16" else FP32
        rc, h = swin_wattn_plan(B, H, W, C, num_heads, window, shift, code, table.data_ptr(),
                                _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_plan", rc)
        self.handle = h

    def set_fwd_kernel(self, kernel):
        """KERNEL_AUTO, KERNEL_MMA_SYNC or KERNEL_TCGEN05 for later forwards."""
        rc = swin_wattn_set_fwd_kernel(self.handle, kernel)
        if rc != OK:
            raise SwinWAttnError("swin_wattn_set_fwd_kernel", rc)

    @property
    def fwd_kernel(self):
        return swin_wattn_fwd_kernel(self.handle)

    def set_bwd_kernel(self, kernel):
        """KERNEL_AUTO, KERNEL_MMA_SYNC or KERNEL_TCGEN05 for later backwards."""
        rc = swin_wattn_set_bwd_kernel(self.handle, kernel)
        if rc != OK:
            raise SwinWAttnError("swin_wattn_set_bwd_kernel", rc)

    @property
    def bwd_kernel(self):
        return swin_wattn_bwd_kernel(self.handle)

    def device_status(self, stream=None):
        """Synchronise and raise if a bounded device wait ran out since the last check."""
        rc = swin_wattn_device_status(self.handle, _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_device_status", rc)

    def set_bias(self, table, stream=None):
        rc = swin_wattn_set_bias(self.handle, table.data_ptr(), _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_set_bias", rc)

    def fwd(self, qkv, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty(self.B, self.H, self.W, self.C, dtype=self.dtype, device=qkv.device)
        rc = swin_wattn_fwd(self.handle, qkv.data_ptr(), out.data_ptr(), _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_fwd", rc)
        return out

    def fwd_fp8(self, qkv8, scales, out=None, stream=None):
        """Forward on 8-bit operands: qkv8 a [B,H,W,3C] CUDA tensor of OCP FP8 E4M3 bytes
        (torch.float8_e4m3fn or uint8), scales (scale_q, scale_k, scale_v); bf16 output."""
        import torch
        if out is None:
            out = torch.empty(self.B, self.H, self.W, self.C, dtype=torch.bfloat16, device=qkv8.device)
        sq, sk, sv = (float(x) for x in scales)
        rc = swin_wattn_fwd_fp8(self.handle, qkv8.data_ptr(), sq, sk, sv, out.data_ptr(), _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_fwd_fp8", rc)
        return out

    def fwd_host(self, qkv_host, out_host, dev_qkv, dev_out, stream=None):
        """Host-resident qkv -> host-resident out through the library's host entry point
        (copies and kernel in order on the stream; synchronise before reading out_host)."""
        rc = swin_wattn_fwd_host(self.handle, qkv_host.data_ptr(), out_host.data_ptr(),
                                 dev_qkv.data_ptr(), dev_out.data_ptr(), _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_fwd_host", rc)
        return out_host

    def bwd(self, qkv, dout, dqkv=None, dtable=None, stream=None):
        import torch
        if dqkv is None:
            dqkv = torch.empty_like(qkv)
        if dtable is None:
            dtable = torch.empty((2 * self.M - 1) ** 2, self.nH, dtype=torch.float32,
                                 device=qkv.device)
        rc = swin_wattn_bwd(self.handle, qkv.data_ptr(), dout.data_ptr(), dqkv.data_ptr(),
                            dtable.data_ptr(), _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_bwd", rc)
        return dqkv, dtable

    def debug_maps(self, stream=None):
        import torch
        dev = torch.device("cuda")
        N, nW = self.M * self.M, (self.H // self.M) * (self.W // self.M)
        gather = torch.empty(nW, N, dtype=torch.int32, device=dev)
        relidx = torch.empty(N, N, dtype=torch.int32, device=dev)
        mask = torch.empty(nW, N, N, dtype=torch.float32, device=dev)
        dense = torch.empty(self.nH, N, N, dtype=torch.float32, device=dev)
        rc = swin_wattn_debug_maps(self.handle, gather.data_ptr(), relidx.data_ptr(),
                                   mask.data_ptr(), dense.data_ptr(), _stream_handle(stream))
        if rc != OK:
            raise SwinWAttnError("swin_wattn_debug_maps", rc)
        return gather, relidx, mask, dense

    def close(self):
        if getattr(self, "handle", None):
            swin_wattn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

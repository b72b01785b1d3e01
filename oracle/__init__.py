"""fp64 CPU oracle for Swin (shifted-)window attention: TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package. The library in ``swin_window_attention_gb300`` never does, and
the two share no code. The arithmetic lives in ``swin_oracle.cpp``; this module only
compiles it with the host compiler and marshals numpy arrays.

Every function takes and returns float64 numpy arrays (int32 for index maps). Inputs are
expected to hold the bf16-rounded values the GPU path sees, widened to float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swin_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle_swin.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int32)
_i = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (OpenMP) if the shared object is missing or stale."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared",
                   "-fno-fast-math", _SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str) -> ctypes.CDLL:
    """Load a compiled oracle and declare its C signatures."""
    lib = ctypes.CDLL(path)
    sig = {
        "oracle_max_threads": ([], _i),
        "oracle_set_threads": ([_i], None),
        "oracle_roll": ([_D, _i, _i, _i, _i, _i, _D], None),
        "oracle_unroll": ([_D, _i, _i, _i, _i, _i, _D], None),
        "oracle_partition": ([_D, _i, _i, _i, _i, _i, _D], None),
        "oracle_reverse": ([_D, _i, _i, _i, _i, _i, _D], None),
        "oracle_relidx": ([_i, _I], None),
        "oracle_dense_bias": ([_D, _i, _i, _D], None),
        "oracle_mask": ([_i, _i, _i, _i, _D], None),
        "oracle_gather": ([_i, _i, _i, _i, _I], None),
        "oracle_probs": ([_D, _D] + [_i] * 10 + [_D], None),
        "oracle_fwd": ([_D, _D] + [_i] * 7 + [_D], None),
        "oracle_bwd": ([_D, _D, _D] + [_i] * 7 + [_D, _D], None),
        "oracle_qkv_proj": ([_D, _D, _D, _D, _D, _i, _i, ctypes.c_double, _D], None),
        "oracle_proj_residual": ([_D, _D, _D, _D, _i, _i, _D], None),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = bind(_LIB_PATH)
    return _lib


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _dp(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _ip(a: np.ndarray):
    return a.ctypes.data_as(_I)


def max_threads() -> int:
    return _load().oracle_max_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def roll(x, s: int) -> np.ndarray:
    """[B,H,W,Ch] -> rolled grid that reads (y+s, x+s) mod (H, W)."""
    x = _f64(x)
    B, H, W, Ch = x.shape
    out = np.empty_like(x)
    _load().oracle_roll(_dp(x), B, H, W, Ch, s, _dp(out))
    return out


def unroll(x, s: int) -> np.ndarray:
    x = _f64(x)
    B, H, W, Ch = x.shape
    out = np.empty_like(x)
    _load().oracle_unroll(_dp(x), B, H, W, Ch, s, _dp(out))
    return out


def partition(x, M: int) -> np.ndarray:
    """[B,H,W,Ch] -> [B, nW, M*M, Ch]."""
    x = _f64(x)
    B, H, W, Ch = x.shape
    out = np.empty((B, (H // M) * (W // M), M * M, Ch), dtype=np.float64)
    _load().oracle_partition(_dp(x), B, H, W, Ch, M, _dp(out))
    return out


def reverse(xw, H: int, W: int, M: int) -> np.ndarray:
    """[B, nW, M*M, Ch] -> [B,H,W,Ch]."""
    xw = _f64(xw)
    B, _, _, Ch = xw.shape
    out = np.empty((B, H, W, Ch), dtype=np.float64)
    _load().oracle_reverse(_dp(xw), B, H, W, Ch, M, _dp(out))
    return out


def relidx(M: int) -> np.ndarray:
    out = np.empty((M * M, M * M), dtype=np.int32)
    _load().oracle_relidx(M, _ip(out))
    return out


def dense_bias(table, nH: int, M: int) -> np.ndarray:
    table = _f64(table)
    assert table.shape == ((2 * M - 1) ** 2, nH)
    out = np.empty((nH, M * M, M * M), dtype=np.float64)
    _load().oracle_dense_bias(_dp(table), nH, M, _dp(out))
    return out


def mask(H: int, W: int, M: int, s: int) -> np.ndarray:
    out = np.empty(((H // M) * (W // M), M * M, M * M), dtype=np.float64)
    _load().oracle_mask(H, W, M, s, _dp(out))
    return out


def gather(H: int, W: int, M: int, s: int) -> np.ndarray:
    out = np.empty(((H // M) * (W // M), M * M), dtype=np.int32)
    _load().oracle_gather(H, W, M, s, _ip(out))
    return out


def probs(qkv, table, nH: int, M: int, s: int, b: int, w: int, h: int) -> np.ndarray:
    qkv, table = _f64(qkv), _f64(table)
    B, H, W, C3 = qkv.shape
    out = np.empty((M * M, M * M), dtype=np.float64)
    _load().oracle_probs(_dp(qkv), _dp(table), B, H, W, C3 // 3, nH, M, s, b, w, h, _dp(out))
    return out


def fwd(qkv, table, nH: int, M: int, s: int) -> np.ndarray:
    """qkv [B,H,W,3C], table [(2M-1)^2, nH] -> Y [B,H,W,C] (all float64)."""
    qkv, table = _f64(qkv), _f64(table)
    B, H, W, C3 = qkv.shape
    C = C3 // 3
    _check(B, H, W, C, nH, M, s, table)
    Y = np.empty((B, H, W, C), dtype=np.float64)
    _load().oracle_fwd(_dp(qkv), _dp(table), B, H, W, C, nH, M, s, _dp(Y))
    return Y


def bwd(qkv, dY, table, nH: int, M: int, s: int):
    """Returns (dqkv [B,H,W,3C], dtable [(2M-1)^2, nH]) for upstream gradient dY."""
    qkv, dY, table = _f64(qkv), _f64(dY), _f64(table)
    B, H, W, C3 = qkv.shape
    C = C3 // 3
    _check(B, H, W, C, nH, M, s, table)
    assert dY.shape == (B, H, W, C)
    dqkv = np.empty_like(qkv)
    dtab = np.empty_like(table)
    _load().oracle_bwd(_dp(qkv), _dp(dY), _dp(table), B, H, W, C, nH, M, s, _dp(dqkv), _dp(dtab))
    return dqkv, dtab


def qkv_proj(x, gamma, beta, w, b, eps: float = 1e-5) -> np.ndarray:
    """LayerNorm over the last axis of x [..., C] then x W^T + b with W [3C, C], b [3C]
    -> [..., 3C] (float64)."""
    x, gamma, beta, w, b = _f64(x), _f64(gamma), _f64(beta), _f64(w), _f64(b)
    C = x.shape[-1]
    if w.shape != (3 * C, C) or b.shape != (3 * C,) or gamma.shape != (C,) or beta.shape != (C,):
        raise ValueError("oracle: qkv_proj shapes")
    T = int(np.prod(x.shape[:-1]))
    out = np.empty(x.shape[:-1] + (3 * C,), dtype=np.float64)
    _load().oracle_qkv_proj(_dp(x), _dp(gamma), _dp(beta), _dp(w), _dp(b), T, C, float(eps), _dp(out))
    return out


def proj_residual(o, wp, bp, residual) -> np.ndarray:
    """residual + o Wp^T + bp over the last axis: o and residual [..., C], Wp [C, C],
    bp [C] -> [..., C] (float64)."""
    o, wp, bp, residual = _f64(o), _f64(wp), _f64(bp), _f64(residual)
    C = o.shape[-1]
    if wp.shape != (C, C) or bp.shape != (C,) or residual.shape != o.shape:
        raise ValueError("oracle: proj_residual shapes")
    T = int(np.prod(o.shape[:-1]))
    out = np.empty(o.shape, dtype=np.float64)
    _load().oracle_proj_residual(_dp(o), _dp(wp), _dp(bp), _dp(residual), T, C, _dp(out))
    return out


def _check(B, H, W, C, nH, M, s, table):
    if H % M or W % M or C % nH or not (0 <= s < M):
        raise ValueError(f"oracle: unsupported shape H={H} W={W} C={C} nH={nH} M={M} s={s}")
    if table.shape != ((2 * M - 1) ** 2, nH):
        raise ValueError(f"oracle: table shape {table.shape}")

"""Helpers for the GPU parity tests: run the library through its C ABI on seeded inputs
and compare with the fp64 oracle on the same bf16-rounded values."""
import json
import os

import numpy as np
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs

# Tolerances for floating-point outputs (bf16 inputs, fp32 accumulation): per tensor,
# max |gpu - oracle| <= 1e-2 and ||gpu - oracle||_2 / ||oracle||_2 <= 5e-3.
#
# A bf16 output cannot be nearer the exact value than its own rounding, and half a bf16
# ulp exceeds 1e-2 for |x| >= 4 (the exact Swin-B 56x56 dq value 4.55 rounds to bf16
# with an error of 0.0114). An element of a bf16 output therefore passes if it lies
# within 1e-2 of the oracle, or, where half a bf16 ulp at the oracle value exceeds 1e-2,
# if it is one of the two bf16 values around the exact one (faithful rounding:
# |gpu - oracle| < one ulp).
TOL_ABS = 1e-2
TOL_REL = 5e-3


def bf16_ulp(ref):
    """The bf16 unit in the last place at |ref| (2^(e - 7) for |ref| in [2^e, 2^(e+1)))."""
    a = np.maximum(np.abs(ref), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7.0)


def allowed_error(ref, bf16_output):
    """Per-element bound: 1e-2, or just under one bf16 ulp where half an ulp exceeds it."""
    if not bf16_output:
        return np.full(np.shape(ref), TOL_ABS)
    u = bf16_ulp(ref)
    return np.where(0.5 * u > TOL_ABS, u * (1.0 - 1e-9), TOL_ABS)


def _is_bf16(got):
    return isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16


def errors(got, ref):
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all()
    d = g - ref
    return float(np.abs(d).max()) if d.size else 0.0, float(
        np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))


def bound_excess(got, ref):
    """max over elements of |gpu - oracle| - allowed_error (<= 0 passes)."""
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if not ref.size:
        return -np.inf
    return float((np.abs(g - ref) - allowed_error(ref, _is_bf16(got))).max())


def log_case(name, ma, rl):
    """Append the measured margins of one comparison to $SWIN_PARITY_LOG (if set)."""
    log = os.environ.get("SWIN_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                "tensor": name, "max_abs": ma, "rel_l2": rl}) + "\n")


def assert_close(name, got, ref):
    ma, rl = errors(got, ref)
    ex = bound_excess(got, ref)
    log_case(name, ma, rl)
    assert ex <= 0.0 and rl <= TOL_REL, f"{name}: max-abs {ma:.3g} (bound exceeded by {ex:.3g}), rel-L2 {rl:.3g}"
    return ma, rl


class Accum:
    """Max-abs and rel-L2 of a large tensor compared piece by piece (every element).
    With rounded=True the per-element bound is 1e-2 + 2^-8 |ref| (assert_close_rounded)."""

    def __init__(self, rounded=False):
        self.max_abs, self.d2, self.r2, self.n = 0.0, 0.0, 0.0, 0
        self.rounded, self.excess, self.excess_r = rounded, -np.inf, -np.inf

    def add(self, got, ref):
        g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
        ref = np.asarray(ref, np.float64)
        assert g.shape == ref.shape, (g.shape, ref.shape)
        assert np.isfinite(g).all()
        d = g - ref
        if d.size:
            self.max_abs = max(self.max_abs, float(np.abs(d).max()))
            self.excess = max(self.excess, float((np.abs(d) - allowed_error(ref, _is_bf16(got))).max()))
            self.excess_r = max(self.excess_r, float((np.abs(d) - (TOL_ABS + 2.0 ** -8 * np.abs(ref))).max()))
        self.d2 += float(np.square(d).sum())
        self.r2 += float(np.square(ref).sum())
        self.n += d.size

    def check(self, name):
        rl = float(np.sqrt(self.d2) / max(np.sqrt(self.r2), 1e-30))
        log_case(name, self.max_abs, rl)
        ex = self.excess_r if self.rounded else self.excess
        assert ex <= 0.0 and rl <= TOL_REL, \
            f"{name}: max-abs {self.max_abs:.3g} (bound exceeded by {ex:.3g}), rel-L2 {rl:.3g} over {self.n} elements"
        return self.max_abs, rl


def batch_chunks(B, images=8):
    """Consecutive image ranges of at most `images` images covering the batch."""
    return [list(range(lo, min(B, lo + images))) for lo in range(0, B, images)]


def assert_fwd_every_image(name, y_cpu, qkv, table, wl, images=8):
    """Y of every image of the batch against the oracle, a few images at a time."""
    acc = Accum()
    for bs in batch_chunks(wl.B, images):
        acc.add(y_cpu[bs], oracle_fwd(qkv, table, wl, batches=bs))
    return acc.check(name)


# The GEMM steps' outputs (qkv, and y = residual + projection) are stored in bf16 with
# values of a few units: a bf16 value carries an error up to half an ulp = 2^-9 |y| from
# its own rounding, and the bf16 operands add about as much again. So each element must lie
# within 1e-2 + 2^-8 |ref| (the 1e-2 absolute bound plus one bf16 ulp of the value), and
# the tensor within rel-L2 5e-3.
def assert_close_rounded(name, got, ref):
    ma, rl = errors(got, ref)
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    excess = float((np.abs(g - ref) - (TOL_ABS + 2.0 ** -8 * np.abs(ref))).max())
    log_case(name, ma, rl)
    assert excess <= 0.0 and rl <= TOL_REL, f"{name}: max-abs {ma:.3g} (bound exceeded by {excess:.3g}), rel-L2 {rl:.3g}"


def workload(B, H, W, C, nH, M, s, dtype="bf16", seed=7):
    return inputs.Workload("case", 9, seed, B, H, W, C, nH, M, s, dtype)


def plan(wl, table_dev):
    return capi.WindowAttention(wl.B, wl.H, wl.W, wl.C, wl.nH, wl.M, wl.s, table_dev,
                                dtype=wl.dtype)


def oracle_fwd(qkv, table, wl, batches=None):
    q = inputs.act_f64(qkv if batches is None else qkv[batches])
    return oracle.fwd(q, table.double().numpy(), wl.nH, wl.M, wl.s)


def oracle_bwd(qkv, dout, table, wl, batches=None):
    q = inputs.act_f64(qkv if batches is None else qkv[batches])
    d = inputs.act_f64(dout if batches is None else dout[batches])
    return oracle.bwd(q, d, table.double().numpy(), wl.nH, wl.M, wl.s)

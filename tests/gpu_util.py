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
TOL_ABS = 1e-2
TOL_REL = 5e-3


def errors(got, ref):
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all()
    d = g - ref
    return float(np.abs(d).max()) if d.size else 0.0, float(
        np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))


def log_case(name, ma, rl):
    """Append the measured margins of one comparison to $SWIN_PARITY_LOG (if set)."""
    log = os.environ.get("SWIN_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
                                "tensor": name, "max_abs": ma, "rel_l2": rl}) + "\n")


def assert_close(name, got, ref):
    ma, rl = errors(got, ref)
    log_case(name, ma, rl)
    assert ma <= TOL_ABS and rl <= TOL_REL, f"{name}: max-abs {ma:.3g}, rel-L2 {rl:.3g}"
    return ma, rl


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

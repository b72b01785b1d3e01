"""Pins of the oracle's consumer step (the output projection, then the bias and the
residual added), on the CPU: against torch's linear in float64 (the library special case
of the definition), closed forms for identity, permutation, zero and rank-one weights,
linearity, and planted mistakes each caught by a pin."""
import os
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "swin_oracle.cpp")


def _torch_ref(o, wp, bp, r):
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    return (t(r) + F.linear(t(o), t(wp), t(bp))).numpy()


def _case(rng, shape, C):
    o = rng.standard_normal(shape + (C,)) * 0.8
    wp = rng.standard_normal((C, C)) * 0.05
    bp = rng.standard_normal(C) * 0.1
    r = rng.standard_normal(shape + (C,)) * 1.5 + 0.2
    return o, wp, bp, r


@pytest.mark.parametrize("shape,C", [((3, 5), 32), ((2, 7, 7), 96), ((11,), 192), ((1, 4, 4), 40)])
def test_matches_torch_linear_plus_residual(shape, C):
    o, wp, bp, r = _case(np.random.default_rng(C), shape, C)
    y = oracle.proj_residual(o, wp, bp, r)
    assert y.shape == shape + (C,)
    assert np.abs(y - _torch_ref(o, wp, bp, r)).max() < 1e-12


def test_closed_forms_identity_zero_and_permutation():
    rng = np.random.default_rng(1)
    C = 24
    o, _, bp, r = _case(rng, (5,), C)
    assert np.abs(oracle.proj_residual(o, np.eye(C), np.zeros(C), r) - (r + o)).max() < 1e-15
    assert np.abs(oracle.proj_residual(o, np.zeros((C, C)), bp, r) - (r + bp[None, :])).max() < 1e-15
    perm = rng.permutation(C)
    P = np.eye(C)[perm]  # row n selects input channel perm[n]
    assert np.abs(oracle.proj_residual(o, P, bp, r) - (r + o[:, perm] + bp)).max() < 1e-15


def test_rank_one_weight():
    """Wp = a c^T: output channel n gets a_n (o . c)."""
    rng = np.random.default_rng(2)
    C = 40
    o, _, bp, r = _case(rng, (6,), C)
    a, c = rng.standard_normal(C), rng.standard_normal(C)
    y = oracle.proj_residual(o, np.outer(a, c), bp, r)
    assert np.abs(y - (r + (o @ c)[:, None] * a[None, :] + bp)).max() < 1e-12


def test_linear_in_the_attention_output():
    rng = np.random.default_rng(3)
    o1, wp, bp, r = _case(rng, (4, 3), 32)
    o2 = rng.standard_normal(o1.shape)
    z = np.zeros_like(r)
    lhs = oracle.proj_residual(o1 + o2, wp, bp, r)
    rhs = oracle.proj_residual(o1, wp, bp, r) + oracle.proj_residual(o2, wp, np.zeros(32), z)
    assert np.abs(lhs - rhs).max() < 1e-12


MUTANTS = {
    "weight_transposed": ("const double* wr = wp + (int64_t)n * C;\n      double acc = 0.0;\n      for (int c = 0; c < C; ++c) acc += orow[c] * wr[c];",
                          "double acc = 0.0;\n      for (int c = 0; c < C; ++c) acc += orow[c] * wp[(int64_t)c * C + n];"),
    "bias_dropped": ("residual[t * C + n] + (acc + bp[n]);", "residual[t * C + n] + acc;"),
    "residual_dropped": ("residual[t * C + n] + (acc + bp[n]);", "acc + bp[n];"),
    "residual_other_token": ("residual[t * C + n] + (acc + bp[n]);", "residual[((t + 1) % T) * C + n] + (acc + bp[n]);"),
    "channel_shifted": ("for (int c = 0; c < C; ++c) acc += orow[c] * wr[c];",
                        "for (int c = 0; c < C; ++c) acc += orow[(c + 1) % C] * wr[c];"),
}


def _pins_pass(lib):
    rng = np.random.default_rng(7)
    for shape, C in (((3, 5), 32), ((1, 4, 4), 40)):
        f = lambda a: np.ascontiguousarray(a, dtype=np.float64)
        o, wp, bp, r = map(f, _case(rng, shape, C))
        T = int(np.prod(shape))
        out = np.empty(shape + (C,))
        lib.oracle_proj_residual(oracle._dp(o), oracle._dp(wp), oracle._dp(bp), oracle._dp(r), T, C,
                                 oracle._dp(out))
        if np.abs(out - _torch_ref(o, wp, bp, r)).max() > 1e-12:
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    msrc = tmp_path / "m.cpp"
    msrc.write_text(src.replace(old, new))
    so = tmp_path / "m.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fopenmp", "-fPIC", "-shared", str(msrc), "-o", str(so)], check=True)
    assert not _pins_pass(oracle.bind(str(so)))


def test_unmutated_oracle_passes_the_same_pins():
    oracle.build()
    assert _pins_pass(oracle._load())

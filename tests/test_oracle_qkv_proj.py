"""Pins of the oracle's producer step (LayerNorm over C, then the qkv projection), on the
CPU: against torch's layer_norm and linear in float64 (the library special case of the
definition), closed forms, invariances, and planted mistakes each caught by a pin."""
import os
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "swin_oracle.cpp")


def _torch_ref(x, g, be, w, b, eps):
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    C = x.shape[-1]
    return F.linear(F.layer_norm(t(x), (C,), t(g), t(be), eps), t(w), t(b)).numpy()


def _case(rng, shape, C):
    x = rng.standard_normal(shape + (C,)) * 1.7 + 0.3
    g = rng.standard_normal(C)
    be = rng.standard_normal(C)
    w = rng.standard_normal((3 * C, C)) * 0.05
    b = rng.standard_normal(3 * C)
    return x, g, be, w, b


@pytest.mark.parametrize("shape,C,eps", [((3, 5), 32, 1e-5), ((2, 7, 7), 96, 1e-5), ((11,), 192, 1e-3),
                                         ((1, 4, 4), 64, 0.0)])
def test_matches_torch_layer_norm_and_linear(shape, C, eps):
    x, g, be, w, b = _case(np.random.default_rng(C), shape, C)
    y = oracle.qkv_proj(x, g, be, w, b, eps)
    assert y.shape == shape + (3 * C,)
    assert np.abs(y - _torch_ref(x, g, be, w, b, eps)).max() < 1e-11


def test_closed_form_identity_projection():
    """gamma = 1, beta = 0, b = 0, W = [I; 2I; 3I], eps = 0: the first C outputs of a token
    have mean 0 and population variance 1, and the other two blocks are 2x and 3x them."""
    rng = np.random.default_rng(1)
    C = 48
    x = rng.standard_normal((6, C)) * 3.0 + 5.0
    eye = np.eye(C)
    y = oracle.qkv_proj(x, np.ones(C), np.zeros(C), np.vstack([eye, 2 * eye, 3 * eye]), np.zeros(3 * C), 0.0)
    q = y[:, :C]
    assert np.abs(q.mean(axis=1)).max() < 1e-12
    assert np.abs(q.var(axis=1) - 1.0).max() < 1e-12
    assert np.abs(y[:, C:2 * C] - 2 * q).max() < 1e-12 and np.abs(y[:, 2 * C:] - 3 * q).max() < 1e-12


def test_shift_and_scale_invariance():
    """LN(x + c) = LN(x) for a per-token constant c; with eps = 0 also LN(a x) = LN(x), a > 0."""
    rng = np.random.default_rng(2)
    x, g, be, w, b = _case(rng, (9,), 64)
    c = rng.standard_normal((9, 1)) * 10
    y0 = oracle.qkv_proj(x, g, be, w, b, 1e-5)
    assert np.abs(oracle.qkv_proj(x + c, g, be, w, b, 1e-5) - y0).max() < 1e-9
    y1 = oracle.qkv_proj(x, g, be, w, b, 0.0)
    assert np.abs(oracle.qkv_proj(x * 7.5, g, be, w, b, 0.0) - y1).max() < 1e-10


def test_bias_and_beta_enter_linearly():
    """With gamma = 0 the output is beta W^T + b for every token."""
    rng = np.random.default_rng(3)
    x, g, be, w, b = _case(rng, (4,), 32)
    y = oracle.qkv_proj(x, np.zeros(32), be, w, b)
    assert np.abs(y - (be @ w.T + b)[None, :]).max() < 1e-12


MUTANTS = {
    "variance_unbiased": ("    var /= C;\n    const double rstd", "    var /= (C - 1);\n    const double rstd"),
    "eps_outside_sqrt": ("1.0 / std::sqrt(var + eps)", "1.0 / (std::sqrt(var) + eps)"),
    "beta_dropped": ("* rstd * gamma[c] + beta[c];", "* rstd * gamma[c];"),
    "weight_transposed": ("const double* wr = w + (int64_t)n * C;\n      double acc = b[n];\n      for (int c = 0; c < C; ++c) acc += xn[c] * wr[c];",
                          "double acc = b[n];\n      for (int c = 0; c < C; ++c) acc += xn[c] * w[(int64_t)c * N + n % C];"),
    "bias_dropped": ("double acc = b[n];", "double acc = 0.0;"),
}


def _pins_pass(lib):
    rng = np.random.default_rng(7)
    for shape, C, eps in (((3, 5), 32, 1e-5), ((1, 4, 4), 64, 0.0)):
        x, g, be, w, b = _case(rng, shape, C)
        T = int(np.prod(shape))
        out = np.empty(shape + (3 * C,))
        f = lambda a: np.ascontiguousarray(a, dtype=np.float64)
        x, g, be, w, b = map(f, (x, g, be, w, b))
        lib.oracle_qkv_proj(oracle._dp(x), oracle._dp(g), oracle._dp(be), oracle._dp(w), oracle._dp(b), T, C,
                            float(eps), oracle._dp(out))
        if np.abs(out - _torch_ref(x, g, be, w, b, eps)).max() > 1e-11:
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

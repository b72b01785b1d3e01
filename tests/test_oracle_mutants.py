"""The oracle's pins must catch plausible mistakes. Each case here compiles a copy of
the oracle source with one planted error (on the CPU, in a temporary directory) and
checks that at least one pin from ``test_oracle_pins`` rejects it: a flipped roll
direction, a transposed relative index, a positive mask, a dropped bias, a dropped
softmax shift, a missing scale, and in the backward a dropped D term, a missing dK
scale and dV taken from P instead of its transpose."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_pins import brute_force_fwd, torch_swin_attention

SRC = os.path.join(os.path.dirname(oracle.__file__), "swin_oracle.cpp")

MUTANTS = {
    "roll_direction": ("pos_mod(y + s, H), xs = pos_mod(x + s, W)",
                       "pos_mod(y - s, H), xs = pos_mod(x - s, W)"),
    "relidx_transposed": ("(yi - yj + M - 1) * (2 * M - 1) + (xi - xj + M - 1)",
                          "(yj - yi + M - 1) * (2 * M - 1) + (xi - xj + M - 1)"),
    "mask_sign": ("? 0.0 : -100.0", "? 0.0 : 100.0"),
    "bias_dropped": ("double v = scale * dot + dense_bias_h[(int64_t)i * N + j];",
                     "double v = scale * dot;"),
    "scale_missing": ("double v = scale * dot +", "double v = dot +"),
    "region_bound": ("if (c < L - s) return 1;", "if (c <= L - s) return 1;"),
    "bwd_D_dropped": ("* (dP[(int64_t)i * N + j] - D);", "* (dP[(int64_t)i * N + j]);"),
    "bwd_dK_scale": ("dk[d] += g * q[d];", "dk[d] += dS[(int64_t)i * N + j] * q[d];"),
    "bwd_dV_transposed": ("const double p = P[(int64_t)i * N + j];\n          const double* g = dO",
                          "const double p = P[(int64_t)j * N + i];\n          const double* g = dO"),
}


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mdir = tmp_path / name
    mdir.mkdir()
    msrc = mdir / "m.cpp"
    msrc.write_text(src.replace(old, new))
    so = mdir / "m.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fopenmp", "-fPIC", "-shared", str(msrc),
                    "-o", str(so)], check=True)
    return oracle.bind(str(so))


def _pins_pass():
    rng = np.random.default_rng(5)
    B, H, W, C, nH, M, s = 1, 8, 8, 8, 2, 4, 2
    qkv = rng.standard_normal((B, H, W, 3 * C))
    table = rng.standard_normal(((2 * M - 1) ** 2, nH)) * 0.5
    G = rng.standard_normal((B, H, W, C))
    Y = oracle.fwd(qkv, table, nH, M, s)
    if np.abs(Y - brute_force_fwd(qkv, table, nH, M, s)).max() > 1e-12:
        return False
    tq = torch.from_numpy(qkv).requires_grad_(True)
    tt = torch.from_numpy(table).requires_grad_(True)
    (torch_swin_attention(tq, tt, nH, M, s) * torch.from_numpy(G)).sum().backward()
    dqkv, dtab = oracle.bwd(qkv, G, table, nH, M, s)
    return (np.abs(dqkv - tq.grad.numpy()).max() < 1e-10
            and np.abs(dtab - tt.grad.numpy()).max() < 1e-9)


def test_unmutated_oracle_passes(oracle_mod):
    assert _pins_pass()


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, tmp_path, name, monkeypatch):
    monkeypatch.setattr(oracle, "_lib", _build_mutant(tmp_path, name))
    assert not _pins_pass()

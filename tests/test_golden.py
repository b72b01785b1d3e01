"""Regression pins: the oracle reproduces the stored tiny-workload values written by
tests/golden/make_golden.py (which calls only the oracle). Also checks that the seeded
input generator still yields the same inputs."""
import os

import numpy as np

from swin_window_attention_gb300 import inputs

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    return np.loadtxt(os.path.join(HERE, name))


def test_tiny_golden(oracle_mod):
    wl = inputs.BY_NAME["tiny"]
    qkv = inputs.act_f64(inputs.make_qkv(wl))
    table = inputs.make_table(wl).double().numpy()
    dO = inputs.act_f64(inputs.make_dout(wl))
    Y = oracle_mod.fwd(qkv, table, wl.nH, wl.M, wl.s)
    dqkv, dtab = oracle_mod.bwd(qkv, dO, table, wl.nH, wl.M, wl.s)
    assert np.abs(Y[0, :, :, ::16].reshape(-1) - _load("tiny_fwd_Y_every16th_channel.txt")).max() < 1e-12
    assert np.abs(dtab.reshape(-1) - _load("tiny_bwd_dtable.txt")).max() < 1e-12
    assert np.abs(dqkv[0, :, :, ::16].reshape(-1)
                  - _load("tiny_bwd_dqkv_every16th_channel.txt")).max() < 1e-12


def test_table_generator_is_truncated():
    for wl in inputs.WORKLOADS:
        t = inputs.make_table(wl)
        assert t.shape == ((2 * wl.M - 1) ** 2, wl.nH)
        assert float(t.abs().max()) <= 0.04

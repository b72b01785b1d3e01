"""Writes the stored expected values under tests/golden/ by calling only the oracle.

The pages print no worked example, so these fixtures are regression pins: the oracle's
own output for the tiny workload (B=1, 8x8 tokens, C=64, two heads, 4x4 windows, shift
2, seeded inputs), sampled every 16th channel, and the full bias-table gradient for the
same inputs with a seeded upstream gradient. Run from the repository root:
``python tests/golden/make_golden.py``.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from swin_window_attention_gb300 import inputs  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def main():
    wl = inputs.BY_NAME["tiny"]
    qkv = inputs.act_f64(inputs.make_qkv(wl))
    table = inputs.make_table(wl).double().numpy()
    dO = inputs.act_f64(inputs.make_dout(wl))
    Y = oracle.fwd(qkv, table, wl.nH, wl.M, wl.s)
    dqkv, dtab = oracle.bwd(qkv, dO, table, wl.nH, wl.M, wl.s)
    hdr = "tiny workload (seed %d), oracle fp64; " % wl.seed
    np.savetxt(os.path.join(HERE, "tiny_fwd_Y_every16th_channel.txt"),
               Y[0, :, :, ::16].reshape(-1), fmt="%.17g",
               header=hdr + "Y[0,:,:,::16] flattened row-major")
    np.savetxt(os.path.join(HERE, "tiny_bwd_dtable.txt"), dtab.reshape(-1), fmt="%.17g",
               header=hdr + "dtable [(2M-1)^2, nH] flattened, upstream grad seed+2")
    np.savetxt(os.path.join(HERE, "tiny_bwd_dqkv_every16th_channel.txt"),
               dqkv[0, :, :, ::16].reshape(-1), fmt="%.17g",
               header=hdr + "dqkv[0,:,:,::16] flattened row-major")


if __name__ == "__main__":
    main()

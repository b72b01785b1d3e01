"""Multi-process host logic of data-parallel use, on CPU with gloo (world size 2): the
batch shards tile the batch exactly, and the summed per-shard bias-table gradients equal
the full-batch gradient. The per-shard gradients here come from the oracle (test code);
the library's own GPU path is covered by the single-GPU shard test."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from swin_window_attention_gb300.dp import allreduce_table_grad, shard_range


@pytest.mark.parametrize("batch,world", [(128, 2), (7, 2), (1, 2), (0, 3), (64, 8), (5, 4)])
def test_shards_tile_the_batch(batch, world):
    spans = [shard_range(batch, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == batch
    for (a, b), (c, d) in zip(spans, spans[1:]):
        assert b == c and b - a >= d - c >= b - a - 1


def test_bad_shard_requests():
    with pytest.raises(ValueError):
        shard_range(4, 0, 0)
    with pytest.raises(ValueError):
        shard_range(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        rng = np.random.default_rng(0)
        B, H, W, C, nH, M, s = 5, 8, 8, 64, 2, 4, 2
        qkv = rng.standard_normal((B, H, W, 3 * C))
        dY = rng.standard_normal((B, H, W, C))
        table = rng.standard_normal(((2 * M - 1) ** 2, nH)) * 0.02
        lo, hi = shard_range(B, world, rank)
        _, dt = oracle.bwd(qkv[lo:hi], dY[lo:hi], table, nH, M, s)
        t = torch.from_numpy(dt)
        allreduce_table_grad(t)
        if rank == 0:
            _, full = oracle.bwd(qkv, dY, table, nH, M, s)
            out.put(float(np.abs(t.numpy() - full).max()))
    finally:
        dist.destroy_process_group()


def test_table_gradient_allreduce_two_ranks(oracle_mod):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    assert q.get(timeout=5) < 1e-12

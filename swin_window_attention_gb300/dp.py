"""Data-parallel use of the fused window attention across processes (one GPU each).

Every (batch, window, head) unit is independent, so the batch is split into contiguous
shards and the forward needs no exchange. The backward has one: the relative-position
bias table is shared by every image, so its gradient is a sum over the shards, folded
into the data-parallel gradient all-reduce (NVIDIA Swin talk transcript, uticex.com
article 1598, section 2: data-parallel training; Baidu AIAK-Training talk, section 2:
synchronous gradient all-reduce after the backward). Nothing else crosses ranks.
"""
from __future__ import annotations


def shard_range(batch: int, world: int, rank: int):
    """Contiguous [lo, hi) batch rows of `rank`: sizes differ by at most one, larger
    shards first."""
    if world < 1 or not 0 <= rank < world or batch < 0:
        raise ValueError(f"bad shard request batch={batch} world={world} rank={rank}")
    base, extra = divmod(batch, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def allreduce_table_grad(dtable, group=None):
    """Sum the [(2M-1)^2, nH] fp32 bias-table gradient over the process group, in place
    (NCCL for CUDA tensors, gloo for CPU tensors). A no-op without a process group."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(dtable, op=dist.ReduceOp.SUM, group=group)
    return dtable

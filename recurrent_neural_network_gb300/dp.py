"""Data-parallel training of the stacked recurrent layers over ranks (one
process per GPU).

Every rank holds the same weights and a contiguous shard of the global batch.
Sequences are independent, so the forward pass, the backward pass through
time and the data gradients of a shard need nothing from the other ranks.
The weight gradients are sums over the batch (dW = sum over t and b of
dG^T [in | h_{t-1}]), so one all-reduce (sum) of dW per training step gives
every rank the gradient of the whole global batch: the one exchange step of a
data-parallel step.  ("Single stream parallelization of generalized LSTM-like
RNNs on a GPU", abstract: training with several parallel streams of
sequences.)

This module only moves data between ranks and slices batches; the arithmetic
of the method runs in librnn on each rank.
"""
from __future__ import annotations

import numpy as np
import torch


def global_batch(wl, world: int):
    """The workload of the whole job: `world` shards of wl.B sequences each."""
    return wl.replace(B=wl.B * world, name=f"{wl.name}_x{world}" if world > 1 else wl.name)


def shard(t, rank: int, world: int, dim: int = 1):
    """This rank's contiguous share of the batch dimension `dim` of a torch
    tensor or numpy array (x, y, dy: dim 1 of [T][B][.]; states: dim 1 of
    [L*D][B][H]).  The batch must divide evenly; None passes through."""
    if t is None:
        return None
    n = t.shape[dim]
    if world < 1 or not 0 <= rank < world or n % world:
        raise ValueError(f"shard: batch {n} over {world} ranks (rank {rank})")
    k = n // world
    if isinstance(t, np.ndarray):
        idx = [slice(None)] * t.ndim
        idx[dim] = slice(rank * k, (rank + 1) * k)
        return np.ascontiguousarray(t[tuple(idx)])
    return t.narrow(dim, rank * k, k).contiguous()


def allreduce_grads_(dw: torch.Tensor, group=None) -> torch.Tensor:
    """Sum the weight gradients over the ranks of `group`, in place, on the
    current stream (NCCL on GPUs, gloo on CPU).  A no-op on a single rank or
    without an initialised process group."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(dw, op=dist.ReduceOp.SUM, group=group)
    return dw

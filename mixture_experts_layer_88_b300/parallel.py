"""Data-parallel replicas of one layer: the exchanges the method has.

Every rank runs the whole layer on its own batch (the path shards by tokens).
The balancing rule of the V3 walk-through (section 2.2) compares each
expert's load with the mean load of the *batch*; with a batch split over R
ranks that is the global load, so before the sign update the [E] load counts
are summed over the ranks (one all-reduce of E int32) and every rank applies
the same update with T = the sum of the ranks' batch sizes.  The replicas'
biases then stay equal.

Training adds the parameter gradients: the loss of the whole batch is the sum
of the ranks' losses and every token's gradient depends only on that token
(its own routing and gates), so the gradient of each shared parameter
(centroids, routed and shared expert weights) is the sum of the ranks'
gradients; dx stays with the rank that owns the tokens.
"""
from __future__ import annotations

import copy

import torch
import torch.distributed as dist


def global_counts(counts: torch.Tensor, group=None) -> torch.Tensor:
    """Sums the [E] int32 load counts over the ranks of `group` in place."""
    if _distributed(group):
        dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    return counts


def _distributed(group=None) -> bool:
    return dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1


def global_tokens(T_local: int, device=None, group=None) -> int:
    """Tokens of the whole batch: the sum of every rank's T (ranks may hold
    batches of different sizes).  One all-reduce of a single int64 on
    `device` (the counts' device, so NCCL groups work too) and a host read of
    the result."""
    if not _distributed(group):
        return int(T_local)
    t = torch.tensor([int(T_local)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return int(t.item())


def global_cfg(cfg, group=None, T_global=None, device=None):
    """A copy of the layer config whose T is the batch over all ranks:
    T_global when the caller knows it, else the ranks' T summed by
    global_tokens."""
    g = copy.copy(cfg)
    g.T = int(T_global) if T_global is not None else global_tokens(cfg.T, device, group)
    return g


def balance_step(cfg, counts: torch.Tensor, bias: torch.Tensor, update, group=None,
                 T_global=None):
    """All-reduce the counts, then update(cfg_global, counts, bias): the sign
    update of every rank against the global mean load.  T_global (the tokens
    of all ranks together) may be given by a caller that knows it; otherwise
    it is summed over the ranks, which reads one value back to the host."""
    global_counts(counts, group)
    return update(global_cfg(cfg, group, T_global, counts.device), counts, bias)


PARAM_GRAD_KEYS = ("dcentroids", "dw13", "dw2", "dws13", "dws2")


def allreduce_grads(grads: dict, group=None, keys=PARAM_GRAD_KEYS) -> dict:
    """Sums the parameter gradients of moe_backward (a dict as from
    alloc_grads) over the ranks of `group` in place, one all-reduce per
    tensor in the order of `keys`; empty tensors (no shared experts) are
    skipped.  dx is left alone."""
    if not _distributed(group):
        return grads
    for k in keys:
        t = grads.get(k)
        if t is not None and t.numel() > 0:
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return grads

"""Data-parallel replicas of one layer: the exchanges the method has.

Every rank runs the whole layer on its own batch (the path shards by tokens).
The balancing rule of the V3 walk-through (section 2.2) compares each
expert's load with the mean load of the *batch*; with a batch split over R
ranks that is the global load, so before the sign update the [E] load counts
are summed over the ranks (one all-reduce of E int32) and every rank applies
the same update with T = R * T_local.  The replicas' biases then stay equal.

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
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    return counts


def global_cfg(cfg, group=None):
    """A copy of the layer config whose T is the batch over all ranks."""
    g = copy.copy(cfg)
    ws = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    g.T = cfg.T * ws
    return g


def balance_step(cfg, counts: torch.Tensor, bias: torch.Tensor, update, group=None):
    """All-reduce the counts, then update(cfg_global, counts, bias): the sign
    update of every rank against the global mean load."""
    global_counts(counts, group)
    return update(global_cfg(cfg, group), counts, bias)


PARAM_GRAD_KEYS = ("dcentroids", "dw13", "dw2", "dws13", "dws2")


def allreduce_grads(grads: dict, group=None, keys=PARAM_GRAD_KEYS) -> dict:
    """Sums the parameter gradients of moe_backward (a dict as from
    alloc_grads) over the ranks of `group` in place, one all-reduce per
    tensor in the order of `keys`; empty tensors (no shared experts) are
    skipped.  dx is left alone."""
    if not (dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1):
        return grads
    for k in keys:
        t = grads.get(k)
        if t is not None and t.numel() > 0:
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return grads

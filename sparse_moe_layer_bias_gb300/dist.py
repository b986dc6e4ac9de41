"""Data-parallel Quantile Balancing across ranks.

Tokens are independent, so data-parallel ranks run the layer on their own
batches with no exchange.  Quantile Balancing has one: each rank bins its own
tokens' router scores, the per-expert B-bin histograms are summed over all
ranks (counts add: the histogram of a union of token sets is the sum of their
histograms; "Kimi-K3-Architecture-Deep-Dive" section 3, Quantile Balancing,
aggregates the histograms across nodes this way),
and every rank then reads the same quantiles and sets the same biases.

The backward has one exchange as well: a weight gradient is a sum over tokens
(of outer products), so the gradient of the whole data-parallel batch is the
sum of the ranks' gradients over their own tokens, while dx stays per rank.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def qb_allreduce_histogram(hist: torch.Tensor, group=None) -> torch.Tensor:
    """Sum an [E, B] int32 histogram over the ranks of `group` in place (a
    no-op without an initialised process group or with one rank)."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(hist, op=dist.ReduceOp.SUM, group=group)
    return hist


def allreduce_weight_grads(grads: dict, group=None) -> dict:
    """Sum each weight gradient (lmoe_backward's fp32 tensors, by name) over
    the ranks of `group` in place, in a fixed name order so every rank issues
    the same sequence of collectives (a no-op without an initialised process
    group or with one rank)."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        for name in sorted(grads):
            dist.all_reduce(grads[name], op=dist.ReduceOp.SUM, group=group)
    return grads

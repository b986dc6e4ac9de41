"""Data-parallel Quantile Balancing across ranks.

Tokens are independent, so data-parallel ranks run the layer on their own
batches with no exchange.  Quantile Balancing has one: each rank bins its own
tokens' router scores, the per-expert B-bin histograms are summed over all
ranks (counts add: the histogram of a union of token sets is the sum of their
histograms; "Kimi-K3-Architecture-Deep-Dive" section 3, Quantile Balancing,
aggregates the histograms across nodes this way),
and every rank then reads the same quantiles and sets the same biases.
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

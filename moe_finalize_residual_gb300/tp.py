"""Tensor-parallel finalize over R ranks: the one-shot exchange of the rounded partial rows.

In the deployment the pages describe, each of R tensor-parallel ranks holds one partial of every token
(its own GEMM2 rows, routing weights and shared-expert output).  The fused op finalizes the rank's
partial, rounds it once, pushes the rounded row to every peer, and every rank then sums the R rows in
the fixed rank order 0..R-1, rounds once, and applies the residual add, RMSNorm and the optional
quantisation redundantly (flashinfer PR #6631, Description: one-shot all-reduce of each rank's finalized
row, rank sum in FP32, one rounding; flashinfer PR #3385, Description: ranks accumulated in the fixed
order 0..world_size-1 from rank-indexed slots).

Here the three steps are composed from this library's calls and one collective:

1. ``p_r``: the finalize-only call on the rank's own partial (one partial: the rounded p_r itself);
2. the one-shot exchange: an all-gather of every rank's ``p_r`` into rank-indexed slots;
3. the fused call over R exchanged partials, partial r having every route masked and slot r as its
   shared row, factor 1: each partial then rounds to ``p_r`` itself, and the kernel's rank sum, residual
   add, RMSNorm and quantisation are those of the single-GPU call, bit for bit.

The compute steps and the collective are parameters, so the protocol runs the same way over any
process group and any implementation of the two steps; by default they are this library's calls and
``torch.distributed.all_gather``.  On one GPU per process this is the path a multi-GPU deployment takes;
every run of this project has one GPU, so it is exercised by CPU process groups and by a single-GPU
emulation of its ranks.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence

import torch


def exchange_all_gather(p_r: torch.Tensor, group=None) -> List[torch.Tensor]:
    """The one-shot exchange: rank r's rounded partial lands in slot r of every rank.  The rows travel as
    raw 32-bit words (two 16-bit values each; H is a multiple of 8), so the exchange moves bytes and never
    converts a value."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    words = p_r.contiguous().view(torch.int32)
    slots = [torch.empty_like(words) for _ in range(world)]
    dist.all_gather(slots, words, group=group)
    return [s.view(p_r.dtype) for s in slots]


def exchanged_partials(slots: Sequence[torch.Tensor], partial_cls):
    """Partials that reproduce the exchanged rows: partial r has its single route masked (-1) and slot r
    as its shared row, so with factor 1 it rounds to slot r exactly."""
    T = slots[0].shape[0]
    masked = torch.full((T, 1), -1, dtype=torch.int32, device=slots[0].device)
    return [partial_cls(s[:1], masked, None, s) for s in slots]


def tp_finalize_fused(local, residual: torch.Tensor, gamma: torch.Tensor, *, routed_scaling_factor: float = 1.0,
                      eps: float = 1e-6, group=None,
                      finalize_partial: Optional[Callable] = None, exchange: Optional[Callable] = None,
                      fused: Optional[Callable] = None, **fused_kwargs):
    """The rank's share of a tensor-parallel finalize: returns what ``moe_finalize_fused`` returns, equal on
    every rank and equal, bit for bit, to the single-GPU call over all R partials.

    ``local`` is this rank's ``Partial``.  ``finalize_partial(local, rsf) -> p_r``, ``exchange(p_r, group) ->
    slots`` and ``fused(partials, residual, gamma, eps, **kw)`` default to the library's finalize-only call,
    ``torch.distributed.all_gather`` and the library's fused call; further keyword arguments (outputs,
    quantisation) go to ``fused``."""
    if finalize_partial is None or fused is None:
        import moe_finalize_residual_gb300 as mfr
        if finalize_partial is None:
            def finalize_partial(part, rsf):
                return mfr.moe_finalize_routed([part], routed_scaling_factor=rsf)
        if fused is None:
            def fused(parts, res, gam, eps_, **kw):
                return mfr.moe_finalize_fused(parts, res, gam, routed_scaling_factor=1.0, eps=eps_, **kw)
    exchange = exchange if exchange is not None else exchange_all_gather
    p_r = finalize_partial(local, routed_scaling_factor)
    slots = exchange(p_r, group)
    partial_cls = type(local)
    return fused(exchanged_partials(slots, partial_cls), residual, gamma, eps, **fused_kwargs)

"""Vocabulary-parallel linear-logp: one tensor-parallel rank per GPU, each holding a
contiguous range of the vocabulary.

Page "feat(rl-kernel): add CUDA linear logp provider integration", Changes / Megatron
integration: the provider is given the tensor-parallel vocabulary range, and tensor
parallelism is the vocabulary reduction group. Page "Perf/cuda compact top p replay",
Summary: shard results are reduced in rank order, and a rank whose shard has no replay
candidate contributes nothing rather than a NaN.

Each rank runs the library on its own shards only (a rank-local partition) and the ranks
exchange what the rank-ordered reduction needs:

  forward   lp_forward (or the logits-reuse / replay routes) on the rank's shards, with
            per-shard statistics -> all-gather of the [K_r, 3, T] statistics in rank
            order -> lp_merge_shard_stats over the whole partition. Every rank gets the
            same bits, and the bits one call over all shards on one GPU returns.
  backward  lp_backward on the rank's shards with the merged LSE (and entropy) -> this
            rank's share of dX; dW and db stay local -> all-gather of the dX shares in
            rank order -> lp_sum_partials adds them in that fixed order (never a
            reduction whose order can vary).

`linear_logp` wraps forward and backward for autograd. This module only moves data
(torch.distributed collectives) and calls the library; every arithmetic step runs in the
library's kernels. Collectives work on any backend: NCCL for GPU tensors, gloo for the
host-side tests of the exchange.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch
import torch.distributed as dist

from . import (VocabPartition, lp_backward_ex, lp_forward, lp_forward_from_logits, lp_merge_shard_stats,
               lp_sum_partials, lp_top_p_replay)

__all__ = ["rank_partition", "gather_in_rank_order", "gather_shard_stats", "merge", "forward",
           "forward_from_logits", "top_p_replay", "backward", "sum_over_ranks", "linear_logp"]


def rank_partition(full: VocabPartition, shard_ids: Sequence[int]) -> VocabPartition:
    """The rank-local partition of a rank holding the consecutive shards `shard_ids` of the
    whole-vocabulary partition `full`."""
    ids = list(shard_ids)
    if not ids or ids != list(range(ids[0], ids[0] + len(ids))):
        raise ValueError("a rank holds a non-empty run of consecutive shards")
    if ids[0] < 0 or ids[-1] >= len(full.ranges):
        raise ValueError("shard index outside the partition")
    return VocabPartition(full.vocab_real, full.vocab_padded, tuple(full.ranges[k] for k in ids), local=True)


def gather_in_rank_order(t: torch.Tensor, group=None) -> List[torch.Tensor]:
    """All-gather one tensor per rank; returns them in rank order (rank 0 first). Ranks may
    contribute different leading extents (e.g. different numbers of shards); the other
    dimensions, the dtype and the device must agree."""
    world = dist.get_world_size(group)
    t = t.contiguous()
    n = torch.tensor([t.shape[0]], dtype=torch.int64, device=t.device)
    ns = [torch.empty_like(n) for _ in range(world)]
    dist.all_gather(ns, n, group=group)
    counts = [int(x.item()) for x in ns]
    most = max(counts)
    if t.shape[0] < most:
        pad = torch.zeros((most - t.shape[0],) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        t = torch.cat([t, pad])
    bufs = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(bufs, t, group=group)
    return [b[:c] for b, c in zip(bufs, counts)]


def gather_shard_stats(shard_stats: torch.Tensor, group=None) -> torch.Tensor:
    """All ranks' per-shard statistics [K_r, 3, T], concatenated in rank order:
    [sum_r K_r, 3, T], the shards of the whole partition in ascending order."""
    return torch.cat(gather_in_rank_order(shard_stats, group), dim=0)


def merge(all_stats: torch.Tensor, y: torch.Tensor, full: VocabPartition, entropy: bool = True) -> dict:
    """The rank-ordered reduction of the gathered statistics (lp_merge_shard_stats)."""
    return lp_merge_shard_stats(all_stats, y, full, entropy=entropy)


def _finish(local: dict, y: torch.Tensor, full: VocabPartition, group, entropy: bool) -> dict:
    out = merge(gather_shard_stats(local["shard_stats"], group), y, full, entropy=entropy)
    out["local"] = local
    return out


def forward(X: torch.Tensor, W_local, b_local, full: VocabPartition, shard_ids: Sequence[int], y: torch.Tensor,
            tau: float, group=None, entropy: bool = True, workspace: Optional[torch.Tensor] = None) -> dict:
    """Fused forward across the tensor-parallel group: logp, lse, entropy of the whole
    vocabulary on every rank (plus this rank's own outputs under "local")."""
    part = rank_partition(full, shard_ids)
    local = lp_forward(X, W_local, b_local, part, y, tau, entropy=entropy, shard_stats=True, workspace=workspace)
    return _finish(local, y, full, group, entropy)


def forward_from_logits(logits_local, full: VocabPartition, shard_ids: Sequence[int], y: torch.Tensor, tau: float,
                        group=None, entropy: bool = True) -> dict:
    """Logits-reuse forward across the group (each rank streams its own shards' logits)."""
    part = rank_partition(full, shard_ids)
    local = lp_forward_from_logits(logits_local, part, y, tau, entropy=entropy, shard_stats=True)
    return _finish(local, y, full, group, entropy)


def top_p_replay(X: torch.Tensor, W_local, b_local, full: VocabPartition, shard_ids: Sequence[int],
                 replay_ids: torch.Tensor, y: torch.Tensor, tau: float, group=None) -> dict:
    """Compact top-p replay across the group: every rank gets the whole row's ids and
    scores those in its own range; the merged logp and LSE are over the whole set."""
    part = rank_partition(full, shard_ids)
    local = lp_top_p_replay(X, W_local, b_local, part, replay_ids, y, tau, shard_stats=True)
    return _finish(local, y, full, group, False)


def sum_over_ranks(partial: torch.Tensor, group=None, out_dtype=torch.float32) -> torch.Tensor:
    """Every rank's fp32 partial result, added in rank order (the same bits on every rank)."""
    shares = [p[0] for p in gather_in_rank_order(partial.unsqueeze(0), group)]
    return lp_sum_partials(shares, out_dtype=out_dtype)


def backward(X: torch.Tensor, W_local, b_local, full: VocabPartition, shard_ids: Sequence[int], y: torch.Tensor,
             tau: float, lse: torch.Tensor, grad_logp: torch.Tensor, entropy: Optional[torch.Tensor] = None,
             grad_entropy: Optional[torch.Tensor] = None, group=None, dx_dtype=torch.float32,
             workspace: Optional[torch.Tensor] = None) -> dict:
    """Backward across the group, given the merged lse (and entropy) of `forward`: dX of the
    whole vocabulary on every rank (the rank-ordered sum of the ranks' shares), and this
    rank's own dW and db."""
    part = rank_partition(full, shard_ids)
    g = lp_backward_ex(X, W_local, b_local, part, y, tau, lse, grad_logp, entropy=entropy,
                       grad_entropy=grad_entropy, workspace=workspace)
    dx_share = g["dX"]
    return {"dX": sum_over_ranks(dx_share, group, out_dtype=dx_dtype), "dW": g["dW"], "db": g["db"],
            "dX_local": dx_share}


class _VocabParallelLogp(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, full, shard_ids, y, tau, group, n, has_bias, *wb):
        W = list(wb[:n])
        bias = list(wb[n:]) if has_bias else None
        out = forward(X, W, bias, full, shard_ids, y, tau, group=group, entropy=True)
        ctx.full, ctx.shard_ids, ctx.tau, ctx.group, ctx.n, ctx.has_bias = full, shard_ids, tau, group, n, has_bias
        ctx.save_for_backward(X, y, out["lse"], out["entropy"], *wb)
        ctx.mark_non_differentiable(out["lse"])
        ctx.set_materialize_grads(False)
        return out["logp"], out["entropy"], out["lse"]

    @staticmethod
    def backward(ctx, g_logp, g_entropy, _g_lse):
        X, y, lse, entropy, *wb = ctx.saved_tensors
        n = ctx.n
        W = wb[:n]
        bias = wb[n:] if ctx.has_bias else None
        if g_logp is None and g_entropy is None:
            return (None,) * (8 + len(wb))
        g = g_logp.to(torch.float32).contiguous() if g_logp is not None else \
            torch.zeros(X.shape[0], dtype=torch.float32, device=X.device)
        h = g_entropy.to(torch.float32).contiguous() if g_entropy is not None else None
        part = rank_partition(ctx.full, ctx.shard_ids)
        want_db = bias is not None and any(b is not None and b.requires_grad for b in bias)
        r = lp_backward_ex(X, W, bias, part, y, ctx.tau, lse, g, bias_grad=want_db,
                           entropy=entropy if h is not None else None, grad_entropy=h,
                           dw_dtype=torch.bfloat16)
        # every rank's fp32 share of dX, added in rank order and rounded once to X's type
        dX = sum_over_ranks(r["dX"], ctx.group, out_dtype=torch.bfloat16) if ctx.needs_input_grad[0] else None
        dW = [d if ctx.needs_input_grad[8 + k] else None for k, d in enumerate(r["dW"])]
        db = [None] * n
        if want_db:
            db = [d if ctx.needs_input_grad[8 + n + k] else None for k, d in enumerate(r["db"])]
        return (dX, None, None, None, None, None, None, None, *dW, *(db if ctx.has_bias else []))


def linear_logp(X: torch.Tensor, W_local, b_local, full: VocabPartition, shard_ids: Sequence[int],
                y: torch.Tensor, tau: float, group=None):
    """Vocabulary-parallel linear-logp with autograd, called by every rank of the group with
    the same X, y and upstream gradients: returns (logp, entropy) of the whole vocabulary,
    differentiable with respect to X (the rank-ordered sum of every rank's share, the same on
    every rank) and this rank's W and bias (bf16 gradients)."""
    ids = list(shard_ids)
    n = len(ids)
    if len(W_local) != n:
        raise ValueError("W_local must have one entry per local shard")
    wb = list(W_local) + (list(b_local) if b_local is not None else [])
    logp, entropy, _ = _VocabParallelLogp.apply(X, full, tuple(ids), y, float(tau), group, n, b_local is not None,
                                                *wb)
    return logp, entropy

"""Vocabulary-parallel (tensor-parallel) cross-entropy over the shard calls of liblossk.so.

The weight's vocabulary rows are split into contiguous shards, one per rank of
a process group ("Fuse distillation + z-loss in the triton monolithic path
(#507)", section "Changes": its tests add a tensor-parallel distributed
subtest; section "Validation": the world_size=2 tensor-parallel subtests).
Rank r holds rows shard_range(vocab_total, world, r) of the weight, every rank
holds every token.  One training step per rank:

  1. lossk_ce_shard_fwd -> the shard's partials float[3][n_tok]
     (its log-sum-exp, the target logit if it holds the target, that flag);
  2. gather_partials: one all-gather of the 3 n_tok floats of every rank,
     stacked in rank order = shard order -> float[world][3][n_tok];
  3. lossk_ce_shard_combine -> lse, ce and the scalars of the whole vocabulary;
  4. lossk_ce_shard_bwd -> the shard's d_weight rows and its share of d_hidden;
  5. sum_d_hidden: one all-reduce (sum) of the shares -> d_hidden.

All arithmetic runs in the library's kernels; this module only moves the
partials and the d_hidden shares between ranks (torch.distributed: NCCL on
GPUs, gloo on CPUs) and marshals the calls.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def _world(group=None) -> int:
    return dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1


def shard_range(vocab_total: int, world: int, rank: int) -> tuple[int, int]:
    """(v0, rows) of rank `rank`'s shard: contiguous, in rank order, sizes
    differing by at most one row, together covering [0, vocab_total)."""
    if world < 1 or not 0 <= rank < world or vocab_total < world:
        raise ValueError(f"cannot split {vocab_total} rows over {world} ranks (rank {rank})")
    base, rem = divmod(vocab_total, world)
    return rank * base + min(rank, rem), base + (1 if rank < rem else 0)


def gather_partials(partials: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's partials [3][n], stacked in rank order: [world][3][n]."""
    world = _world(group)
    if world == 1:
        return partials.unsqueeze(0)
    parts = [torch.empty_like(partials) for _ in range(world)]
    dist.all_gather(parts, partials.contiguous(), group=group)
    return torch.stack(parts)


def sum_d_hidden(d_hidden_part: torch.Tensor, group=None) -> torch.Tensor:
    """The ranks' d_hidden shares summed in place (every rank gets d_hidden)."""
    if _world(group) > 1:
        dist.all_reduce(d_hidden_part, op=dist.ReduceOp.SUM, group=group)
    return d_hidden_part


def ce_fwd_bwd(hidden, weight_shard, targets, v0: int, vocab_total: int, loss_mask=None,
               z_weight: float = 0.0, grad_scale: float = 1.0, group=None, want_d_weight: bool = True):
    """One vocabulary-parallel training step on this rank's shard.

    Returns lse, ce and scalars (of the whole vocabulary, identical on every
    rank), d_hidden (summed over the ranks) and this shard's d_weight rows."""
    from . import lossk as L
    p = L.lossk_ce_shard_fwd(hidden, weight_shard, targets, v0, vocab_total)
    pa = gather_partials(p, group)
    c = L.lossk_ce_shard_combine(pa, loss_mask=loss_mask, z_weight=z_weight)
    g = L.lossk_ce_shard_bwd(hidden, weight_shard, targets, v0, vocab_total, c["lse"], loss_mask=loss_mask,
                             z_weight=z_weight, grad_scale=grad_scale, want_d_weight=want_d_weight)
    sum_d_hidden(g["d_hidden"], group)
    return {"lse": c["lse"], "ce": c["ce"], "scalars": c["scalars"], "d_hidden": g["d_hidden"],
            "d_weight": g["d_weight"], "partials": p}

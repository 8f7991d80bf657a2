"""Data-parallel exchange for sequence-sharded GRPO loss calls.

RL-Kernel "GRPO Loss" page, "Tensor and Data Parallel": a DP rank owns a
contiguous range of whole sequences (ranks in order); the only quantities
that cross ranks are the integer active-token counts (gathered, so the
normaliser is exact at every degree) and the per-sequence totals, gathered
and concatenated in rank order -- an exact byte copy, never an all_reduce,
whose combine order would follow the collective's topology.

    counts = dp.gather_counts(g.grpo_count_active(mask_local))
    tot = g.totals_buffer(B_local)
    res = g.grpo_loss_fwd_bwd(..., shard=g.Shard(seq_begin, counts, tot))
    out3 = g.grpo_loss_finalize(dp.gather_totals(tot), counts, ...)

gives, on every rank, the loss of the unsharded batch bit for bit; each
rank's gradient is its slice of the unsharded gradient, bit for bit.
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist


def _world(group) -> int:
    return dist.get_world_size(group) if dist.is_initialized() else 1


def gather_counts(local_counts: torch.Tensor, group=None) -> torch.Tensor:
    """The batch's (N, S): every rank's int64 [2] counts, summed as integers
    (exact in any order)."""
    if _world(group) == 1:
        return local_counts.clone()
    parts = [torch.empty_like(local_counts) for _ in range(_world(group))]
    dist.all_gather(parts, local_counts.contiguous(), group=group)
    return torch.stack(parts).sum(0)


def gather_totals(local_totals: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's per-sequence total records (uint8 [B_rank, 32]),
    concatenated in rank order.  Ranks may own different numbers of
    sequences: sizes are exchanged first and the records padded to the
    largest share for the collective, then trimmed."""
    world = _world(group)
    if world == 1:
        return local_totals.clone()
    dev = local_totals.device
    n = torch.tensor([local_totals.shape[0]], dtype=torch.int64, device=dev)
    sizes = [torch.empty_like(n) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    sizes = [int(s.item()) for s in sizes]
    width = local_totals.shape[1]
    pad = torch.zeros((max(sizes), width), dtype=local_totals.dtype, device=dev)
    pad[: local_totals.shape[0]] = local_totals
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    return torch.cat([p[:s] for p, s in zip(parts, sizes)])


def shard_bounds(num_sequences: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous [begin, end) of whole sequences for `rank` of `world`, in
    rank order (the page's sequence_shard_bounds), as even as possible."""
    base, extra = divmod(num_sequences, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def sequence_sharded_loss(fn, local_args: dict, mask_local: torch.Tensor, seq_begin: int,
                          *, beta: float, reduction="token_mean",
                          norm_constant: Optional[float] = None, group=None, **kw) -> dict:
    """One rank's share of a sequence-sharded call: `fn` is
    grpo_loss_fwd_bwd or grpo_loss_from_logps, `local_args` its positional
    tensors (this rank's sequences; rewards for the whole batch), `kw` its
    keyword options.  Returns the call's result with ``out3`` replaced by
    the batch's loss outputs."""
    from . import Shard, grpo_count_active, grpo_loss_finalize, totals_buffer
    counts = gather_counts(grpo_count_active(mask_local), group)
    tot = totals_buffer(mask_local.shape[0], mask_local.device)
    res = fn(*local_args.values(), beta=beta, reduction=reduction, norm_constant=norm_constant,
             shard=Shard(seq_begin, counts, tot), **kw)
    res["out3"] = grpo_loss_finalize(gather_totals(tot, group), counts, beta=beta,
                                     reduction=reduction, norm_constant=norm_constant)
    res["loss"], res["policy_loss"], res["kl"] = res["out3"][0], res["out3"][1], res["out3"][2]
    res["global_counts"] = counts
    return res

"""Data-parallel exchange for sequence-sharded GRPO loss calls.

RL-Kernel "GRPO Loss" page, "Tensor and Data Parallel": a DP rank owns a
contiguous range of whole sequences (ranks in order); the only quantities
that cross ranks are the integer active-token counts (gathered, so the
normaliser is exact at every degree) and the per-sequence totals, gathered
and concatenated in rank order -- an exact byte copy, never an all_reduce,
whose combine order would follow the collective's topology.  A TP rank
holds a slice of the vocabulary; its chunk records travel the same way
(gather_vocab_partials).

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


def gather_rows(local: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's tensor concatenated along dim 0 in rank order, as an
    exact copy.  Ranks may hold different numbers of rows (the trailing
    dims must agree): sizes are exchanged first and the rows padded to the
    largest share for the collective, then trimmed."""
    world = _world(group)
    if world == 1:
        return local.clone()
    dev = local.device
    n = torch.tensor([local.shape[0]], dtype=torch.int64, device=dev)
    sizes = [torch.empty_like(n) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    sizes = [int(s.item()) for s in sizes]
    pad = torch.zeros((max(sizes),) + tuple(local.shape[1:]), dtype=local.dtype, device=dev)
    pad[: local.shape[0]] = local
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    return torch.cat([p[:s] for p, s in zip(parts, sizes)])


def gather_totals(local_totals: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's per-sequence total records (uint8 [B_rank, 32]),
    concatenated in rank order."""
    return gather_rows(local_totals, group)


def gather_vocab_partials(parts: dict, group=None) -> dict:
    """The tensor-parallel exchange of grpo_vocab_partials' outputs: the
    chunk records of every rank concatenated in rank order (= chunk order),
    and the action logits summed over ranks in rank order (exact: exactly
    one rank holds each action, the others contribute 0)."""
    out = {k: gather_rows(parts[k], group) for k in ("part_p", "part_r")}
    act = parts["action_logits"]
    if _world(group) == 1:
        out["action_logits"] = act.clone()
    else:
        every = [torch.empty_like(act) for _ in range(_world(group))]
        dist.all_gather(every, act.contiguous(), group=group)
        out["action_logits"] = torch.stack(every).sum(0)
    return out


def vocab_shard_bounds(V: int, chunk: int, world: int, rank: int) -> tuple[int, int]:
    """[begin, end) of the vocabulary for `rank` of `world`: whole chunks, in
    rank order, as even as possible (the page's vocab_shard_bounds)."""
    nck = (V + chunk - 1) // chunk
    a, b = shard_bounds(nck, world, rank)
    return min(V, a * chunk), min(V, b * chunk)


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

"""Vocabulary-sharded verify across ranks: one fixed-width exchange per step.

When the logits of a step are split along the vocabulary (each rank holding
columns [v0, v1) of every row, as a tensor-parallel lm head leaves them), the
verify needs one exchange (jianc99/sglang PR #8, DFLASH adaptive-verification
commit: the scatter works on a vocabulary shard, the target-verify gather is
deferred).  Each rank reduces its slice of every row of the window to one
fixed-width record (sv_verify_chain_shard_rows); one all-gather gives every
rank every shard's records (their size depends only on the number of
requests and drafted positions, never on the data or on a rank-local
branch); every rank then merges them into the same outputs
(sv_verify_chain_shard_merge), which equal sv_verify_chain's on the whole
rows.  This module only places the shards and moves the records.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import sv


def shard_bounds(vocab: int, world: int, rank: int) -> tuple[int, int]:
    """Columns [v0, v1) of rank `rank` when `world` ranks split `vocab` in
    contiguous, balanced slices (the first vocab % world ranks one wider)."""
    if not 0 <= rank < world or vocab < world:
        raise ValueError("need 0 <= rank < world <= vocab")
    base, extra = divmod(vocab, world)
    v0 = rank * base + min(rank, extra)
    return v0, v0 + base + (1 if rank < extra else 0)


def exchange_records(records: torch.Tensor, group=None) -> torch.Tensor:
    """All ranks' records, [world, record bytes of one rank], ordered by rank:
    one all-gather of equal-sized buffers (NCCL for device tensors, gloo for
    host tensors)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(records) for _ in range(world)]
    dist.all_gather(parts, records.contiguous(), group=group)
    return torch.stack(parts)


def verify_chain_sharded(target_shard: torch.Tensor, draft_shard: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                         temperature: torch.Tensor, top_k: Optional[torch.Tensor], top_p: Optional[torch.Tensor],
                         v0: int, vocab: int, verify_len: Optional[torch.Tensor] = None, seed: int = 0,
                         group=None, ws: Optional[sv.Workspace] = None) -> sv.VerifyOut:
    """One verify step over this rank's vocabulary shard: records, the
    exchange (skipped when torch.distributed is not initialised: one shard
    holds the whole vocabulary), the merge.  Every rank returns the same
    outputs."""
    rec = sv.verify_chain_shard_rows(target_shard, draft_shard, draft_tokens, temperature, top_k, top_p, v0, vocab,
                                     verify_len=verify_len, ws=ws)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        all_rec = exchange_records(rec, group)
    else:
        all_rec = rec[None]
    return sv.verify_chain_shard_merge(all_rec, all_rec.shape[0], draft_tokens, temperature, top_k, top_p, vocab,
                                       verify_len=verify_len, seed=seed, ws=ws)

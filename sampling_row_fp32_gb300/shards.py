"""Vocabulary shards: the host side of selecting over a row split by id range.

llama.cpp PR 49 ("Problem") runs the output head under a tensor split: each
GPU computes the logits of one contiguous share of the vocabulary. Selection
then runs per shard and merges:

1. `shard_offsets(V, G)` splits [0, V) into G contiguous ranges. Every
   boundary is a multiple of 4, so each slice starts on a 16-byte boundary
   and takes the library's bulk-copy path.
2. Each rank runs `sel_topk` (k = the policy's top_k, or 1 for argmax) on
   its slice, with shard-local ids.
3. `gather_lists` all-gathers the per-rank lists into `[rows][G][k]`, rank
   order = shard order (NCCL between GPUs; gloo works the same on CPU).
4. `sel_merge_shards` / `sel_sample_shards` (C ABI) merge on the device. The
   result equals `sel_topk` / `sel_sample` on the unsharded row.

Only the gather moves data between ranks: G * k (value, id) pairs per row.
"""
from __future__ import annotations

import torch

ALIGN = 4  # elements: a 16-byte boundary for fp32


def shard_offsets(V: int, G: int, min_size: int = 1, align: int = ALIGN) -> list[int]:
    """G + 1 increasing offsets splitting [0, V) into G near-equal ranges whose
    inner boundaries are multiples of `align`, each at least `min_size` ids.
    Raises ValueError if V cannot be split so."""
    if G < 1:
        raise ValueError("G must be >= 1")
    if V < 1:
        raise ValueError("V must be >= 1")
    offs = [0]
    for g in range(1, G):
        o = (V * g // G) // align * align
        offs.append(o)
    offs.append(V)
    for g in range(G):
        if offs[g + 1] - offs[g] < max(1, min_size):
            raise ValueError(f"cannot split V={V} into {G} shards of >= {min_size} ids "
                             f"on {align}-element boundaries")
    return offs


def shard_range(V: int, G: int, rank: int, min_size: int = 1) -> tuple[int, int]:
    """The [lo, hi) id range of shard `rank`."""
    offs = shard_offsets(V, G, min_size)
    return offs[rank], offs[rank + 1]


def gather_lists(vals: torch.Tensor, ids: torch.Tensor, group=None):
    """All-gather this rank's per-row lists ([rows][k] values and shard-local
    ids) into [rows][G][k] tensors on every rank, shard g = rank g. Uses the
    default process group unless `group` is given."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if vals.shape != ids.shape or vals.dim() != 2:
        raise ValueError("vals and ids must both be [rows][k]")
    ids32 = ids.view(torch.int32) if ids.dtype == torch.uint32 else ids
    vs = [torch.empty_like(vals) for _ in range(world)]
    is_ = [torch.empty_like(ids32) for _ in range(world)]
    dist.all_gather(vs, vals.contiguous(), group=group)
    dist.all_gather(is_, ids32.contiguous(), group=group)
    return torch.stack(vs, dim=1).contiguous(), torch.stack(is_, dim=1).contiguous()

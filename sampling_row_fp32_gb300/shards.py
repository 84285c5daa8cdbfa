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

Filters that look at the whole row take one more record per row and shard
(`sel_topk_stats` writes the list and a 48-byte `sel_row_stats` record from
one read of the slice):

- top-n-sigma (top_k > 0): the gathered statistics give the row's standard
  deviation; `sel_sample_shards` writes the result directly.
- top_k = 0 (full-row sampling): `sel_sample_shards` writes a 48-byte plan
  per row (the survivor set, decided from the merged 64 candidates and the
  merged normaliser). Each shard then sums its survivors' mass
  (`sel_shard_draw_mass`), `gather_masses` all-gathers the [rows][G] masses,
  each shard runs `sel_shard_draw` (the shard the draw falls in writes the
  global id, the others SEL_OTHER_SHARD and probability 0), and
  `combine_draws` all-reduces them (minimum id, summed probability).

Speculative acceptance on shards follows the same pattern: `spec_shard_stats`
reduces each slice of every target and draft row to a 32-byte part (max,
normaliser, first argmax id, logit at the draft token), `gather_parts`
all-gathers them, `spec_accept_shards` runs the acceptance chain on every
rank, and, in the rejection rule, the residual draw runs on the slices
(`spec_shard_draw_mass`, `gather_masses`, `spec_shard_draw`) before
`combine_emitted` all-reduces the emitted tokens (minimum).
"""
from __future__ import annotations

import numpy as np
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


# struct sel_row_stats, as numpy sees it (48 bytes)
ROW_STATS_DTYPE = np.dtype([("max", "<f4"), ("flags", "<u4"), ("x0", "<f4"), ("n", "<u4"),
                            ("s1", "<f8"), ("s2", "<f8"), ("z", "<f8"), ("h", "<f8")])
assert ROW_STATS_DTYPE.itemsize == 48
FULL_ROW_CANDIDATES = 64
OTHER_SHARD = 0xFFFFFFFE


def stats_records(stats: torch.Tensor) -> np.ndarray:
    """[..., 48] uint8 statistics (device or host) as a numpy record array."""
    a = stats.detach().cpu().contiguous().numpy()
    return a.view(ROW_STATS_DTYPE)[..., 0]


def full_row_list_len(offsets: list[int]) -> int:
    """Entries per shard list for full-row sampling on shards: the 64
    candidates, or fewer when a shard is narrower."""
    return min(FULL_ROW_CANDIDATES, min(offsets[g + 1] - offsets[g] for g in range(len(offsets) - 1)))


def gather_stats(stats: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather this rank's [rows][48] statistics into [rows][G][48]."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if stats.dim() != 2 or stats.shape[1] != ROW_STATS_DTYPE.itemsize or stats.dtype != torch.uint8:
        raise ValueError("stats must be [rows, 48] uint8")
    parts = [torch.empty_like(stats) for _ in range(world)]
    dist.all_gather(parts, stats.contiguous(), group=group)
    return torch.stack(parts, dim=1).contiguous()


def gather_masses(mass: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather this rank's [rows] float64 survivor masses into [rows][G]."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if mass.dim() != 1 or mass.dtype != torch.float64:
        raise ValueError("mass must be [rows] float64")
    parts = [torch.empty_like(mass) for _ in range(world)]
    dist.all_gather(parts, mass.contiguous(), group=group)
    return torch.stack(parts, dim=1).contiguous()


def _ids64(ids: torch.Tensor) -> torch.Tensor:
    # ids as unsigned 32-bit values in int64, so that the minimum orders
    # SEL_OTHER_SHARD and SEL_INVALID_ID above every real id
    return ids.view(torch.int32).to(torch.int64) & 0xFFFFFFFF


def combine_draws(ids: torch.Tensor, probs: torch.Tensor, group=None):
    """All-reduce the shards' sel_shard_draw outputs: the row's id (minimum:
    one shard holds the id, the others SEL_OTHER_SHARD; a failed row is
    SEL_INVALID_ID everywhere) and probability (sum: the others hold 0).
    Returns (ids as int64 holding uint32 values, probs float32)."""
    import torch.distributed as dist

    i = _ids64(ids)
    p = probs.clone()
    dist.all_reduce(i, op=dist.ReduceOp.MIN, group=group)
    dist.all_reduce(p, op=dist.ReduceOp.SUM, group=group)
    return i, p


def combine_draws_local(ids: list[torch.Tensor], probs: list[torch.Tensor]):
    """combine_draws for shards held by one process (shard g's outputs at
    index g)."""
    i = torch.stack([_ids64(t) for t in ids]).min(dim=0).values
    p = torch.stack(probs).sum(dim=0)
    return i, p


def gather_parts(parts: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather this rank's [S][2K+1][32] spec parts into [S][G][2K+1][32]."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if parts.dim() != 3 or parts.shape[2] != 32 or parts.dtype != torch.uint8:
        raise ValueError("parts must be [S, 2K+1, 32] uint8")
    out = [torch.empty_like(parts) for _ in range(world)]
    dist.all_gather(out, parts.contiguous(), group=group)
    return torch.stack(out, dim=1).contiguous()


def gather_spec_masses(mass: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather this rank's [S][2] float64 draw masses into [S][G][2]."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if mass.dim() != 2 or mass.shape[1] != 2 or mass.dtype != torch.float64:
        raise ValueError("mass must be [S, 2] float64")
    out = [torch.empty_like(mass) for _ in range(world)]
    dist.all_gather(out, mass.contiguous(), group=group)
    return torch.stack(out, dim=1).contiguous()


def combine_emitted(emitted: torch.Tensor, group=None) -> torch.Tensor:
    """All-reduce (minimum) the ranks' emitted tokens after spec_shard_draw:
    the drawn token's shard holds its global id, the others SEL_OTHER_SHARD.
    Returns int64 holding the uint32 values."""
    import torch.distributed as dist

    e = _ids64(emitted)
    dist.all_reduce(e, op=dist.ReduceOp.MIN, group=group)
    return e


def combine_emitted_local(emitted: list[torch.Tensor]) -> torch.Tensor:
    """combine_emitted for shards held by one process."""
    return torch.stack([_ids64(e) for e in emitted]).min(dim=0).values

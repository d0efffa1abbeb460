"""Column-parallel latent-MoE tail across tensor-parallel ranks, one GPU per rank.

The multi-GPU form of the tail in PR #50383's `_shard_up_proj_tail` (key source,
tier 2, "COLUMN_PARALLEL"), and the split its PR #51253 runner test checks
(`_check_matches_replicated`, `_check_writes_only_its_own_shard`). Every rank
holds its own routed partial [T, L] and shared partial [T, H]:

1. the routed partials are summed over the ranks (all-reduce), so every rank has
   the whole latent sum;
2. every rank normalizes it (RMSNorm with weight g, or none);
3. rank r owns the output columns [start_r, end_r) and adds latent . W[start_r:end_r]^T
   into those columns of its own shared partial, in place (the narrowed beta-add
   `hidden_shard.addmm_(latent, up_proj_shard.t())`); every other column of its
   buffer keeps the shared partial;
4. an all-reduce of the whole [T, H] buffer over the ranks sums the shared
   partials and stitches the column shards at once, because each column received
   its projection on exactly one rank.

Steps 2-3 run in this library's CUDA kernels through the C ABI
(`latent_tail_norm`, `latent_tail_project_cols` with the rank's shared partial
as both its only partial and its output); steps 1 and 4 are NCCL collectives of
torch.distributed. The column ranges need not divide H evenly: they are
multiples of 8 that tile [0, H).

`routed_exchange="all_gather"` replaces the bf16 all-reduce of step 1 by an
all-gather of the ranks' partials, which the norm kernel then sums in FP32 (the
same stacked-partials reduction as a single-GPU call), at the cost of moving
world x [T, L] instead of about 2 x [T, L] per rank.
"""

from __future__ import annotations

from typing import Callable, Optional


def shard_range(H: int, rank: int, world: int) -> tuple[int, int]:
    """Columns [start, end) that `rank` of `world` owns: multiples of 8 tiling
    [0, H), as equal as 8-column granularity allows (equal to the pages'
    H / tp slices whenever tp divides H / 8)."""
    if H % 8 != 0:
        raise ValueError("H must be a multiple of 8")
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    groups = H // 8
    return (groups * rank // world) * 8, (groups * (rank + 1) // world) * 8


def _cuda_project(routed_stack, norm_weight, eps, W, shared_rank, start, end, stream=None):
    """Steps 2-3 on this rank's GPU: latent = rms_norm(sum of routed_stack), then
    shared_rank[:, start:end] += latent . W[start:end]^T in place."""
    import torch

    from . import binding

    T, L = routed_stack.shape[1], routed_stack.shape[2]
    latent = torch.empty(T, L, dtype=torch.bfloat16, device=routed_stack.device)
    binding.latent_tail_norm(routed_stack, norm_weight, latent, eps, stream)
    binding.latent_tail_project_cols(latent, shared_rank.unsqueeze(0), W, shared_rank, start, end,
                                     stream)


def shard_up_proj_partial(routed_partial, shared_partial, norm_weight, W, eps: float,
                          group=None, routed_exchange: str = "all_reduce",
                          project: Optional[Callable] = None):
    """Steps 1-3: returns this rank's [T, H] buffer before the final reduction
    (`shared_partial` itself, updated in place on the rank's columns only).

    routed_partial [T, L], shared_partial [T, H] bf16 on this rank's device;
    norm_weight [L] fp32 or None; W [H, L] bf16 (replicated). `project`
    replaces the CUDA steps 2-3 (same signature as the default); it exists for
    the host-side tests of the partition and of the collectives."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    T, L = routed_partial.shape
    H = W.shape[0]
    if tuple(shared_partial.shape) != (T, H) or tuple(W.shape) != (H, L):
        raise ValueError("routed_partial [T, L], shared_partial [T, H], W [H, L]")
    if routed_exchange == "all_reduce":
        summed = routed_partial.clone()
        dist.all_reduce(summed, group=group)
        routed_stack = summed.unsqueeze(0)
    elif routed_exchange == "all_gather":
        parts = [torch.empty_like(routed_partial) for _ in range(world)]
        dist.all_gather(parts, routed_partial.contiguous(), group=group)
        routed_stack = torch.stack(parts)
    else:
        raise ValueError("routed_exchange must be 'all_reduce' or 'all_gather'")
    start, end = shard_range(H, rank, world)
    (project or _cuda_project)(routed_stack.contiguous(), norm_weight, eps, W, shared_partial,
                               start, end)
    return shared_partial


def column_parallel_tail(routed_partial, shared_partial, norm_weight, W, eps: float,
                         group=None, routed_exchange: str = "all_reduce",
                         project: Optional[Callable] = None):
    """The whole tail (steps 1-4): every rank returns the full [T, H] output,
    W . rms_norm(sum over ranks of routed) + sum over ranks of shared. The
    result is written into `shared_partial`, which is also returned."""
    import torch.distributed as dist

    out = shard_up_proj_partial(routed_partial, shared_partial, norm_weight, W, eps, group,
                                routed_exchange, project)
    dist.all_reduce(out, group=group)
    return out

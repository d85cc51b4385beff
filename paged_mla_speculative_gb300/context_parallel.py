"""Context-parallel verify: one batch's keys sharded over the ranks of a group.

The partial + reduce design of "The Decisive A/B: When Benchmarking Honesty
Reveals the Real Bottleneck" (section "The Context") splits a request's KV
into ranges whose normalised partials (out_s, lse_s) a reduce step merges.
Taken across GPUs it becomes the context-parallel split of a long request:
rank r of a group of S computes the partial of shard r of every request's
keys (``mla_verify_attn_partial``), the ranks all-gather the partials into
shard-major buffers -- the one exchange step, B*T*H*513 floats per rank --
and every rank merges them (``mla_verify_combine_parts``).  Shard r covers
the request's 128-key blocks floor(r*nb/S) .. floor((r+1)*nb/S) - 1, so every
rank reads a disjoint slice of the cache.

This module is the host logic only: the gather and the order of the steps.
The partial and the merge run in the library's kernels; ``run_sharded``
takes them as callables, which is how the exchange is tested on CPU ranks.
"""
from __future__ import annotations

from typing import Callable, Optional, Tuple

import torch
import torch.distributed as dist


def _group_rank_size(group) -> Tuple[int, int]:
    if not dist.is_available() or not dist.is_initialized():
        return 0, 1
    return dist.get_rank(group), dist.get_world_size(group)


def gather_parts(part_out: torch.Tensor, part_lse: torch.Tensor, group=None):
    """All-gather one partial per rank into shard-major tensors.

    part_out [B,T,H,512], part_lse [B,T,H] (fp32, contiguous) ->
    parts_out [S,B,T,H,512], parts_lse [S,B,T,H], entry s from rank s.
    """
    rank, world = _group_rank_size(group)
    if world == 1:
        return part_out.unsqueeze(0), part_lse.unsqueeze(0)
    parts_out = torch.empty((world,) + tuple(part_out.shape), dtype=part_out.dtype,
                            device=part_out.device)
    parts_lse = torch.empty((world,) + tuple(part_lse.shape), dtype=part_lse.dtype,
                            device=part_lse.device)
    if dist.get_backend(group) == "nccl":
        dist.all_gather_into_tensor(parts_out, part_out.contiguous(), group=group)
        dist.all_gather_into_tensor(parts_lse, part_lse.contiguous(), group=group)
    else:
        dist.all_gather(list(parts_out.unbind(0)), part_out.contiguous(), group=group)
        dist.all_gather(list(parts_lse.unbind(0)), part_lse.contiguous(), group=group)
    return parts_out, parts_lse


def run_sharded(partial_fn: Callable[[int, int], Tuple[torch.Tensor, torch.Tensor]],
                combine_fn: Callable[[torch.Tensor, torch.Tensor], Tuple[torch.Tensor, torch.Tensor]],
                group=None):
    """partial_fn(shard, num_shards) -> (part_out, part_lse) of this rank's
    shard; gather; combine_fn(parts_out, parts_lse) -> (out, lse)."""
    rank, world = _group_rank_size(group)
    part_out, part_lse = partial_fn(rank, world)
    parts_out, parts_lse = gather_parts(part_out, part_lse, group)
    return combine_fn(parts_out, parts_lse)


def mla_verify_attn_context_parallel(plan, q, kv_cache, kv_indices, kv_indptr, kv_lens,
                                     draft_parent, scale: float, group=None,
                                     out: Optional[torch.Tensor] = None,
                                     lse: Optional[torch.Tensor] = None, stream=None):
    """The verify attention with every request's keys sharded over `group`
    (each rank passes the same q / indices / lengths / parents and reads its
    own shard of the cache); every rank returns the full (out, lse)."""
    from . import binding

    def partial(shard, num_shards):
        return binding.mla_verify_attn_partial(plan, q, kv_cache, kv_indices, kv_indptr, kv_lens,
                                               draft_parent, scale, shard, num_shards,
                                               stream=stream)

    def combine(parts_out, parts_lse):
        return binding.mla_verify_combine_parts(plan, parts_out, parts_lse, out, lse, stream=stream)

    return run_sharded(partial, combine, group)

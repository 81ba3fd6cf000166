"""Decode context parallelism (DCP) over a torch.distributed process group.

Each rank attends to its share of every query token's top-k (a contiguous
range of the selection's columns), the ranks' normalised partial outputs and
natural-log LSEs are exchanged, and every rank merges them with
sparse_mla_merge_states. The Prime Inference post (section "Native NVFP4
sparse MLA decode kernel") tried this split across GPUs and found it not worth
it at 2048 selected tokens per query; it is here for longer selections.

With the gloo backend the partials are staged through host memory; with
nccl they stay on the device. Every step of the attention and of the merge
runs in the library's CUDA kernels; this module only shards indices and moves
the partial states.
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import sparse_mla_decode, sparse_mla_merge_states


def shard_bounds(topk: int, rank: int, world: int):
    """Column range [lo, hi) of the top-k that `rank` of `world` attends to."""
    per = (topk + world - 1) // world
    lo = min(rank * per, topk)
    return lo, min(lo + per, topk)


def shard_topk(topk_idx: torch.Tensor, rank: int, world: int) -> torch.Tensor:
    """This rank's columns of topk_idx [num_q, topk]; a rank whose range is
    empty gets one column of -1 (an empty part: output 0, LSE -inf)."""
    lo, hi = shard_bounds(topk_idx.shape[1], rank, world)
    if hi <= lo:
        return torch.full((topk_idx.shape[0], 1), -1, dtype=topk_idx.dtype,
                          device=topk_idx.device)
    return topk_idx[:, lo:hi].contiguous()


def gather_states(part_out: torch.Tensor, part_lse: torch.Tensor, group=None):
    """All ranks' partial states stacked in rank order: ([W,num_q,H,512], [W,num_q,H]).
    Host-staged through the gloo backend, device-resident through nccl."""
    world = dist.get_world_size(group)
    host = dist.get_backend(group) == "gloo"
    dev = part_out.device
    po = part_out.cpu() if host else part_out
    pl = part_lse.cpu() if host else part_lse
    outs = [torch.empty_like(po) for _ in range(world)]
    lses = [torch.empty_like(pl) for _ in range(world)]
    dist.all_gather(outs, po.contiguous(), group=group)
    dist.all_gather(lses, pl.contiguous(), group=group)
    return torch.stack(outs).to(dev), torch.stack(lses).to(dev)


def dcp_sparse_mla_decode(q_latent, q_rope, q_seq, topk_idx, block_table, seq_lens,
                          page_size: int, cache, num_blocks: int, block_stride_bytes: int,
                          row_format: int, sm_scale: float, latent_scale: float = 1.0,
                          rope_scale: float = 1.0, out_fp32: bool = False, group=None,
                          invalid_count: Optional[torch.Tensor] = None):
    """sparse_mla_decode with the top-k split over the ranks of `group`.

    Every rank passes the same query tokens and full top-k (and holds the
    cache rows its share selects); every rank returns the merged result.
    """
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    local = shard_topk(topk_idx, rank, world)
    part_out, part_lse = sparse_mla_decode(q_latent, q_rope, q_seq, local, block_table, seq_lens,
                                           page_size, cache, num_blocks, block_stride_bytes,
                                           row_format, sm_scale, latent_scale, rope_scale,
                                           out_fp32=True, invalid_count=invalid_count)
    all_out, all_lse = gather_states(part_out, part_lse, group)
    return sparse_mla_merge_states(all_out, all_lse, out_fp32=out_fp32)

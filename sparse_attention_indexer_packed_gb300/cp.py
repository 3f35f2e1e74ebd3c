"""Indexer context parallelism: each rank holds one contiguous shard of every
request's index keys and scores it (idx_score_local_blocks, the per-shard
scorer sglang #42614 calls score_local_blocks); the ranks then exchange their
lists and every rank re-selects (idx_topk_merge).

The exchange is one all-gather of R * P*G * topk (id, score) pairs per rank over
torch.distributed (NCCL between GPUs); nothing else crosses ranks.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _lib


def gather_shard_lists(ids: torch.Tensor, scores: torch.Tensor, group=None):
    """All-gather every rank's [R, P*G, topk] lists into [world, R, P*G, topk]
    tensors, shard w at index w (the rank order of ``group``)."""
    world = dist.get_world_size(group)
    ids = ids.contiguous()
    scores = scores.contiguous()
    out_ids = [torch.empty_like(ids) for _ in range(world)]
    out_sc = [torch.empty_like(scores) for _ in range(world)]
    dist.all_gather(out_ids, ids, group=group)
    dist.all_gather(out_sc, scores, group=group)
    return torch.stack(out_ids), torch.stack(out_sc)


def context_parallel_step(q, q_scale, k_payload, k_scale, k_dtype, page_table, block_begin,
                          slot_ids, row_lens, n_slots, packed_queries, gqa, init_blocks,
                          local_blocks, topk, out_ids, out_scores, workspace, group=None,
                          stream=None) -> None:
    """This rank's part of the step: score its shard (page_table covers global
    blocks [block_begin, block_begin + max_pages / 2)), exchange, re-select into
    out_ids / out_scores [R, P*G, topk] (the same on every rank)."""
    R, M = int(q.shape[0]), packed_queries * gqa
    local_ids = torch.empty((R, M, topk), dtype=torch.int32, device=q.device)
    local_sc = torch.empty((R, M, topk), dtype=torch.float32, device=q.device)
    _lib.idx_score_local_blocks(q, q_scale, k_payload, k_scale, k_dtype, page_table, block_begin,
                                slot_ids, row_lens, packed_queries, gqa, init_blocks,
                                local_blocks, topk, local_ids, local_sc, workspace, stream)
    all_ids, all_sc = gather_shard_lists(local_ids, local_sc, group)
    _lib.idx_topk_merge(all_ids, all_sc, slot_ids, row_lens, n_slots, packed_queries, gqa,
                        init_blocks, local_blocks, topk, out_ids, out_scores, stream)

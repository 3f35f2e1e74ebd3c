"""Packed index score + block top-k, as a plain definition in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The step, as the pages define it:

* sglang #45451, Modifications: a request's packed_queries draft rows times its
  gqa heads (at most 16) share one dot tile against the request's index K; each
  row keeps its own length mask; the block score is the max (Accuracy Tests:
  "selected-block scores (max; ...)").
* sglang #42614 "[AMD] MiniMax-M3 indexer CP: packed scoring for EAGLE verify
  rows", Modifications 1: tile row i is (draft row i // gqa, head i % gqa);
  masking and the forced init/local blocks use each row's own length; a slot
  past the request table is graph padding and reads nothing.
* same page, Accuracy Tests: selection is exact (the same block IDs as a
  per-row selector, on every head); K is reached through a permuted, gapped
  slot table, never through the row or group index.

Readings where the pages are silent (each listed in the design notes):
  score = raw dot q.k with no softmax scale; block = 128 tokens, page = 64
  tokens; a row that ends at token t has length t + 1; the forced blocks are
  emitted with their real block max and count towards topk; candidates are
  ranked by block max descending, ties to the lower block id; output order is
  the forced blocks ascending, then the chosen candidates in rank order, then
  (-1, -inf) pads; a row with fewer than topk blocks emits all of them and pads;
  a request whose slot is outside [0, n_slots) is a pad (all rows padded); a row
  of length <= 0 is all padding; fp8 keys are code x per-key fp32 scale and fp8
  queries code x per-row fp32 scale.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import formats

PAGE = 64
BLOCK = 128


def key_rows(page_table: np.ndarray, slot: int, n_tokens: int) -> np.ndarray:
    """Physical pool rows of tokens [0, n_tokens) of the request in ``slot``:
    page_table[slot, t // 64] * 64 + t % 64 (slot-table addressing,
    sglang #42614 Accuracy Tests)."""
    t = np.arange(n_tokens, dtype=np.int64)
    return page_table[slot, t // PAGE].astype(np.int64) * PAGE + t % PAGE


def dequant_keys(k_dtype: str, payload: np.ndarray, scale, rows: np.ndarray) -> np.ndarray:
    """Dequantised float64 keys [len(rows), 128] read from the pool planes."""
    if k_dtype == "bf16":
        return formats.bf16_dequantize(payload[rows])
    if k_dtype == "fp8_e4m3":
        return formats.fp8_dequantize(payload[rows], scale[rows])
    if k_dtype == "nvfp4":
        return formats.nvfp4_dequantize(payload[rows], scale[rows])
    raise ValueError(k_dtype)


def dequant_query(q_dtype: str, q_row: np.ndarray, q_scale) -> np.ndarray:
    """One packed query row [128] as float64 (bf16 bits, or e4m3 code x scale)."""
    if q_dtype == "bf16":
        return formats.bf16_bits_to_f32(q_row).astype(np.float64)
    if q_dtype == "fp8_e4m3":
        return formats.E4M3_TABLE[np.asarray(q_row, dtype=np.uint8)] * float(q_scale)
    raise ValueError(q_dtype)


def num_blocks(length: int) -> int:
    """Blocks a row of ``length`` tokens covers: ceil(length / 128)."""
    return 0 if length <= 0 else (length + BLOCK - 1) // BLOCK


def row_block_max(q: np.ndarray, keys: np.ndarray, length: int) -> np.ndarray:
    """blockmax[b] = max over tokens t in [128 b, min(128 b + 128, length)) of
    q . k_t, for b < ceil(length / 128) (the row's own causal length mask)."""
    nb = num_blocks(length)
    s = keys[:length] @ q                       # float64 dot per token
    return np.array([s[b * BLOCK:min((b + 1) * BLOCK, length)].max() for b in range(nb)],
                    dtype=np.float64)


def row_block_lse(q: np.ndarray, keys: np.ndarray, length: int) -> np.ndarray:
    """The log-sum-exp block score (sglang #45451, Accuracy Tests: selected-block
    scores "max; lse"): lse[b] = ln sum over tokens t in
    [128 b, min(128 b + 128, length)) of exp(q . k_t), natural log, raw scores."""
    nb = num_blocks(length)
    s = keys[:length] @ q
    out = []
    for b in range(nb):
        blk = s[b * BLOCK:min((b + 1) * BLOCK, length)]
        m = blk.max()
        out.append(m + np.log(np.exp(blk - m).sum()))
    return np.array(out, dtype=np.float64)


def forced_blocks(nb: int, init_blocks: int, local_blocks: int) -> list:
    """The blocks a row always keeps: its first init_blocks and last
    local_blocks, from the row's own block count (sglang #42614, Modifications 1)."""
    f = set(range(min(init_blocks, nb)))
    f |= set(range(max(0, nb - local_blocks), nb))
    return sorted(f)


def select_row(blockmax: np.ndarray, init_blocks: int, local_blocks: int, topk: int):
    """Block top-k of one row: the forced blocks plus the best remaining
    candidates by block max (ties to the lower id), padded to topk.
    Returns (ids int64 [topk], scores float64 [topk])."""
    nb = len(blockmax)
    forced = forced_blocks(nb, init_blocks, local_blocks)
    assert len(forced) <= topk, "forced blocks exceed topk"
    fset = set(forced)
    cands = [b for b in range(nb) if b not in fset]
    cands.sort(key=lambda b: (-blockmax[b], b))
    take = max(0, min(topk, nb) - len(forced))
    chosen = forced + cands[:take]
    ids = np.full(topk, -1, dtype=np.int64)
    scores = np.full(topk, -np.inf, dtype=np.float64)
    ids[:len(chosen)] = chosen
    scores[:len(chosen)] = [blockmax[b] for b in chosen]
    return ids, scores


def shard_select(blockmax: np.ndarray, b0: int, b1: int, init_blocks: int, local_blocks: int,
                 topk: int):
    """What one context shard of a row contributes (indexer context parallelism:
    sglang #42614 names the per-shard scorer score_local_blocks; reading: rank w
    holds the row's blocks [b0, b1) and scores only those).  ``blockmax`` is the
    row's whole block-score vector; only [b0, b1) of it is used.  The forced set
    and the number c of candidates to choose come from the row's global block
    count.  The shard emits its forced blocks (ascending), then its best
    min(c, its candidates) candidates by (score desc, id asc), then (-1, -inf)
    pads.  Returns (ids int64 [topk], scores float64 [topk])."""
    nb = len(blockmax)
    forced = forced_blocks(nb, init_blocks, local_blocks)
    fset = set(forced)
    c = max(0, min(topk, nb) - len(forced))
    lo, hi = max(0, b0), min(nb, b1)
    mine_f = [b for b in forced if lo <= b < hi]
    cands = [b for b in range(lo, hi) if b not in fset]
    cands.sort(key=lambda b: (-blockmax[b], b))
    chosen = mine_f + cands[:c]
    ids = np.full(topk, -1, dtype=np.int64)
    scores = np.full(topk, -np.inf, dtype=np.float64)
    ids[:len(chosen)] = chosen
    scores[:len(chosen)] = [blockmax[b] for b in chosen]
    return ids, scores


def merge_shards(lists, nb: int, init_blocks: int, local_blocks: int, topk: int):
    """Re-select a row from its shards' lists (the exchange step of indexer
    context parallelism): the forced blocks of the row's global block count,
    ascending, with the scores their shard reported, then the best c of all the
    shards' other entries by (score desc, id asc), then pads.  ``lists`` is a
    sequence of (ids, scores) as shard_select returns them."""
    forced = forced_blocks(nb, init_blocks, local_blocks)
    fset = set(forced)
    c = max(0, min(topk, nb) - len(forced))
    fscore = {}
    pool = []
    for ids, scores in lists:
        for b, v in zip(ids, scores):
            b = int(b)
            if b < 0:
                continue
            if b in fset:
                fscore[b] = v
            else:
                pool.append((b, v))
    pool.sort(key=lambda e: (-e[1], e[0]))
    chosen = [(b, fscore[b]) for b in forced] + pool[:c]
    ids = np.full(topk, -1, dtype=np.int64)
    scores = np.full(topk, -np.inf, dtype=np.float64)
    ids[:len(chosen)] = [b for b, _ in chosen]
    scores[:len(chosen)] = [v for _, v in chosen]
    return ids, scores


def request_slot(slot_ids, r: int) -> int:
    """The slot a request's keys live under (never its row or group index)."""
    return int(slot_ids[r])


def group_extent(lens) -> int:
    """Tokens of K a packed group needs: its longest row (rows of one group may
    straddle a block boundary; sglang #42614, Modifications 1)."""
    return max(lens)


def tile_row(i: int, gqa: int):
    """Packed tile row i -> (draft row i // gqa, head i % gqa)."""
    return i // gqa, i % gqa


@dataclasses.dataclass
class StepResult:
    ids: np.ndarray        # int64 [R, M, topk]
    scores: np.ndarray     # float64 [R, M, topk]
    blockmax: dict         # (r, i) -> float64 [nb] (rows with nb > 0 only)


def index_step(*, q, q_dtype, q_scale, payload, scale, k_dtype, page_table, slot_ids,
               row_lens, packed_queries, gqa, init_blocks, local_blocks, topk,
               requests=None, block_score="max") -> StepResult:
    """The whole step for every request (or only ``requests``; other requests'
    rows are left as pads in the result).  block_score: "max" (the block's
    largest score) or "lse" (its log-sum-exp); ``blockmax`` holds whichever.

    q: [R, P, G, 128] bf16 bits (uint16) or e4m3 codes (uint8); q_scale: [R, P*G]
    fp32 or None; payload/scale: pool planes (uint8 rows); page_table int
    [n_slots, max_pages]; slot_ids int [R]; row_lens int [R, P].
    """
    q = np.asarray(q)
    R = q.shape[0]
    P, G = packed_queries, gqa
    M = P * G
    n_slots, max_pages = page_table.shape
    ids = np.full((R, M, topk), -1, dtype=np.int64)
    scores = np.full((R, M, topk), -np.inf, dtype=np.float64)
    blockmax = {}
    todo = range(R) if requests is None else requests
    for r in todo:
        slot = request_slot(slot_ids, r)
        if slot < 0 or slot >= n_slots:            # graph padding: no reads
            continue
        lens = [int(x) for x in row_lens[r]]
        extent = group_extent(lens)
        if extent <= 0:
            continue
        assert extent <= max_pages * PAGE, "row longer than the page table"
        keys = dequant_keys(k_dtype, payload, scale, key_rows(page_table, slot, extent))
        for i in range(M):
            j, h = tile_row(i, G)
            L = lens[j]
            if L <= 0:
                continue
            qs = None if q_scale is None else q_scale[r, i]
            qv = dequant_query(q_dtype, q[r, j, h], qs)
            if block_score == "max":
                bm = row_block_max(qv, keys, L)
            elif block_score == "lse":
                bm = row_block_lse(qv, keys, L)
            else:
                raise ValueError(block_score)
            blockmax[(r, i)] = bm
            ids[r, i], scores[r, i] = select_row(bm, init_blocks, local_blocks, topk)
    return StepResult(ids=ids, scores=scores, blockmax=blockmax)

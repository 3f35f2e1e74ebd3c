"""Indexer context parallelism on one GPU (needs a GPU): each request's context
is cut into W contiguous shards, every shard is scored with
idx_score_local_blocks through its own slice of the page table (as the rank
holding it would), and idx_topk_merge combines the lists.  The merged result
must equal idx_score_topk over the whole context bit for bit (same block sums,
same selection), and each shard's list must match the oracle's shard_select."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _util import near_tie_violation, oracle_kwargs, score_tol
import _gpu
import sparse_attention_indexer_packed_gb300 as idx

pytestmark = pytest.mark.gpu


def _shards(b, planes, S, dev="cuda"):
    s = b.spec
    pt = b.page_table
    W = -(-pt.shape[1] // (2 * S))
    pad = W * 2 * S - pt.shape[1]
    if pad:
        pt = torch.cat([pt, pt[:, :1].repeat(1, pad)], dim=1)   # never read: past every row
    payload, scale = planes
    q = b.q.to(dev)
    qs = None if b.q_scale is None else b.q_scale.to(dev)
    sl, ln = b.slot_ids.to(dev), b.row_lens.to(dev)
    ids = torch.empty((W, b.R, b.M, s.topk), dtype=torch.int32, device=dev)
    sc = torch.empty((W, b.R, b.M, s.topk), dtype=torch.float32, device=dev)
    ws = idx.alloc_workspace(b.R, s.packed_queries, s.gqa, 2 * S, device=dev)
    for w in range(W):
        ptw = pt[:, 2 * S * w:2 * S * (w + 1)].contiguous().to(dev)
        idx.idx_score_local_blocks(q, qs, payload, scale, s.k_dtype, ptw, S * w, sl, ln,
                                   s.packed_queries, s.gqa, s.init_blocks, s.local_blocks,
                                   s.topk, ids[w], sc[w], ws)
        assert idx.idx_workspace_errors(ws) == 0
    out_ids = torch.empty((b.R, b.M, s.topk), dtype=torch.int32, device=dev)
    out_sc = torch.empty((b.R, b.M, s.topk), dtype=torch.float32, device=dev)
    idx.idx_topk_merge(ids, sc, sl, ln, b.n_slots, s.packed_queries, s.gqa, s.init_blocks,
                       s.local_blocks, s.topk, out_ids, out_sc)
    torch.cuda.synchronize()
    return W, ids.cpu().numpy(), sc.cpu().numpy(), out_ids.cpu().numpy(), out_sc.cpu().numpy()


@pytest.mark.parametrize("k_dtype,q_dtype", [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"),
                                             ("nvfp4", "bf16")])
@pytest.mark.parametrize("S", [8, 24])
def test_shards_merge_to_the_whole_context(k_dtype, q_dtype, S):
    spec = workloads.small_spec("cp", 601, k_dtype, q_dtype, R=5, len_range=(1, 9000),
                                pad_requests=(2,), topk=16, init_blocks=1, local_blocks=3)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    whole = _gpu.run(b, planes=planes)
    W, sh_ids, sh_sc, m_ids, m_sc = _shards(b, planes, S)
    assert W >= 3
    assert np.array_equal(m_ids, whole.ids)
    assert np.array_equal(m_sc.view(np.uint32), whole.scores.view(np.uint32))
    # every shard's own list against the oracle's reading of it
    ref = oracle.index.index_step(**oracle_kwargs(b))
    for (r, i), bm in ref.blockmax.items():
        for w in range(W):
            want_ids, want_sc = oracle.index.shard_select(bm, w * S, (w + 1) * S,
                                                          spec.init_blocks, spec.local_blocks,
                                                          spec.topk)
            n = int((want_ids >= 0).sum())
            assert int((sh_ids[w, r, i] >= 0).sum()) == n, (r, i, w)
            got = sh_ids[w, r, i, :n]
            # forced part exact; chosen part equal as a set up to near ties: the
            # shard's own k-th and (k+1)-th candidates within tolerance
            assert np.all(np.abs(sh_sc[w, r, i, :n] - bm[got]) <= score_tol(bm[got]))
            want = set(want_ids[:n].tolist())
            if set(got.tolist()) != want:
                nb = len(bm)
                forced = set(oracle.index.forced_blocks(nb, spec.init_blocks, spec.local_blocks))
                cands = [x for x in range(w * S, min(nb, (w + 1) * S)) if x not in forced]
                c = n - len(forced & want)
                err = near_tie_violation(bm, cands, c, set(got.tolist()) ^ want)
                assert err is None, (r, i, w, err)


def test_merge_of_one_shard_is_the_shard():
    """world = 1 with the whole context as the shard: the merge returns the list."""
    spec = workloads.small_spec("cp1", 602, "bf16", "bf16", R=3, len_range=(1, 4000), topk=8)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    whole = _gpu.run(b, planes=planes)
    S = -(-b.page_table.shape[1] // 2)
    W, _, _, m_ids, m_sc = _shards(b, planes, S)
    assert W == 1
    assert np.array_equal(m_ids, whole.ids)
    assert np.array_equal(m_sc.view(np.uint32), whole.scores.view(np.uint32))

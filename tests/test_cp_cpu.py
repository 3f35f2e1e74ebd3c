"""Indexer context parallelism on CPU ranks (gloo, world size 2): each rank
holds one contiguous shard of every request's blocks, computes its shard's lists
(here with the oracle: the CUDA scorer needs a GPU), and the package's exchange
(cp.gather_shard_lists) gathers them in rank order; the merge of the gathered
lists must equal the single-device selection on every row."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard_lists(rank, world):
    """Every rank's lists for the same seeded batch; shard w holds blocks
    [w * S, (w + 1) * S) of every request."""
    import oracle
    import workloads
    from _util import oracle_kwargs
    spec = workloads.small_spec("cpx", 611, "bf16", "bf16", R=3, len_range=(1, 5000),
                                pad_requests=(1,), topk=12, init_blocks=1, local_blocks=2)
    b = workloads.make_batch(spec)
    ref = oracle.index.index_step(**oracle_kwargs(b))
    nb_max = (int(b.row_lens.max()) + 127) // 128
    S = -(-nb_max // world)
    ids = np.full((world, b.R, b.M, spec.topk), -1, np.int32)
    sc = np.full((world, b.R, b.M, spec.topk), -np.inf, np.float32)
    for (r, i), bm in ref.blockmax.items():
        for w in range(world):
            li, ls_ = oracle.index.shard_select(bm, w * S, (w + 1) * S, spec.init_blocks,
                                                spec.local_blocks, spec.topk)
            ids[w, r, i] = li
            sc[w, r, i] = ls_
    return b, spec, ref, ids, sc


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import oracle
    from sparse_attention_indexer_packed_gb300 import cp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b, spec, ref, ids, sc = _shard_lists(rank, world)
        g_ids, g_sc = cp.gather_shard_lists(torch.from_numpy(ids[rank]), torch.from_numpy(sc[rank]))
        assert tuple(g_ids.shape) == (world, b.R, b.M, spec.topk)
        assert np.array_equal(g_ids.numpy(), ids)          # rank order, every shard intact
        assert np.array_equal(g_sc.numpy(), sc)
        bad = 0
        for r in range(b.R):
            for i in range(b.M):
                bm = ref.blockmax.get((r, i))
                if bm is None:
                    assert (g_ids[:, r, i] == -1).all()    # pad request / empty row
                    continue
                lists = [(g_ids[w, r, i].numpy(), g_sc[w, r, i].numpy().astype(np.float64))
                         for w in range(world)]
                m_ids, m_sc = oracle.index.merge_shards(lists, len(bm), spec.init_blocks,
                                                        spec.local_blocks, spec.topk)
                bad += int(m_ids.tolist() != ref.ids[r, i].tolist())
                # the lists carry fp32 scores; pads are -inf on both sides
                want = ref.scores[r, i].astype(np.float32).astype(np.float64)
                bad += int(not np.array_equal(m_sc, want))
        out[rank] = bad
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks_exchange_and_merge():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    assert out[0] == 0 and out[1] == 0

"""Requests of more than 16 packed rows (the 128-row tensor-core tiles) against the
fp64 oracle on the same seeded inputs (needs a GPU).

The oracle's definition is per row, so it is the same for 16 and for 512 rows of
a request; what changes on the GPU is the tiling (128-row tcgen05 tiles, a tile
boundary may cut a draft row's heads apart, the last tile of a request is
partial) and the prefill shape (P query tokens of a chunk, each with its own
length).  Same bar as the 16-row path: block scores within 1e-3 * (1 + |s|),
selections equal except at near ties (tests/_util.compare_row).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _util import compare_row, oracle_kwargs, score_tol
import _gpu
import sparse_attention_indexer_packed_gb300 as idx

pytestmark = pytest.mark.gpu


def _check(batch, out, ref):
    s = batch.spec
    worst = 0.0
    for (r, i), bm in ref.blockmax.items():
        got = out.blockmax[r * batch.M + i, :len(bm)].astype(np.float64)
        worst = max(worst, float((np.abs(got - bm) / score_tol(bm)).max()))
    assert worst <= 1.0, f"block score off by {worst:.3f} x tolerance"
    bad = []
    for r in range(batch.R):
        for i in range(batch.M):
            bm = ref.blockmax.get((r, i), np.zeros(0))
            err = compare_row(out.ids[r, i], out.scores[r, i], ref.ids[r, i], ref.scores[r, i],
                              bm, s.init_blocks, s.local_blocks)
            if err:
                bad.append(f"request {r} row {i}: {err}")
    assert not bad, "\n".join(bad[:20]) + f"\n({len(bad)} rows differ)"


CASES = []
for k_dtype, q_dtype in [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"), ("nvfp4", "bf16")]:
    for seed, R, (P, G), lens, pads, init, local, topk in [
        (401, 4, (8, 4), (1, 6000), (), 1, 2, 16),        # 32 rows: one partial tile
        (402, 3, (40, 4), (200, 5000), (1,), 1, 4, 32),   # 160 rows: two tiles, a pad request
        (403, 3, (50, 3), (1, 3000), (), 2, 2, 8),        # 150 rows: a tile cuts a draft row
        (404, 2, (256, 2), (4000, 4500), (), 1, 4, 64),   # prefill chunk: 256 query tokens
        (405, 3, (75, 4), (100, 6000), (0,), 1, 2, 16),   # 300 rows: a tile pair + a lone tile
        (406, 5, (8, 8), (1, 5000), (1, 2), 1, 2, 16),    # one tile a request, two pad requests
    ]:
        CASES.append(pytest.param(k_dtype, q_dtype, seed, R, P, G, lens, pads, init, local, topk,
                                  id=f"{k_dtype}-{seed}-P{P}G{G}"))


def _spec(k_dtype, q_dtype, seed, R, P, G, lens, pads, init, local, topk):
    return workloads.small_spec(f"w{seed}", seed, k_dtype, q_dtype, R=R, P=P, G=G,
                                init_blocks=init, local_blocks=local, topk=topk, len_range=lens,
                                pad_requests=pads)


@pytest.mark.parametrize("k_dtype,q_dtype,seed,R,P,G,lens,pads,init,local,topk", CASES)
def test_wide_parity(k_dtype, q_dtype, seed, R, P, G, lens, pads, init, local, topk):
    b = workloads.make_batch(_spec(k_dtype, q_dtype, seed, R, P, G, lens, pads, init, local, topk))
    out = _gpu.run(b)
    assert out.flags == 0
    _check(b, out, oracle.index.index_step(**oracle_kwargs(b)))


@pytest.mark.parametrize("k_dtype,q_dtype", [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"),
                                             ("nvfp4", "bf16")])
def test_wide_lse_parity(k_dtype, q_dtype):
    """Log-sum-exp block score (sglang #45451, Accuracy Tests) on the wide tiles."""
    b = workloads.make_batch(_spec(k_dtype, q_dtype, 411, 3, 40, 4, (1, 5000), (), 1, 2, 16))
    out = _gpu.run(b, block_score="lse")
    assert out.flags == 0
    _check(b, out, oracle.index.index_step(**oracle_kwargs(b), block_score="lse"))


@pytest.mark.parametrize("P,G", [(40, 4), (8, 8)])
@pytest.mark.parametrize("k_dtype,q_dtype", [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"),
                                             ("nvfp4", "bf16")])
def test_wide_results_do_not_depend_on_the_grid(k_dtype, q_dtype, P, G):
    """With 1, 3 and 7 CTAs every CTA walks through many tiles (query-tile
    reloads, key-stage and accumulator ring wrap-arounds); the scores are
    bit-identical to the full grid's, because each block's sums do not depend on
    who computes them.  P x G = 64 is one tile per request (each group a lone
    tile)."""
    b = workloads.make_batch(_spec(k_dtype, q_dtype, 421, 3, P, G, (1, 4000), (), 1, 2, 16))
    planes = _gpu.device_planes(b)
    full = _gpu.run(b, planes=planes)
    try:
        for lim in (1, 3, 7):
            idx.idx_set_grid_limit(lim)
            part = _gpu.run(b, planes=planes)
            assert part.flags == 0
            assert np.array_equal(part.ids, full.ids)
            assert np.array_equal(part.scores.view(np.uint32), full.scores.view(np.uint32))
    finally:
        idx.idx_set_grid_limit(0)


@pytest.mark.parametrize("k_dtype,q_dtype", [("bf16", "bf16"), ("nvfp4", "bf16")])
def test_prefill_extents_from_aligned_and_unaligned_lengths(k_dtype, q_dtype):
    """A prefill-shaped call's tile extents come from thousands of row lengths,
    which the ABI takes at any 4-byte alignment.  750 rows a request (not a
    multiple of 4), 3 heads a row (draft rows cut by tile and pair boundaries),
    empty rows among them: the lengths read from a 16-byte aligned array and
    from one that is not agree with the oracle and with each other bit for
    bit."""
    rng = np.random.default_rng(441)
    lens = []
    for r in range(3):
        x = rng.integers(1, 4200, size=250)
        x[rng.random(250) < 0.1] = 0
        lens.append([int(v) for v in x])
    spec = workloads.small_spec("w441", 441, k_dtype, q_dtype, R=3, P=250, G=3, init_blocks=1,
                                local_blocks=2, topk=16, explicit_lens=lens)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    aligned = _gpu.run(b, planes=planes)
    assert aligned.flags == 0
    _check(b, aligned, oracle.index.index_step(**oracle_kwargs(b)))
    dl = b.row_lens.to("cuda").reshape(-1)
    buf = torch.empty(dl.numel() + 1, dtype=dl.dtype, device="cuda")
    buf[1:] = dl
    shifted = buf[1:].view(b.row_lens.shape)
    assert shifted.data_ptr() % 16 != 0
    unaligned = _gpu.run(b, planes=planes, row_lens=shifted)
    assert unaligned.flags == 0
    assert np.array_equal(unaligned.ids, aligned.ids)
    assert np.array_equal(unaligned.scores.view(np.uint32), aligned.scores.view(np.uint32))


def test_most_rows_per_request():
    """IDX_MAX_ROWS_PER_REQUEST (32768) rows in one request: 4096 query tokens
    x 8 heads, 256 tiles in 128 pairs, rows from ~100 to 5000 tokens."""
    b = workloads.make_batch(_spec("bf16", "bf16", 431, 1, 4096, 8, (4200, 5000), (), 1, 4, 24))
    out = _gpu.run(b)
    assert out.flags == 0
    _check(b, out, oracle.index.index_step(**oracle_kwargs(b)))

"""The benchmark workloads at full size, in the launch configuration bench.py
times (needs a GPU): the four decode workloads on the 16-row path and the
verify / prefill workloads on the tensor-core path.

The oracle recomputes a few sampled requests one by one, and every request's
block scores on the first and last 64 blocks of each row; every row is also
checked through properties that hold at any size, using the block maxima the
score kernel left in the workspace: the forced blocks are present, the row
emits min(topk, nb) distinct blocks, every chosen candidate scores at least as
high as every unchosen one (ties allowed), and emitted scores equal the
workspace's block maxima.  For NVFP4 the stored bytes of the sampled requests
are compared bit for bit with the oracle's quantiser.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _util import compare_row, oracle_kwargs, oracle_planes, np_bits16, np_u8
import _gpu

pytestmark = pytest.mark.gpu

FULL = ["bf16_16x131k", "fp8_16x131k", "fp8_16x131k_local0", "fp8_32x524k", "nvfp4_64x150k",
        # more than 16 rows per request: the tensor-core path
        "verify_bf16_16x32k_p8g8", "prefill_bf16_4x32k_c512", "prefill_fp8_4x32k_c512",
        "prefill_nvfp4_4x32k_c512"]


def _row_invariants(batch, out):
    s = batch.spec
    bad = []
    lens = batch.group_lens()
    for r in range(batch.R):
        for i in range(batch.M):
            ids = out.ids[r, i]
            sc = out.scores[r, i]
            L = int(batch.row_lens[r, i // s.gqa]) if lens[r] > 0 else 0
            nb = (L + 127) // 128 if L > 0 else 0
            n = min(s.topk, nb)
            got = ids[:n]
            if np.any(ids[n:] != -1) or len(set(got.tolist())) != n or (n and (got.min() < 0 or got.max() >= nb)):
                bad.append((r, i, "ids"))
                continue
            if nb == 0:
                continue
            bm = out.blockmax[r * batch.M + i, :nb]
            forced = set(range(min(s.init_blocks, nb))) | set(range(max(0, nb - s.local_blocks), nb))
            if not forced <= set(got.tolist()):
                bad.append((r, i, "forced"))
                continue
            if not np.array_equal(sc[:n].view(np.uint32), bm[got].view(np.uint32)):
                bad.append((r, i, "scores"))
                continue
            chosen = [b for b in got.tolist() if b not in forced]
            rest = np.ones(nb, bool)
            rest[got] = False
            for f in forced:
                rest[f] = False
            if chosen and rest.any() and bm[chosen].min() < bm[rest].max():
                bad.append((r, i, "threshold"))
    assert not bad, bad[:10]


@pytest.mark.parametrize("name", FULL)
def test_fullsize_workload(name):
    spec = workloads.WORKLOADS[name]
    batch = workloads.make_batch(spec)
    out = _gpu.run(batch)
    assert out.flags == 0, hex(out.flags)
    _row_invariants(batch, out)
    # sampled requests against the oracle: the first, the last and one in between
    # (a prefill request is 2048 rows: the last one alone)
    sample = sorted({0, batch.R // 2, batch.R - 1}) if batch.M <= 64 else [batch.R - 1]
    planes = oracle_planes(batch, requests=sample)
    if spec.k_dtype == "nvfp4":
        rows = np.concatenate([batch.slot_mapping.numpy()[batch.staging_offsets[r]:
                                                          batch.staging_offsets[r] + batch.group_lens()[r]]
                               for r in sample])
        dev_pay = np_u8(out.payload[torch.from_numpy(rows).to(out.payload.device)].cpu())
        dev_sc = np_u8(out.scale[torch.from_numpy(rows).to(out.scale.device)].cpu())
        assert np.array_equal(dev_pay, planes[0][rows])
        assert np.array_equal(dev_sc, planes[1][rows])
    ref = oracle.index.index_step(**oracle_kwargs(batch, planes=planes), requests=sample)
    errs = []
    for r in sample:
        for i in range(batch.M):
            e = compare_row(out.ids[r, i], out.scores[r, i], ref.ids[r, i], ref.scores[r, i],
                            ref.blockmax.get((r, i), np.zeros(0)), spec.init_blocks, spec.local_blocks)
            if e:
                errs.append((r, i, e))
            bm = ref.blockmax.get((r, i))
            if bm is not None:
                got = out.blockmax[r * batch.M + i, :len(bm)].astype(np.float64)
                if np.any(np.abs(got - bm) > 1e-3 * (1 + np.abs(bm))):
                    errs.append((r, i, "block max"))
    assert not errs, errs[:10]
    _check_edges(batch, out)


EDGE_BLOCKS = 64


def _edge_keys(batch, r, t0, t1):
    """The oracle's dequantised keys of request r's tokens [t0, t1): read from the
    pool planes through the slot table, or for NVFP4 quantised by the oracle from
    the staged bf16 keys."""
    s = batch.spec
    if s.k_dtype == "nvfp4":
        off = batch.staging_offsets[r]
        bits = np_bits16(batch.staging[off + t0:off + t1])
        return oracle.formats.nvfp4_dequantize(*oracle.formats.nvfp4_quantize(bits))
    rows = oracle.index.key_rows(batch.page_table.numpy(), int(batch.slot_ids[r]), t1)[t0:]
    scale = None if batch.scale is None else np_u8(batch.scale[torch.from_numpy(rows)])
    return oracle.index.dequant_keys(s.k_dtype, np_u8(batch.payload[torch.from_numpy(rows)]),
                                     scale, np.arange(len(rows)))


def _check_edges(batch, out):
    """Every request against the oracle on the first and the last EDGE_BLOCKS
    blocks of each row: the block scores the kernel left in the workspace."""
    s = batch.spec
    lens = batch.group_lens()
    q = np_bits16(batch.q) if s.q_dtype == "bf16" else np_u8(batch.q)
    bad, checked = [], 0
    for r in range(batch.R):
        if lens[r] <= 0:
            continue
        ext = lens[r]
        nbx = (ext + 127) // 128
        head = min(nbx, EDGE_BLOCKS)
        tail0 = max(head, nbx - EDGE_BLOCKS)
        k_head = _edge_keys(batch, r, 0, min(ext, head * 128))
        k_tail = _edge_keys(batch, r, tail0 * 128, ext) if tail0 < nbx else None
        # every row of a decode or verify request; a prefill chunk's 2048 rows
        # every 37th and its last
        rows = range(batch.M) if batch.M <= 64 else sorted(set(range(0, batch.M, 37)) | {batch.M - 1})
        for i in rows:
            j, h = divmod(i, s.gqa)
            L = int(batch.row_lens[r, j])
            nb = (L + 127) // 128
            if nb <= 0:
                continue
            qs = None if batch.q_scale is None else float(batch.q_scale[r, i])
            qv = oracle.index.dequant_query(s.q_dtype, q[r, j, h], qs)
            got = out.blockmax[r * batch.M + i, :nb].astype(np.float64)
            want = oracle.index.row_block_max(qv, k_head, min(L, head * 128))
            ranges = [(0, want)]
            if k_tail is not None and L > tail0 * 128:
                ranges.append((tail0, oracle.index.row_block_max(qv, k_tail, L - tail0 * 128)))
            for b0, w in ranges:
                g = got[b0:b0 + len(w)]
                checked += len(w)
                if np.any(np.abs(g - w) > 1e-3 * (1 + np.abs(w))):
                    bad.append((r, i, b0))
    assert checked > 0
    assert not bad, bad[:10]

"""The benchmark workloads at full size, in the launch configuration bench.py
times (needs a GPU): the four decode workloads on the 16-row path and the
verify / prefill workloads on the tensor-core path.

The oracle recomputes a few sampled requests one by one; every other row is
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
from _util import compare_row, oracle_kwargs, oracle_planes, np_u8
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

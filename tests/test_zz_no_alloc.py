"""idx_score_topk_noalloc: the index step for callers that cannot allocate
device memory (an engine that owns every byte of device memory through its own
pool, a plugin with no allocator hook, a step that must not risk the device
synchronisation an allocation can cause).  It keeps its scratch in a fixed array
inside the library instead of a caller-provided workspace.

The test calls it through the C ABI twice in a row and checks each output
against the ordinary entry point's, within the tolerance the other parity tests
use.  This file is collected last, so a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
import sparse_attention_indexer_packed_gb300 as idx
from sparse_attention_indexer_packed_gb300 import _lib
from _util import score_tol
import _gpu

pytestmark = pytest.mark.gpu


def _ordinary(b, planes, dev):
    s = b.spec
    ids = torch.empty((b.R, b.M, s.topk), dtype=torch.int32, device=dev)
    sc = torch.empty((b.R, b.M, s.topk), dtype=torch.float32, device=dev)
    ws = idx.alloc_workspace(b.R, s.packed_queries, s.gqa, b.max_pages, device=dev)
    idx.idx_score_topk(b.q.to(dev), None if b.q_scale is None else b.q_scale.to(dev), planes[0],
                       planes[1], s.k_dtype, b.page_table.to(dev), b.slot_ids.to(dev),
                       b.row_lens.to(dev), s.packed_queries, s.gqa, s.init_blocks,
                       s.local_blocks, s.topk, ids, sc, ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy()


def _noalloc_via_c_abi(b, planes, dev, ids, sc):
    """Direct ctypes call of the C entry point (no Python wrapper in between)."""
    s = b.spec
    L = idx.lib()
    q = b.q.to(dev)
    qs = None if b.q_scale is None else b.q_scale.to(dev)
    pt = b.page_table.to(dev)
    sl = b.slot_ids.to(dev)
    rl = b.row_lens.to(dev)
    rc = L.idx_score_topk_noalloc(
        q.data_ptr(), None if qs is None else qs.data_ptr(),
        _lib.IDX_BF16 if s.q_dtype == "bf16" else _lib.IDX_FP8_E4M3,
        planes[0].data_ptr(), None if planes[1] is None else planes[1].data_ptr(),
        _lib.DTYPES[s.k_dtype], b.num_pages, pt.data_ptr(), b.n_slots, b.max_pages,
        sl.data_ptr(), rl.data_ptr(), b.R, s.packed_queries, s.gqa, s.init_blocks,
        s.local_blocks, s.topk, ids.data_ptr(), sc.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, L.idx_last_error()
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy()


def _same(a_ids, a_sc, b_ids, b_sc):
    assert np.array_equal(a_ids, b_ids)
    fin = np.isfinite(b_sc)
    assert np.array_equal(np.isfinite(a_sc), fin)
    assert np.all(np.abs(a_sc[fin].astype(np.float64) - b_sc[fin]) <= score_tol(b_sc[fin]))


@pytest.mark.parametrize("k_dtype,q_dtype,seed", [("bf16", "bf16", 701), ("fp8_e4m3", "fp8_e4m3", 702),
                                                  ("nvfp4", "bf16", 703)])
def test_noalloc_matches_the_workspace_entry_point_twice(k_dtype, q_dtype, seed):
    dev = "cuda"
    spec = workloads.small_spec(f"na{seed}", seed, k_dtype, q_dtype, R=6, len_range=(1, 20000),
                                topk=32, pad_requests=(4,))
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    ref_ids, ref_sc = _ordinary(b, planes, dev)
    ids = torch.full((b.R, b.M, spec.topk), -7, dtype=torch.int32, device=dev)
    sc = torch.full((b.R, b.M, spec.topk), 123.0, dtype=torch.float32, device=dev)
    # two calls in a row on the shared scratch: the second must not see the first
    for _ in range(2):
        got_ids, got_sc = _noalloc_via_c_abi(b, planes, dev, ids, sc)
        _same(got_ids, got_sc, ref_ids, ref_sc)
        ids.fill_(-7)
        sc.fill_(123.0)


def _pair_twice(b, dev="cuda"):
    planes = _gpu.device_planes(b)
    ref_ids, ref_sc = _ordinary(b, planes, dev)
    s = b.spec
    ids = torch.full((b.R, b.M, s.topk), -7, dtype=torch.int32, device=dev)
    sc = torch.full((b.R, b.M, s.topk), 123.0, dtype=torch.float32, device=dev)
    for _ in range(2):
        got_ids, got_sc = _noalloc_via_c_abi(b, planes, dev, ids, sc)
        _same(got_ids, got_sc, ref_ids, ref_sc)
        assert idx.idx_noalloc_errors() == 0
        ids.fill_(-7)
        sc.fill_(123.0)


def test_noalloc_wide_tiles():
    """More than 16 packed rows (8 draft rows x 8 heads): the tensor-core path on
    the shared scratch."""
    spec = workloads.small_spec("naw", 711, "bf16", "bf16", R=5, P=8, G=8, len_range=(1, 12000),
                                topk=32, pad_requests=(1,))
    _pair_twice(workloads.make_batch(spec))


def test_noalloc_dynamic_schedule():
    """Enough blocks per CTA (16 requests of up to 80K tokens, ~60 blocks per SM)
    that, from the second call on, part of the blocks is handed out at run time
    through the counter in the scratch header."""
    spec = workloads.small_spec("nad", 712, "bf16", "bf16", R=16, len_range=(60000, 80000),
                                topk=64, init_blocks=1, local_blocks=4)
    _pair_twice(workloads.make_batch(spec))


def test_noalloc_near_the_scratch_limit():
    """A page table wide enough that the call needs all but a few KB of the
    16 MiB array; the last request is long, so its block scores sit at the
    array's far end."""
    spec = workloads.small_spec("nam", 713, "bf16", "bf16", R=64, len_range=(1, 3000), topk=16)
    b = workloads.make_batch(spec)
    b.row_lens[-1] = torch.arange(4, dtype=torch.int32) + (300000 - 3)
    # rebuild the batch with the long last request and a table of 8190 pages
    spec = workloads.Spec(**{**spec.__dict__, "explicit_lens": b.row_lens.tolist(),
                             "len_range": None, "max_pages": 8190})
    b = workloads.make_batch(spec)
    need = idx.idx_score_topk_workspace_bytes(b.R, 4, 4, b.max_pages)
    assert (16 << 20) - 8192 < need <= (16 << 20)
    _pair_twice(b)


def test_noalloc_errors_report_a_timeout():
    """idx_noalloc_errors reads the flags of the last no-allocation call: a call
    whose waits run out (the stall test, 20 ms limit) reports IDX_DEVERR_TIMEOUT,
    and the next normal call reports none."""
    spec = workloads.small_spec("nae", 714, "bf16", "bf16", R=4, len_range=(2000, 9000), topk=16)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    ids = torch.empty((b.R, b.M, spec.topk), dtype=torch.int32, device="cuda")
    sc = torch.empty((b.R, b.M, spec.topk), dtype=torch.float32, device="cuda")
    try:
        idx.idx_set_wait_limit_ns(20_000_000)
        idx.idx_set_stall_test(True)
        _noalloc_via_c_abi(b, planes, "cuda", ids, sc)
        assert idx.idx_noalloc_errors() & 2
    finally:
        idx.idx_set_stall_test(False)
        idx.idx_set_wait_limit_ns(0)
    ref_ids, ref_sc = _ordinary(b, planes, "cuda")
    got_ids, got_sc = _noalloc_via_c_abi(b, planes, "cuda", ids, sc)
    assert idx.idx_noalloc_errors() == 0
    _same(got_ids, got_sc, ref_ids, ref_sc)


def test_noalloc_refuses_calls_larger_than_its_scratch():
    L = idx.lib()
    limit = L.idx_score_topk_workspace_bytes(4096, 4, 4, 65536)
    assert limit > (16 << 20)
    fake = 0x10000
    rc = L.idx_score_topk_noalloc(fake, None, 0, fake, None, 0, 1 << 20, fake, 10, 65536, fake,
                                  fake, 4096, 4, 4, 1, 4, 64, fake, fake, None)
    assert rc == -1
    assert b"scratch" in L.idx_last_error()

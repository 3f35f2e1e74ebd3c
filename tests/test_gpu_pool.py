"""The library-owned pool (idx_pool_alloc / idx_pool_free) on the GPU: the planes
it allocates have the row sizes the store and the score kernels assume (ROCm/ATOM
#2745, Summary, "Pool and binding": payload and scale as separate planes), keys
stored or copied into them score exactly as from caller-owned planes, and
idx_pool_free releases them and zeroes the struct."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
import sparse_attention_indexer_packed_gb300 as idx
from sparse_attention_indexer_packed_gb300 import _lib
from _util import compare_row, oracle_kwargs
import _gpu

pytestmark = pytest.mark.gpu

ROW_BYTES = {"bf16": (256, 0), "fp8_e4m3": (128, 4), "nvfp4": (64, 8)}


class _DeviceBytes:
    """A view of library-owned device memory as a torch tensor (CUDA array
    interface; no copy, no ownership)."""

    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (int(ptr), False), "version": 3,
                                         "strides": None}


def _plane(ptr, rows, row_bytes):
    t = torch.as_tensor(_DeviceBytes(ptr, rows * row_bytes), device="cuda")
    assert t.data_ptr() == int(ptr)
    return t.view(rows, row_bytes)


@pytest.mark.parametrize("k_dtype,q_dtype,seed", [("bf16", "bf16", 801),
                                                  ("fp8_e4m3", "fp8_e4m3", 802),
                                                  ("nvfp4", "bf16", 803)])
def test_library_pool_stores_and_scores(k_dtype, q_dtype, seed):
    spec = workloads.small_spec(f"pool{seed}", seed, k_dtype, q_dtype, R=5, len_range=(1, 9000),
                                topk=24, pad_requests=(3,))
    b = workloads.make_batch(spec)
    pool = idx.idx_pool_alloc(k_dtype, b.num_pages)
    try:
        pb, sb = ROW_BYTES[k_dtype]
        assert (pool.dtype, pool.page_size, pool.dim) == (_lib.DTYPES[k_dtype], 64, 128)
        assert pool.num_pages == b.num_pages
        assert (pool.payload_row_bytes, pool.scale_row_bytes) == (pb, sb)
        assert pool.payload and (pool.scale is None) == (sb == 0)
        assert pool.payload % 256 == 0 and (not pool.scale or pool.scale % 256 == 0)
        rows = b.num_pages * 64
        payload = _plane(pool.payload, rows, pb)
        scale = _plane(pool.scale, rows, sb) if sb else None
        # the batch's bytes into the library's planes; NVFP4 keys through the store
        payload.copy_(b.payload.cuda())
        if scale is not None:
            scale.copy_(b.scale.cuda())
        if k_dtype == "nvfp4":
            idx.idx_store_nvfp4(b.staging.cuda(), b.slot_mapping.cuda(), pool)
        torch.cuda.synchronize()
        out = _gpu.run(b, planes=(payload, scale))
        assert out.flags == 0
        # the same call on caller-owned planes gives the same bits
        ref_planes = _gpu.device_planes(b)
        if k_dtype == "nvfp4":
            assert torch.equal(payload, ref_planes[0]) and torch.equal(scale, ref_planes[1])
        own = _gpu.run(b, planes=ref_planes)
        assert np.array_equal(out.ids, own.ids)
        assert np.array_equal(out.scores.view(np.uint32), own.scores.view(np.uint32))
        ref = oracle.index.index_step(**oracle_kwargs(b))
        bad = [(r, i) for r in range(b.R) for i in range(b.M)
               if compare_row(out.ids[r, i], out.scores[r, i], ref.ids[r, i], ref.scores[r, i],
                              ref.blockmax.get((r, i), np.zeros(0)), spec.init_blocks,
                              spec.local_blocks)]
        assert not bad, bad[:10]
        del payload, scale
    finally:
        idx.idx_pool_free(pool)
    assert (pool.dtype, pool.num_pages, pool.payload, pool.scale,
            pool.payload_row_bytes, pool.scale_row_bytes) == (0, 0, None, None, 0, 0)


def test_pool_alloc_refuses_bad_arguments_and_oom():
    L = idx.lib()
    p = _lib.IdxPool()
    assert L.idx_pool_alloc(7, 10, 64, 128, ctypes.byref(p)) == -1
    assert L.idx_pool_alloc(0, 10, 32, 128, ctypes.byref(p)) == -1
    assert L.idx_pool_alloc(0, 0, 64, 128, ctypes.byref(p)) == -1
    assert L.idx_pool_alloc(0, 1 << 25, 64, 128, ctypes.byref(p)) == -1   # 2^31 rows
    # a plane of ~550 GB, twice what the GPU holds: cudaMalloc refuses it and the
    # call reports IDX_ERR_OOM with nothing allocated
    assert L.idx_pool_alloc(0, (1 << 31) // 64 - 1, 64, 128, ctypes.byref(p)) == -4
    assert not p.payload and not p.scale
    # the context is still usable
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0

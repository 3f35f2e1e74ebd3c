"""GB300 (sm_103a) packed index-score + block top-k for sparse-attention decode.

The compute path is libidx.so (CUDA kernels behind a C ABI, include/idx.h); this
package is its thin ctypes binding.  See ``_lib`` for the functions.
"""
from ._lib import (  # noqa: F401
    DTYPES, IDX_BF16, IDX_FP8_E4M3, IDX_NVFP4, IdxError, IdxPool, abi_version, alloc_workspace,
    idx_noalloc_errors, idx_pool_alloc, idx_pool_free, idx_score_local_blocks, idx_score_topk,
    idx_score_topk_lse, idx_score_topk_noalloc, idx_score_topk_perrow, idx_score_topk_workspace_bytes,
    idx_set_grid_limit, idx_set_kernel_events, idx_set_kernel_waits, idx_set_stall_test, idx_set_wait_limit_ns,
    idx_store_nvfp4,
    idx_topk_merge,
    idx_workspace_errors, lib, pool_struct,
)
from . import cp  # noqa: F401,E402

"""ctypes binding of libidx (include/idx.h): argument marshalling only.

Every function here forwards to the C ABI of the same name with the device
pointers of the torch tensors it is given; all arithmetic runs in the library's
CUDA kernels.  There is no CPU path: a tensor that is not on a CUDA device, or a
missing libidx.so, raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libidx.so")

IDX_BF16, IDX_FP8_E4M3, IDX_NVFP4 = 0, 1, 2
IDX_OK = 0
PAGE, BLOCK, DIM = 64, 128, 128
WORKSPACE_HEADER_BYTES = 1024
DEVERR_BAD_PAGE, DEVERR_TIMEOUT, DEVERR_LEN_CLAMPED = 1, 2, 4

DTYPES = {"bf16": IDX_BF16, "fp8_e4m3": IDX_FP8_E4M3, "nvfp4": IDX_NVFP4}


class IdxPool(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("dim", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("payload", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("payload_row_bytes", ctypes.c_int64),
                ("scale_row_bytes", ctypes.c_int64)]


class IdxError(RuntimeError):
    pass


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "idx_abi_version": (_I, []),
    "idx_status_string": (ctypes.c_char_p, [_I]),
    "idx_last_error": (ctypes.c_char_p, []),
    "idx_pool_alloc": (_I, [_I, _I64, _I, _I, ctypes.POINTER(IdxPool)]),
    "idx_pool_free": (_I, [ctypes.POINTER(IdxPool)]),
    "idx_store_nvfp4": (_I, [_P, _P, _I64, ctypes.POINTER(IdxPool), _P]),
    "idx_score_topk_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "idx_score_topk": (_I, [_P, _P, _I, _P, _P, _I, _I64, _P, _I, _I, _P, _P, _I, _I, _I,
                            _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "idx_score_topk_lse": (_I, [_P, _P, _I, _P, _P, _I, _I64, _P, _I, _I, _P, _P, _I, _I, _I,
                                _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "idx_score_topk_perrow": (_I, [_P, _P, _I, _P, _P, _I, _I64, _P, _I, _I, _P, _P, _I, _I,
                                   _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "idx_score_local_blocks": (_I, [_P, _P, _I, _P, _P, _I, _I64, _P, _I, _I, _I, _P, _P, _I,
                                    _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "idx_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "idx_set_stall_test": (_I, [_I]),
    "idx_topk_merge": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "idx_score_topk_noalloc": (_I, [_P, _P, _I, _P, _P, _I, _I64, _P, _I, _I, _P, _P, _I, _I,
                                    _I, _I, _I, _I, _P, _P, _P]),
    "idx_set_kernel_events": (_I, [_P, _P, _P]),
    "idx_set_kernel_waits": (_I, [_P, _P]),
    "idx_set_grid_limit": (_I, [_I]),
    "idx_workspace_errors": (_I, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
    "idx_noalloc_errors": (_I, [_P, ctypes.POINTER(ctypes.c_uint32)]),
}


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise IdxError(f"{LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != IDX_OK:
        msg = lib().idx_last_error().decode()
        name = lib().idx_status_string(rc).decode()
        raise IdxError(f"{what} failed: {name}: {msg}")


def _dev(t: Optional[torch.Tensor], name: str, required: bool = True) -> Optional[int]:
    if t is None:
        if required:
            raise IdxError(f"{name} is required")
        return None
    if not t.is_cuda:
        raise IdxError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise IdxError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def pool_struct(dtype: str, payload: torch.Tensor, scale: Optional[torch.Tensor]) -> IdxPool:
    """Describe caller-owned planes (torch tensors) as an idx_pool."""
    rows, row_bytes = payload.shape[0], payload.shape[1] * payload.element_size()
    p = IdxPool()
    p.dtype = DTYPES[dtype]
    p.page_size = PAGE
    p.dim = DIM
    p.num_pages = rows // PAGE
    p.payload = _dev(payload, "payload")
    p.scale = _dev(scale, "scale", required=False)
    p.payload_row_bytes = row_bytes
    p.scale_row_bytes = 0 if scale is None else scale.shape[1] * scale.element_size()
    return p


def abi_version() -> int:
    return lib().idx_abi_version()


def idx_pool_alloc(dtype: str, num_pages: int) -> IdxPool:
    p = IdxPool()
    _check(lib().idx_pool_alloc(DTYPES[dtype], num_pages, PAGE, DIM, ctypes.byref(p)),
           "idx_pool_alloc")
    return p


def idx_pool_free(pool: IdxPool) -> None:
    _check(lib().idx_pool_free(ctypes.byref(pool)), "idx_pool_free")


def idx_store_nvfp4(src_bf16: torch.Tensor, slot_mapping: torch.Tensor, pool, stream=None) -> None:
    """pool: an IdxPool, or a (payload, scale) pair of uint8 tensors."""
    if isinstance(pool, tuple):
        pool = pool_struct("nvfp4", pool[0], pool[1])
    if src_bf16.dtype != torch.bfloat16 or slot_mapping.dtype != torch.int64:
        raise IdxError("src_bf16 must be bfloat16 and slot_mapping int64")
    n = int(slot_mapping.numel())
    _check(lib().idx_store_nvfp4(_dev(src_bf16, "src_bf16"), _dev(slot_mapping, "slot_mapping"),
                                 n, ctypes.byref(pool), _stream_ptr(stream)), "idx_store_nvfp4")


def idx_score_topk_workspace_bytes(num_requests: int, packed_queries: int, gqa: int,
                                   max_pages: int) -> int:
    return int(lib().idx_score_topk_workspace_bytes(num_requests, packed_queries, gqa, max_pages))


def alloc_workspace(num_requests: int, packed_queries: int, gqa: int, max_pages: int,
                    device="cuda") -> torch.Tensor:
    n = idx_score_topk_workspace_bytes(num_requests, packed_queries, gqa, max_pages)
    return torch.empty(max(n, WORKSPACE_HEADER_BYTES), dtype=torch.uint8, device=device)


def _q_dtype(q: torch.Tensor) -> int:
    if q.dtype == torch.bfloat16:
        return IDX_BF16
    if q.dtype in (torch.uint8, torch.float8_e4m3fn):
        return IDX_FP8_E4M3
    raise IdxError(f"unsupported q dtype {q.dtype}")


def _score(fn_name: str, q, q_scale, k_payload, k_scale, k_dtype: str, page_table, slot_ids,
           row_lens, packed_queries, gqa, init_blocks, local_blocks, topk, out_ids, out_scores,
           workspace, stream):
    R = int(q.shape[0])
    num_pages = int(k_payload.shape[0]) // PAGE
    n_slots, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
    for t, name, dt in [(page_table, "page_table", torch.int32), (slot_ids, "slot_ids", torch.int32),
                        (row_lens, "row_lens", torch.int32), (out_ids, "out_ids", torch.int32),
                        (out_scores, "out_scores", torch.float32)]:
        if t.dtype != dt:
            raise IdxError(f"{name} must be {dt}")
    fn = getattr(lib(), fn_name)
    rc = fn(_dev(q, "q"), _dev(q_scale, "q_scale", required=False), _q_dtype(q),
            _dev(k_payload, "k_payload"), _dev(k_scale, "k_scale", required=False),
            DTYPES[k_dtype], num_pages, _dev(page_table, "page_table"), n_slots, max_pages,
            _dev(slot_ids, "slot_ids"), _dev(row_lens, "row_lens"), R, packed_queries, gqa,
            init_blocks, local_blocks, topk, _dev(out_ids, "out_ids"),
            _dev(out_scores, "out_scores"), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(rc, fn_name)


def idx_score_topk(q, q_scale, k_payload, k_scale, k_dtype, page_table, slot_ids, row_lens,
                   packed_queries, gqa, init_blocks, local_blocks, topk, out_ids, out_scores,
                   workspace, stream=None) -> None:
    _score("idx_score_topk", q, q_scale, k_payload, k_scale, k_dtype, page_table, slot_ids,
           row_lens, packed_queries, gqa, init_blocks, local_blocks, topk, out_ids, out_scores,
           workspace, stream)


def idx_score_topk_lse(q, q_scale, k_payload, k_scale, k_dtype, page_table, slot_ids, row_lens,
                       packed_queries, gqa, init_blocks, local_blocks, topk, out_ids, out_scores,
                       workspace, stream=None) -> None:
    _score("idx_score_topk_lse", q, q_scale, k_payload, k_scale, k_dtype, page_table, slot_ids,
           row_lens, packed_queries, gqa, init_blocks, local_blocks, topk, out_ids, out_scores,
           workspace, stream)


def idx_score_topk_perrow(q, q_scale, k_payload, k_scale, k_dtype, page_table, slot_ids, row_lens,
                          packed_queries, gqa, init_blocks, local_blocks, topk, out_ids,
                          out_scores, workspace, stream=None) -> None:
    _score("idx_score_topk_perrow", q, q_scale, k_payload, k_scale, k_dtype, page_table, slot_ids,
           row_lens, packed_queries, gqa, init_blocks, local_blocks, topk, out_ids, out_scores,
           workspace, stream)


def idx_score_local_blocks(q, q_scale, k_payload, k_scale, k_dtype, page_table, block_begin,
                           slot_ids, row_lens, packed_queries, gqa, init_blocks, local_blocks,
                           topk, out_ids, out_scores, workspace, stream=None) -> None:
    """One context shard: page_table [n_slots, max_pages] covers global blocks
    [block_begin, block_begin + max_pages / 2) of every request."""
    R = int(q.shape[0])
    num_pages = int(k_payload.shape[0]) // PAGE
    n_slots, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
    for t, name, dt in [(page_table, "page_table", torch.int32), (slot_ids, "slot_ids", torch.int32),
                        (row_lens, "row_lens", torch.int32), (out_ids, "out_ids", torch.int32),
                        (out_scores, "out_scores", torch.float32)]:
        if t.dtype != dt:
            raise IdxError(f"{name} must be {dt}")
    rc = lib().idx_score_local_blocks(
        _dev(q, "q"), _dev(q_scale, "q_scale", required=False), _q_dtype(q),
        _dev(k_payload, "k_payload"), _dev(k_scale, "k_scale", required=False), DTYPES[k_dtype],
        num_pages, _dev(page_table, "page_table"), n_slots, max_pages, int(block_begin),
        _dev(slot_ids, "slot_ids"), _dev(row_lens, "row_lens"), R, packed_queries, gqa,
        init_blocks, local_blocks, topk, _dev(out_ids, "out_ids"), _dev(out_scores, "out_scores"),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(rc, "idx_score_local_blocks")


def idx_topk_merge(cand_ids, cand_scores, slot_ids, row_lens, n_slots, packed_queries, gqa,
                   init_blocks, local_blocks, topk, out_ids, out_scores, stream=None) -> None:
    """cand_ids / cand_scores: [world, R, P*G, topk], the shards' lists."""
    world, R = int(cand_ids.shape[0]), int(cand_ids.shape[1])
    for t, name, dt in [(cand_ids, "cand_ids", torch.int32), (cand_scores, "cand_scores", torch.float32),
                        (slot_ids, "slot_ids", torch.int32), (row_lens, "row_lens", torch.int32),
                        (out_ids, "out_ids", torch.int32), (out_scores, "out_scores", torch.float32)]:
        if t.dtype != dt:
            raise IdxError(f"{name} must be {dt}")
    rc = lib().idx_topk_merge(_dev(cand_ids, "cand_ids"), _dev(cand_scores, "cand_scores"), world,
                              _dev(slot_ids, "slot_ids"), _dev(row_lens, "row_lens"), int(n_slots),
                              R, packed_queries, gqa, init_blocks, local_blocks, topk,
                              _dev(out_ids, "out_ids"), _dev(out_scores, "out_scores"),
                              _stream_ptr(stream))
    _check(rc, "idx_topk_merge")


def idx_set_wait_limit_ns(ns: int) -> None:
    """Limit of the score kernels' pipeline waits (0: the default 2 s)."""
    _check(lib().idx_set_wait_limit_ns(int(ns)), "idx_set_wait_limit_ns")


def idx_set_stall_test(on: bool) -> None:
    """Diagnostic: one role per score CTA waits on a barrier nothing completes."""
    _check(lib().idx_set_stall_test(1 if on else 0), "idx_set_stall_test")


def idx_set_kernel_events(score_begin=None, score_end=None, topk_end=None) -> None:
    """Arm torch.cuda.Event objects (enable_timing=True) for the next score call."""
    h = [None if e is None else e.cuda_event for e in (score_begin, score_end, topk_end)]
    _check(lib().idx_set_kernel_events(*h), "idx_set_kernel_events")


def idx_set_kernel_waits(before_score=None, before_topk=None) -> None:
    """Arm torch.cuda.Event objects the next score call's stream waits for before
    its score kernel / its top-k kernel (include/idx.h: idx_set_kernel_waits)."""
    h = [None if e is None else e.cuda_event for e in (before_score, before_topk)]
    _check(lib().idx_set_kernel_waits(*h), "idx_set_kernel_waits")


def idx_score_topk_noalloc(q, q_scale, k_payload, k_scale, k_dtype, page_table, slot_ids,
                           row_lens, packed_queries, gqa, init_blocks, local_blocks, topk,
                           out_ids, out_scores, stream=None) -> None:
    """idx_score_topk with the library's fixed scratch array instead of a workspace,
    for callers that cannot allocate device memory (see include/idx.h)."""
    R = int(q.shape[0])
    n_slots, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
    rc = lib().idx_score_topk_noalloc(
        _dev(q, "q"), _dev(q_scale, "q_scale", required=False), _q_dtype(q),
        _dev(k_payload, "k_payload"), _dev(k_scale, "k_scale", required=False), DTYPES[k_dtype],
        int(k_payload.shape[0]) // PAGE, _dev(page_table, "page_table"), n_slots, max_pages,
        _dev(slot_ids, "slot_ids"), _dev(row_lens, "row_lens"), R, packed_queries, gqa,
        init_blocks, local_blocks, topk, _dev(out_ids, "out_ids"), _dev(out_scores, "out_scores"),
        _stream_ptr(stream))
    _check(rc, "idx_score_topk_noalloc")


def idx_set_grid_limit(max_ctas: int) -> None:
    """Cap the score kernel's grid (0 = one CTA per SM); results do not change."""
    _check(lib().idx_set_grid_limit(int(max_ctas)), "idx_set_grid_limit")


def idx_workspace_errors(workspace: torch.Tensor, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().idx_workspace_errors(_dev(workspace, "workspace"), _stream_ptr(stream),
                                      ctypes.byref(v)), "idx_workspace_errors")
    return int(v.value)


def idx_noalloc_errors(stream=None) -> int:
    """Device error flags of the last idx_score_topk_noalloc call on this device."""
    v = ctypes.c_uint32(0)
    _check(lib().idx_noalloc_errors(_stream_ptr(stream), ctypes.byref(v)), "idx_noalloc_errors")
    return int(v.value)

"""The C ABI library loads without a GPU, exports every symbol include/idx.h
declares, and rejects bad arguments on the host (no compute call runs here)."""
import ctypes
import os
import re

import pytest

import sparse_attention_indexer_packed_gb300 as idx
from sparse_attention_indexer_packed_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "idx.h")).read()
    return sorted(set(re.findall(r"IDX_API\s+[\w\s\*]+?\b(idx_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return idx.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "idx_score_topk" in names and "idx_store_nvfp4" in names and "idx_pool_alloc" in names
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib._SIGNATURES), set(names) ^ set(_lib._SIGNATURES)


def test_version_and_status_strings(L):
    assert idx.abi_version() == 1
    assert L.idx_status_string(0) == b"IDX_OK"
    assert L.idx_status_string(-1) == b"IDX_ERR_INVALID"
    assert L.idx_status_string(-2) == b"IDX_ERR_UNSUPPORTED"


def test_workspace_bytes(L):
    assert idx.idx_score_topk_workspace_bytes(16, 4, 4, 2048) == 1024 + 16 * 16 * 1024 * 4
    assert idx.idx_score_topk_workspace_bytes(1, 1, 1, 3) == 1024 + 2 * 4
    assert idx.idx_score_topk_workspace_bytes(0, 4, 4, 10) == 1024
    # more than 16 packed rows: f16 query rows (256 B) and a scale (4 B) a row,
    # from the 256-byte boundary after the block scores
    rows, blocks = 4 * 512 * 4, 256
    after = (1024 + rows * blocks * 4 + 255) // 256 * 256
    assert idx.idx_score_topk_workspace_bytes(4, 512, 4, 512) == after + rows * 260
    assert idx.idx_score_topk_workspace_bytes(1, 17, 1, 3) == (1024 + 17 * 2 * 4 + 255) // 256 * 256 + 17 * 260


FAKE = 0x10000  # a non-NULL, 256-aligned value; every case below fails validation first


def _call(L, **over):
    a = dict(q=FAKE, q_scale=None, q_dtype=0, k_payload=FAKE, k_scale=None, k_dtype=0,
             num_pages=100, page_table=FAKE, n_slots=4, max_pages=8, slot_ids=FAKE,
             row_lens=FAKE, R=2, P=4, G=4, init=1, local=2, topk=8, out_ids=FAKE,
             out_scores=FAKE, ws=FAKE, ws_bytes=1 << 20, stream=None)
    a.update(over)
    return L.idx_score_topk(a["q"], a["q_scale"], a["q_dtype"], a["k_payload"], a["k_scale"],
                            a["k_dtype"], a["num_pages"], a["page_table"], a["n_slots"],
                            a["max_pages"], a["slot_ids"], a["row_lens"], a["R"], a["P"], a["G"],
                            a["init"], a["local"], a["topk"], a["out_ids"], a["out_scores"],
                            a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(P=200, G=200), -1),             # more than IDX_MAX_ROWS_PER_REQUEST rows
    (dict(R=17, P=128, G=128), -1),       # 17 x 128 tensor-core tiles > 2048 per call
    (dict(P=0), -1),
    (dict(topk=0), -1),
    (dict(topk=257), -1),
    (dict(init=4, local=5, topk=8), -1),  # forced blocks cannot fit
    (dict(local=-1), -1),
    (dict(R=-1), -1),
    (dict(q=None), -1),
    (dict(ws=None), -1),
    (dict(ws=FAKE + 16), -1),             # misaligned workspace
    (dict(ws_bytes=100), -1),             # workspace too small
    (dict(k_dtype=1, q_dtype=0), -2),     # fp8 keys with bf16 q
    (dict(k_dtype=2, q_dtype=1), -2),     # NVFP4 keys with fp8 q
    (dict(k_dtype=1, q_dtype=1, k_scale=FAKE), -1),  # fp8 q without q_scale
    (dict(k_dtype=1, q_dtype=1, q_scale=FAKE), -1),  # fp8 keys without k_scale
    (dict(n_slots=0), -1),
    (dict(max_pages=0), -1),
    (dict(num_pages=0), -1),
])
def test_host_side_validation(L, over, status):
    assert _call(L, **over) == status
    assert L.idx_last_error() != b""


def test_pool_alloc_validation(L):
    p = _lib.IdxPool()
    assert L.idx_pool_alloc(0, 10, 32, 128, ctypes.byref(p)) == -1
    assert L.idx_pool_alloc(0, 10, 64, 64, ctypes.byref(p)) == -1
    assert L.idx_pool_alloc(7, 10, 64, 128, ctypes.byref(p)) == -1
    assert L.idx_pool_alloc(0, 0, 64, 128, ctypes.byref(p)) == -1


def test_store_validation(L):
    p = _lib.IdxPool()
    p.dtype, p.page_size, p.dim, p.num_pages = 0, 64, 128, 10   # not NVFP4
    p.payload, p.scale, p.payload_row_bytes, p.scale_row_bytes = FAKE, FAKE, 256, 0
    assert L.idx_store_nvfp4(FAKE, FAKE, 10, ctypes.byref(p), None) == -1
    p.dtype, p.payload_row_bytes, p.scale_row_bytes = 2, 64, 8
    assert L.idx_store_nvfp4(FAKE, FAKE, -1, ctypes.byref(p), None) == -1
    assert L.idx_store_nvfp4(FAKE, FAKE, 0, ctypes.byref(p), None) == 0   # no-op


def test_cpu_tensors_are_refused():
    import torch
    with pytest.raises(idx.IdxError):
        idx.idx_store_nvfp4(torch.zeros((1, 128), dtype=torch.bfloat16),
                            torch.zeros(1, dtype=torch.int64),
                            (torch.zeros((64, 64), dtype=torch.uint8), torch.zeros((64, 8), dtype=torch.uint8)))


def _shard(L, **over):
    a = dict(q=FAKE, q_scale=None, q_dtype=0, k_payload=FAKE, k_scale=None, k_dtype=0,
             num_pages=100, page_table=FAKE, n_slots=4, max_pages=8, block_begin=0,
             slot_ids=FAKE, row_lens=FAKE, R=2, P=4, G=4, init=1, local=2, topk=8,
             out_ids=FAKE, out_scores=FAKE, ws=FAKE, ws_bytes=1 << 20, stream=None)
    a.update(over)
    return L.idx_score_local_blocks(a["q"], a["q_scale"], a["q_dtype"], a["k_payload"],
                                    a["k_scale"], a["k_dtype"], a["num_pages"], a["page_table"],
                                    a["n_slots"], a["max_pages"], a["block_begin"], a["slot_ids"],
                                    a["row_lens"], a["R"], a["P"], a["G"], a["init"], a["local"],
                                    a["topk"], a["out_ids"], a["out_scores"], a["ws"],
                                    a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over", [
    dict(block_begin=-1),
    dict(max_pages=7),          # a shard holds whole 128-token blocks
    dict(P=8, G=4),             # more than one 16-row tile: refused in shard mode
    dict(topk=0),
    dict(q=None),
])
def test_shard_scoring_validation(L, over):
    assert _shard(L, **over) == -1
    assert L.idx_last_error() != b""


def _merge(L, **over):
    a = dict(ids=FAKE, sc=FAKE, world=3, slot_ids=FAKE, row_lens=FAKE, n_slots=4, R=2, P=4,
             G=4, init=1, local=2, topk=8, out_ids=FAKE, out_scores=FAKE, stream=None)
    a.update(over)
    return L.idx_topk_merge(a["ids"], a["sc"], a["world"], a["slot_ids"], a["row_lens"],
                            a["n_slots"], a["R"], a["P"], a["G"], a["init"], a["local"],
                            a["topk"], a["out_ids"], a["out_scores"], a["stream"])


@pytest.mark.parametrize("over", [
    dict(world=0),
    dict(world=9),              # more than IDX_MAX_CP_WORLD shards
    dict(R=-1),
    dict(R=2049),
    dict(P=0),
    dict(topk=257),
    dict(init=5, local=5, topk=8),
    dict(n_slots=0),
    dict(ids=None),
    dict(out_scores=None),
])
def test_merge_validation(L, over):
    assert _merge(L, **over) == -1
    assert L.idx_last_error() != b""


def test_merge_of_no_requests_is_a_no_op(L):
    assert _merge(L, R=0, ids=None, sc=None, slot_ids=None, row_lens=None, out_ids=None,
                  out_scores=None) == 0

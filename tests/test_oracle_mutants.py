"""Plant mistakes in the oracle (on the CPU) and check that its pins catch
every one.

The mutants restate the injected bugs the verify test of sglang #42614 ("[AMD]
MiniMax-M3 indexer CP: packed scoring for EAGLE verify rows", Accuracy Tests)
must fail on: the group's block count in place of each row's, the group sized
by its shortest row, the forced local window dropped, a wrong score-row index,
the fp8 cast dropped, and keys addressed by request index instead of the slot
table.  Added for the NVFP4 store (ROCm/ATOM #2745, Summary): nibbles swapped,
scale rounded toward zero, division replaced by a reciprocal multiply; and for
the selection: ties to the higher id.
"""
import numpy as np
import pytest

import test_oracle_formats as F
import test_oracle_index as I
from oracle import formats, index

_orig_quantize = formats.nvfp4_quantize
_orig_row_block_max = index.row_block_max
_orig_forced = index.forced_blocks


def _pins():
    """Every pin, as (name, thunk)."""
    out = []
    for kd, qd in [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"), ("nvfp4", "bf16")]:
        out.append((f"blockmax_bruteforce[{kd}]", lambda kd=kd, qd=qd: I.test_blockmax_bruteforce(kd, qd)))
    for name in ["test_scores_closed_form_unit_queries", "test_selection_bruteforce_distinct",
                 "test_selection_ties_go_to_lower_id", "test_output_order_forced_then_rank",
                 "test_fewer_blocks_than_topk_pads", "test_forced_blocks_definition",
                 "test_tiny_rows_straddle_a_block_boundary", "test_packed_equals_rows_scored_alone",
                 "test_page_permutation_invariance", "test_pad_slots_and_empty_rows",
                 "test_local_zero_lets_partial_last_block_compete",
                 "test_fp8_query_scale_applies_per_packed_row",
                 "test_fp8_key_and_query_dequant_match_torch", "test_bf16_key_dequant_matches_torch",
                 "test_nvfp4_dequant_of_a_hand_worked_group"]:
        out.append((name, getattr(I, name)))
    for case in F._read_golden():
        out.append(("nvfp4_golden", lambda case=case: F.test_nvfp4_golden_groups(case)))
    out.append(("nvfp4_roundtrip", F.test_nvfp4_roundtrip_error_bound))
    return out


def _quantize_with(e4m3_enc=None, divide=None, swap_nibbles=False):
    def q(keys_bf16_bits):
        x = formats.bf16_bits_to_f32(keys_bf16_bits)
        T, D = x.shape
        g = x.reshape(T, D // 16, 16)
        amax = np.abs(g).max(axis=2).astype(np.float32)
        s_f = (amax / np.float32(6.0)).astype(np.float32)
        s_code = (e4m3_enc or formats.e4m3_encode)(s_f)
        s_val = formats.E4M3_TABLE[s_code].astype(np.float32)
        safe = np.where(s_val > 0, s_val, np.float32(1.0)).astype(np.float32)
        v = (divide or (lambda a, b: a / b))(g, safe[:, :, None]).astype(np.float32)
        codes = formats.e2m1_encode(v).reshape(T, D // 16, 16)
        codes = np.where((s_val > 0)[:, :, None], codes, 0).astype(np.uint8).reshape(T, D)
        lo, hi = codes[:, 0::2], codes[:, 1::2]
        if swap_nibbles:
            lo, hi = hi, lo
        return (lo | (hi << 4)).astype(np.uint8), s_code.astype(np.uint8)
    return q


def _e4m3_truncating(x):
    x = np.asarray(x, dtype=np.float64)
    mags = formats.E4M3_TABLE[:0x7F]
    code = np.clip(np.searchsorted(mags, np.abs(x), side="right") - 1, 0, 0x7E)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def _fp8_codes_as_ints_keys(codes, scale_bytes):
    s = np.ascontiguousarray(scale_bytes, dtype=np.uint8).view("<f4").reshape(-1)
    return np.asarray(codes, dtype=np.float64) * s.astype(np.float64)[:, None]


def _fp8_codes_as_ints_query(q_dtype, q_row, q_scale):
    if q_dtype == "fp8_e4m3":
        return np.asarray(q_row, dtype=np.float64) * float(q_scale)
    return formats.bf16_bits_to_f32(q_row).astype(np.float64)


def _select_ties_high(blockmax, init_blocks, local_blocks, topk):
    nb = len(blockmax)
    forced = index.forced_blocks(nb, init_blocks, local_blocks)
    cands = sorted((b for b in range(nb) if b not in set(forced)), key=lambda b: (-blockmax[b], -b))
    take = max(0, min(topk, nb) - len(forced))
    chosen = forced + cands[:take]
    ids = np.full(topk, -1, dtype=np.int64)
    sc = np.full(topk, -np.inf)
    ids[:len(chosen)] = chosen
    sc[:len(chosen)] = [blockmax[b] for b in chosen]
    return ids, sc


MUTANTS = {
    # (i) the group's block count in place of each row's (no per-row mask either)
    "group_block_count": [(index, "row_block_max", lambda q, keys, length: _orig_row_block_max(q, keys, len(keys)))],
    # (ii) the group sized by its shortest row
    "group_sized_by_shortest_row": [(index, "group_extent", lambda lens: min(lens))],
    # (iii) the forced local window dropped
    "local_window_dropped": [(index, "forced_blocks", lambda nb, init, local: _orig_forced(nb, init, 0))],
    # (iv) a wrong score-row index
    "wrong_score_row": [(index, "tile_row", lambda i, g: (i % g, i // g))],
    # (v) the fp8 cast dropped: codes used as plain integers
    "fp8_cast_dropped": [(formats, "fp8_dequantize", _fp8_codes_as_ints_keys),
                         (index, "dequant_query", _fp8_codes_as_ints_query)],
    # (vi) keys addressed by request index instead of the slot table
    "address_by_request_index": [(index, "request_slot", lambda slot_ids, r: r)],
    "nvfp4_nibbles_swapped": [(formats, "nvfp4_quantize", _quantize_with(swap_nibbles=True))],
    "nvfp4_scale_truncates": [(formats, "nvfp4_quantize", _quantize_with(e4m3_enc=_e4m3_truncating))],
    "nvfp4_reciprocal_multiply": [(formats, "nvfp4_quantize",
                                   _quantize_with(divide=lambda a, b: a * (np.float32(1.0) / b)))],
    "ties_to_higher_id": [(index, "select_row", _select_ties_high)],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    for mod, attr, fn in MUTANTS[name]:
        monkeypatch.setattr(mod, attr, fn)
    caught = []
    for pin, thunk in _pins():
        try:
            thunk()
        except Exception:          # an assertion or a crash both count as caught
            caught.append(pin)
    assert caught, f"mutant {name} passed every pin"

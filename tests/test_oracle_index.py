"""Pins for the oracle's scoring and selection (CPU only).

* block maxima against pure-Python loops (math.fsum over exact products);
* selection against brute-force search over all candidate subsets;
* closed forms: unit-vector queries turn scores into known key entries;
* invariants the pages fix: packed rows equal rows scored alone (sglang
  #45451, Modifications), per-row masking and forced blocks from each row's own
  length with rows straddling a block boundary, slot-table addressing and pad
  slots (sglang #42614, Modifications 1 and Accuracy Tests).
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import formats, index
from _util import oracle_kwargs, np_bits16


# ----------------------------------------------------------------------------
# block max: brute force
# ----------------------------------------------------------------------------
def _bruteforce_blockmax(qv, keys, L):
    out = []
    for b in range((L + 127) // 128):
        best = -math.inf
        for t in range(128 * b, min(128 * b + 128, L)):
            s = math.fsum(float(qv[d]) * float(keys[t, d]) for d in range(keys.shape[1]))
            best = max(best, s)
        out.append(best)
    return out


@pytest.mark.parametrize("k_dtype,q_dtype", [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"),
                                             ("nvfp4", "bf16")])
def test_blockmax_bruteforce(k_dtype, q_dtype):
    spec = workloads.small_spec("bm", 21, k_dtype, q_dtype, R=2, P=2, G=2,
                                explicit_lens=[[130, 300], [1, 257]])
    b = workloads.make_batch(spec)
    kw = oracle_kwargs(b)
    res = index.index_step(**kw)
    for r in range(b.R):
        slot = int(b.slot_ids[r])
        Lg = int(b.row_lens[r].max())
        keys = index.dequant_keys(k_dtype, kw["payload"], kw["scale"],
                                  index.key_rows(kw["page_table"], slot, Lg))
        for i in range(b.M):
            j, h = i // spec.gqa, i % spec.gqa
            L = int(b.row_lens[r, j])
            qs = None if kw["q_scale"] is None else kw["q_scale"][r, i]
            qv = index.dequant_query(q_dtype, kw["q"][r, j, h], qs)
            ref = _bruteforce_blockmax(qv, keys, L)
            np.testing.assert_allclose(res.blockmax[(r, i)], ref, rtol=1e-12, atol=1e-9)


def test_scores_closed_form_unit_queries():
    """q_i = e_i makes every token score equal to key entry i, so the block max
    is the max of column i over the block: keys hold small integers here."""
    L = 300
    t = np.arange(L)[:, None]
    d = np.arange(128)[None, :]
    kv = ((t * 7 + d * 3) % 11 - 5).astype(np.float32)          # exact in bf16
    payload = torch.from_numpy(kv).to(torch.bfloat16).view(torch.uint8).numpy()
    pad = np.zeros((5 * 64 - L, 256), np.uint8)
    payload = np.concatenate([payload, pad])
    page_table = np.array([[0, 1, 2, 3, 4]], np.int32)
    q = np.zeros((1, 4, 4, 128), np.float32)
    for i in range(16):
        q[0, i // 4, i % 4, i] = 1.0
    qb = np_bits16(torch.from_numpy(q).to(torch.bfloat16))
    res = index.index_step(q=qb, q_dtype="bf16", q_scale=None, payload=payload, scale=None,
                           k_dtype="bf16", page_table=page_table, slot_ids=np.array([0]),
                           row_lens=np.array([[L, L, L, L]]), packed_queries=4, gqa=4,
                           init_blocks=0, local_blocks=0, topk=3)
    for i in range(16):
        col = kv[:, i]
        expect = [col[0:128].max(), col[128:256].max(), col[256:300].max()]
        assert res.blockmax[(0, i)].tolist() == expect


# ----------------------------------------------------------------------------
# selection: brute force over subsets
# ----------------------------------------------------------------------------
def _bruteforce_select(bm, init_blocks, local_blocks, topk):
    nb = len(bm)
    forced = set(range(min(init_blocks, nb))) | set(range(max(0, nb - local_blocks), nb))
    cands = [b for b in range(nb) if b not in forced]
    c = max(0, min(topk, nb) - len(forced))
    best = None
    for sub in itertools.combinations(cands, c):
        # better = larger sorted score vector; among equal, lexicographically smaller ids
        key = (sorted((bm[b] for b in sub), reverse=True), [-x for x in sorted(sub)])
        if best is None or key > best[0]:
            best = (key, set(sub))
    return forced | (best[1] if best else set())


def test_selection_bruteforce_distinct():
    rng = np.random.default_rng(3)
    for _ in range(300):
        nb = int(rng.integers(0, 13))
        init = int(rng.integers(0, 3))
        local = int(rng.integers(0, 3))
        topk = int(rng.integers(init + local, init + local + 6)) if init + local > 0 else int(rng.integers(1, 7))
        bm = rng.standard_normal(nb) * 10
        ids, sc = index.select_row(bm, init, local, topk)
        got = set(int(x) for x in ids if x >= 0)
        assert got == _bruteforce_select(bm, init, local, topk)
        n = len(got)
        assert n == min(topk, nb)
        assert np.all(ids[n:] == -1) and np.all(np.isneginf(sc[n:]))
        assert np.array_equal(sc[:n], bm[ids[:n]])


def test_selection_ties_go_to_lower_id():
    rng = np.random.default_rng(4)
    for _ in range(200):
        nb = int(rng.integers(1, 11))
        bm = rng.integers(0, 3, nb).astype(np.float64)     # many exact ties
        topk = int(rng.integers(1, 6))
        ids, _ = index.select_row(bm, 0, 0, topk)
        got = set(int(x) for x in ids if x >= 0)
        assert got == _bruteforce_select(bm, 0, 0, topk)


def test_output_order_forced_then_rank():
    bm = np.array([0.0, 5.0, 9.0, 1.0, 7.0, 3.0, 8.0])
    ids, sc = index.select_row(bm, init_blocks=1, local_blocks=2, topk=5)
    # forced: 0 (init), 5, 6 (local); then best candidates 2 (9.0), 4 (7.0)
    assert ids.tolist() == [0, 5, 6, 2, 4]
    assert sc.tolist() == [0.0, 3.0, 8.0, 9.0, 7.0]


def test_fewer_blocks_than_topk_pads():
    bm = np.array([1.0, 2.0, 3.0])
    ids, sc = index.select_row(bm, 1, 1, 8)
    assert ids.tolist() == [0, 2, 1, -1, -1, -1, -1, -1]
    assert np.isneginf(sc[3:]).all()


def test_forced_blocks_definition():
    assert index.forced_blocks(10, 1, 4) == [0, 6, 7, 8, 9]
    assert index.forced_blocks(3, 1, 4) == [0, 1, 2]
    assert index.forced_blocks(5, 0, 0) == []
    assert index.forced_blocks(0, 1, 4) == []
    assert index.forced_blocks(33, 1, 2) == [0, 31, 32]


# ----------------------------------------------------------------------------
# invariants of the packed step
# ----------------------------------------------------------------------------
def _tiny():
    return workloads.make_batch(workloads.WORKLOADS["tiny_bf16_1x4k"])


def test_tiny_rows_straddle_a_block_boundary():
    b = _tiny()
    kw = oracle_kwargs(b)
    res = index.index_step(**kw)
    nbs = [len(res.blockmax[(0, i)]) for i in range(16)]
    # rows end at tokens 4095..4098: lengths 4096..4099 -> 32 and 33 blocks
    assert nbs == [32] * 4 + [33] * 12
    for i in range(16):
        nb = nbs[i]
        ids = res.ids[0, i].tolist()
        # forced: block 0 and the row's own last two blocks
        assert ids[:3] == [0, nb - 2, nb - 1]


def test_packed_equals_rows_scored_alone():
    """Each packed row (draft row i // G, head i % G) equals the same row run as
    its own one-row request (P = G = 1)."""
    spec = workloads.small_spec("pk", 31, "bf16", "bf16", R=3, P=4, G=4, len_range=(100, 2000))
    b = workloads.make_batch(spec)
    kw = oracle_kwargs(b)
    packed = index.index_step(**kw)
    for r in range(b.R):
        for i in range(b.M):
            j, h = i // spec.gqa, i % spec.gqa
            kw1 = dict(kw)
            kw1.update(q=kw["q"][r:r + 1, j:j + 1, h:h + 1], slot_ids=kw["slot_ids"][r:r + 1],
                       row_lens=kw["row_lens"][r:r + 1, j:j + 1], packed_queries=1, gqa=1)
            alone = index.index_step(**kw1)
            assert np.array_equal(alone.ids[0, 0], packed.ids[r, i])
            assert np.array_equal(alone.scores[0, 0], packed.scores[r, i])


def test_page_permutation_invariance():
    """Moving a request's pages to other physical pages (and updating the page
    table) changes nothing: keys are reached only through the slot table."""
    spec = workloads.small_spec("perm", 41, "fp8_e4m3", "fp8_e4m3", R=3, len_range=(50, 3000))
    b = workloads.make_batch(spec)
    kw = oracle_kwargs(b)
    base = index.index_step(**kw)
    rng = np.random.default_rng(0)
    npg = b.num_pages
    perm = rng.permutation(npg)
    payload = np.empty_like(kw["payload"])
    scale = np.empty_like(kw["scale"])
    for p in range(npg):
        payload[perm[p] * 64:(perm[p] + 1) * 64] = kw["payload"][p * 64:(p + 1) * 64]
        scale[perm[p] * 64:(perm[p] + 1) * 64] = kw["scale"][p * 64:(p + 1) * 64]
    kw2 = dict(kw, payload=payload, scale=scale, page_table=perm[kw["page_table"]].astype(np.int32))
    moved = index.index_step(**kw2)
    assert np.array_equal(base.ids, moved.ids)
    assert np.array_equal(base.scores, moved.scores)


def test_slots_are_gapped_and_not_the_request_index():
    b = workloads.make_batch(workloads.WORKLOADS["verify_bf16_4x32k"])
    s = b.slot_ids.tolist()
    assert len(set(s)) == len(s)
    assert all(s[r] != r for r in range(len(s)))
    assert s != sorted(s) or max(s) >= len(s)


def test_pad_slots_and_empty_rows():
    spec = workloads.small_spec("pad", 51, "bf16", "bf16", R=4, P=2, G=2,
                                explicit_lens=[[0, 0], [5, 300], [200, 200], [1, 1]],
                                pad_requests=(2, 3))
    b = workloads.make_batch(spec)
    assert int(b.slot_ids[2]) < 0 and int(b.slot_ids[3]) >= b.n_slots
    res = index.index_step(**oracle_kwargs(b))
    for r in (0, 2, 3):
        assert np.all(res.ids[r] == -1) and np.all(np.isneginf(res.scores[r]))
    # request 1: draft row 0 (5 tokens, one block), draft row 1 (300 tokens, 3 blocks)
    assert [int((res.ids[1, i] >= 0).sum()) for i in range(4)] == [1, 1, 3, 3]


def test_local_zero_lets_partial_last_block_compete():
    """With local_blocks = 0 the partial last block is an ordinary candidate:
    it is chosen only on its score."""
    L = 129
    rows = np.arange(L)
    kv = np.zeros((3 * 64, 128), np.float32)
    kv[rows, 0] = np.where(rows == 128, 5.0, 1.0)   # the lone token of block 1 scores 5
    payload = torch.from_numpy(kv).to(torch.bfloat16).view(torch.uint8).numpy()
    q = np.zeros((1, 1, 1, 128), np.float32)
    q[..., 0] = 1.0
    qb = np_bits16(torch.from_numpy(q).to(torch.bfloat16))
    common = dict(q=qb, q_dtype="bf16", q_scale=None, payload=payload, scale=None,
                  k_dtype="bf16", page_table=np.array([[0, 1, 2]], np.int32),
                  slot_ids=np.array([0]), row_lens=np.array([[L]]), packed_queries=1, gqa=1)
    r = index.index_step(**common, init_blocks=0, local_blocks=0, topk=1)
    assert r.ids[0, 0].tolist() == [1]
    kv[128, 0] = 0.5
    payload = torch.from_numpy(kv).to(torch.bfloat16).view(torch.uint8).numpy()
    common["payload"] = payload
    r = index.index_step(**common, init_blocks=0, local_blocks=0, topk=1)
    assert r.ids[0, 0].tolist() == [0]
    r = index.index_step(**common, init_blocks=0, local_blocks=1, topk=1)
    assert r.ids[0, 0].tolist() == [1]


def test_fp8_query_scale_applies_per_packed_row():
    spec = workloads.small_spec("qs", 61, "fp8_e4m3", "fp8_e4m3", R=1, P=2, G=2,
                                explicit_lens=[[256, 256]])
    b = workloads.make_batch(spec)
    kw = oracle_kwargs(b)
    base = index.index_step(**kw)
    qs = kw["q_scale"].copy()
    qs[0, 3] *= 2.0
    doubled = index.index_step(**dict(kw, q_scale=qs))
    np.testing.assert_array_equal(doubled.blockmax[(0, 0)], base.blockmax[(0, 0)])
    np.testing.assert_allclose(doubled.blockmax[(0, 3)], 2 * base.blockmax[(0, 3)], rtol=1e-15)


# ----------------------------------------------------------------------------
# dequantisation of the stored planes, against torch's own conversions
# ----------------------------------------------------------------------------
def test_fp8_key_and_query_dequant_match_torch():
    spec = workloads.small_spec("dq", 71, "fp8_e4m3", "fp8_e4m3", R=2, len_range=(64, 500))
    b = workloads.make_batch(spec)
    kw = oracle_kwargs(b)
    rows = np.arange(0, b.num_pages * 64, 37)
    got = index.dequant_keys("fp8_e4m3", kw["payload"], kw["scale"], rows)
    codes = b.payload[torch.from_numpy(rows)].view(torch.float8_e4m3fn).to(torch.float64)
    sc = b.scale[torch.from_numpy(rows)].contiguous().view(torch.float32).to(torch.float64)
    np.testing.assert_array_equal(got, (codes * sc).numpy())
    qv = index.dequant_query("fp8_e4m3", kw["q"][1, 2, 3], kw["q_scale"][1, 2 * 4 + 3])
    ref = b.q[1, 2, 3].view(torch.float8_e4m3fn).to(torch.float64) * float(b.q_scale[1, 11])
    np.testing.assert_array_equal(qv, ref.numpy())


def test_bf16_key_dequant_matches_torch():
    spec = workloads.small_spec("dqb", 72, "bf16", "bf16", R=1, len_range=(64, 200))
    b = workloads.make_batch(spec)
    rows = np.arange(0, b.num_pages * 64, 29)
    got = index.dequant_keys("bf16", oracle_kwargs(b)["payload"], None, rows)
    ref = b.payload[torch.from_numpy(rows)].contiguous().view(torch.bfloat16).to(torch.float64)
    np.testing.assert_array_equal(got, ref.numpy())


def test_nvfp4_dequant_of_a_hand_worked_group():
    # first hand-worked group of tests/golden/nvfp4_groups.txt: scale 1.0 and the
    # codes rounded by hand, decoded: 6 -6 0 1 1 2 2 4 4 -0 1 .5 3 4 2 1.5
    payload = np.zeros((1, 64), np.uint8)
    scale = np.zeros((1, 8), np.uint8)
    payload[0, 8:16] = [0xF7, 0x20, 0x42, 0x64, 0x86, 0x12, 0x65, 0x34]
    scale[0, 1] = 0x38
    v = formats.nvfp4_dequantize(payload, scale)
    assert v[0, 16:32].tolist() == [6, -6, 0, 1, 1, 2, 2, 4, 4, -0.0, 1, 0.5, 3, 4, 2, 1.5]
    assert np.all(v[0, :16] == 0) and np.all(v[0, 32:] == 0)
    scale[0, 1] = 0x30   # 0.5
    v = formats.nvfp4_dequantize(payload, scale)
    assert v[0, 16:20].tolist() == [3, -3, 0, 0.5]


# ----------------------------------------------------------------------------
# log-sum-exp block score
# ----------------------------------------------------------------------------
def _bruteforce_blocklse(qv, keys, L):
    out = []
    for b in range((L + 127) // 128):
        ss = [math.fsum(float(qv[d]) * float(keys[t, d]) for d in range(keys.shape[1]))
              for t in range(128 * b, min(128 * b + 128, L))]
        m = max(ss)
        out.append(m + math.log(math.fsum(math.exp(x - m) for x in ss)))
    return out


@pytest.mark.parametrize("k_dtype,q_dtype", [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3")])
def test_blocklse_bruteforce(k_dtype, q_dtype):
    spec = workloads.small_spec("lse", 22, k_dtype, q_dtype, R=2, P=2, G=2,
                                explicit_lens=[[130, 300], [1, 257]])
    b = workloads.make_batch(spec)
    kw = oracle_kwargs(b)
    res = index.index_step(**kw, block_score="lse")
    for r in range(b.R):
        slot = int(b.slot_ids[r])
        keys = index.dequant_keys(k_dtype, kw["payload"], kw["scale"],
                                  index.key_rows(kw["page_table"], slot, int(b.row_lens[r].max())))
        for i in range(b.M):
            j, h = i // spec.gqa, i % spec.gqa
            L = int(b.row_lens[r, j])
            qs = None if kw["q_scale"] is None else kw["q_scale"][r, i]
            qv = index.dequant_query(q_dtype, kw["q"][r, j, h], qs)
            np.testing.assert_allclose(res.blockmax[(r, i)], _bruteforce_blocklse(qv, keys, L),
                                       rtol=1e-12, atol=1e-9)


def test_blocklse_closed_forms_and_bounds():
    """n equal scores c give c + ln n; one token gives its score; in general
    max <= lse <= max + ln(n valid tokens)."""
    L = 300
    kv = np.zeros((5 * 64, 128), np.float32)
    kv[:L, 0] = 2.0                       # every score equals 2 (q = e_0)
    kv[:L, 1] = np.random.default_rng(1).standard_normal(L)
    payload = torch.from_numpy(kv).to(torch.bfloat16).view(torch.uint8).numpy()
    q = np.zeros((1, 2, 1, 128), np.float32)
    q[0, 0, 0, 0] = 1.0
    q[0, 1, 0, 1] = 1.0
    qb = np_bits16(torch.from_numpy(q).to(torch.bfloat16))
    common = dict(q=qb, q_dtype="bf16", q_scale=None, payload=payload, scale=None, k_dtype="bf16",
                  page_table=np.array([[0, 1, 2, 3, 4]], np.int32), slot_ids=np.array([0]),
                  row_lens=np.array([[L, 257]]), packed_queries=2, gqa=1, init_blocks=0,
                  local_blocks=0, topk=3)
    lse = index.index_step(**common, block_score="lse")
    mx = index.index_step(**common, block_score="max")
    np.testing.assert_allclose(lse.blockmax[(0, 0)], [2 + math.log(128), 2 + math.log(128),
                                                      2 + math.log(44)], rtol=1e-12)
    # row 1 (257 tokens): its last block holds one token, so lse = that score
    assert lse.blockmax[(0, 1)][-1] == mx.blockmax[(0, 1)][-1]
    counts = [128, 128, 1]
    for b in range(3):
        m, v = mx.blockmax[(0, 1)][b], lse.blockmax[(0, 1)][b]
        assert m <= v <= m + math.log(counts[b]) + 1e-12


# ---- indexer context parallelism: shard lists and their merge --------------
def _random_partition(rng, nb):
    cuts = sorted(set(rng.integers(0, nb + 1, size=rng.integers(0, 4)).tolist()) | {0, nb})
    return list(zip(cuts[:-1], cuts[1:]))


@pytest.mark.parametrize("seed", range(40))
def test_merge_of_shards_equals_the_single_device_selection(seed):
    """For any split of a row's blocks into contiguous shards, merging the
    shards' lists gives exactly select_row over the whole row: each shard keeps
    its best c candidates, so every globally chosen block reaches the merge.
    Rows with many tied scores (few distinct values) are included."""
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(1, 60))
    if seed % 3 == 0:
        bm = rng.integers(0, 3, size=nb).astype(np.float64)   # heavy ties
    else:
        bm = rng.standard_normal(nb)
    init, local = int(rng.integers(0, 3)), int(rng.integers(0, 4))
    topk = int(rng.integers(init + local, init + local + 12)) or 1
    parts = _random_partition(rng, nb)
    lists = [index.shard_select(bm, b0, b1, init, local, topk) for b0, b1 in parts]
    ids, sc = index.merge_shards(lists, nb, init, local, topk)
    ref_ids, ref_sc = index.select_row(bm, init, local, topk)
    assert ids.tolist() == ref_ids.tolist()
    assert sc.tolist() == ref_sc.tolist()


def test_shard_lists_brute_force():
    """A shard's list on a tiny row, against brute force over every subset of
    its candidates: the chosen ones are the subset of the right size whose
    sorted (score desc, id asc) sequence is lexicographically best."""
    bm = np.array([0.5, 2.0, -1.0, 2.0, 0.25, 3.0, 0.5, 1.0])
    init, local, topk = 1, 1, 5          # forced {0, 7}; c = 3
    ids, sc = index.shard_select(bm, 2, 7, init, local, topk)
    cands = [2, 3, 4, 5, 6]
    best = None
    for sub in itertools.combinations(cands, 3):
        key = sorted(((-bm[b], b) for b in sub))
        if best is None or key < best[0]:
            best = (key, sub)
    want = [b for _, b in best[0]]
    assert ids.tolist() == want + [-1, -1]
    # a shard holding a forced block lists it first
    ids0, _ = index.shard_select(bm, 0, 3, init, local, topk)
    assert ids0.tolist()[:1] == [0] and set(ids0.tolist()[1:3]) == {1, 2}

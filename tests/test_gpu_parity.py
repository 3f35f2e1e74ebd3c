"""CUDA path vs the fp64 oracle on the same seeded inputs (needs a GPU).

Bar: NVFP4 stored bytes bit-exact; block-max scores within 1e-3 * (1 + |s|);
top-k id sets exact except where the oracle's k-th and (k+1)-th candidates
lie within that tolerance, and then only in candidates within it of the k-th
(tests/_util.compare_row).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _util import compare_row, near_tie_violation, oracle_kwargs, oracle_planes, np_u8, score_tol
import _gpu

pytestmark = pytest.mark.gpu


def _check_all_rows(batch, out, ref, init_blocks=None, local_blocks=None):
    s = batch.spec
    init_blocks = s.init_blocks if init_blocks is None else init_blocks
    local_blocks = s.local_blocks if local_blocks is None else local_blocks
    bad = []
    for r in range(batch.R):
        for i in range(batch.M):
            bm = ref.blockmax.get((r, i), np.zeros(0))
            err = compare_row(out.ids[r, i], out.scores[r, i], ref.ids[r, i], ref.scores[r, i],
                              bm, init_blocks, local_blocks)
            if err:
                bad.append(f"request {r} row {i}: {err}")
    assert not bad, "\n".join(bad[:20]) + f"\n({len(bad)} rows differ)"


def _check_blockmax(batch, out, ref):
    """Every block max the oracle defines, against the workspace."""
    worst = 0.0
    for (r, i), bm in ref.blockmax.items():
        got = out.blockmax[r * batch.M + i, :len(bm)].astype(np.float64)
        err = np.abs(got - bm) / score_tol(bm)
        worst = max(worst, float(err.max()))
    assert worst <= 1.0, f"block max off by {worst:.3f} x tolerance"


TINY_BF16 = workloads.WORKLOADS["tiny_bf16_1x4k"]


def test_tiny_bf16():
    b = workloads.make_batch(TINY_BF16)
    out = _gpu.run(b)
    ref = oracle.index.index_step(**oracle_kwargs(b))
    assert out.flags == 0
    _check_blockmax(b, out, ref)
    _check_all_rows(b, out, ref)


SMALL = []
for k_dtype, q_dtype in [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"), ("nvfp4", "bf16")]:
    for seed, (P, G), lens, pads, init, local, topk in [
        (101, (4, 4), (1, 9000), (), 1, 2, 16),
        (102, (4, 4), (1, 3000), (1, 3), 1, 4, 64),
        (103, (1, 16), (100, 6000), (), 2, 2, 8),
        (104, (16, 1), (1, 5000), (0,), 0, 0, 5),
        (105, (2, 3), (1, 4000), (), 1, 0, 12),
        (106, (4, 4), (120, 700), (), 1, 4, 64),      # nb < topk for most rows
    ]:
        SMALL.append(pytest.param(k_dtype, q_dtype, seed, P, G, lens, pads, init, local, topk,
                                  id=f"{k_dtype}-{seed}-P{P}G{G}"))


@pytest.mark.parametrize("k_dtype,q_dtype,seed,P,G,lens,pads,init,local,topk", SMALL)
def test_small_parity(k_dtype, q_dtype, seed, P, G, lens, pads, init, local, topk):
    spec = workloads.small_spec(f"s{seed}", seed, k_dtype, q_dtype, R=6, P=P, G=G,
                                init_blocks=init, local_blocks=local, topk=topk, len_range=lens,
                                pad_requests=pads)
    b = workloads.make_batch(spec)
    out = _gpu.run(b)
    ref = oracle.index.index_step(**oracle_kwargs(b))
    assert out.flags == 0
    _check_blockmax(b, out, ref)
    _check_all_rows(b, out, ref)


LSE = []
for k_dtype, q_dtype in [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"), ("nvfp4", "bf16")]:
    for seed, (P, G), lens, pads, init, local, topk in [
        (111, (4, 4), (1, 9000), (2,), 1, 2, 16),
        (112, (1, 16), (100, 6000), (), 2, 2, 8),
        (113, (2, 3), (1, 4000), (), 1, 0, 12),
    ]:
        LSE.append(pytest.param(k_dtype, q_dtype, seed, P, G, lens, pads, init, local, topk,
                                id=f"{k_dtype}-{seed}-P{P}G{G}"))


@pytest.mark.parametrize("k_dtype,q_dtype,seed,P,G,lens,pads,init,local,topk", LSE)
def test_lse_block_score_parity(k_dtype, q_dtype, seed, P, G, lens, pads, init, local, topk):
    """Log-sum-exp block score (sglang #45451, Accuracy Tests): every block's
    score and every row's selection against the oracle's lse reading."""
    spec = workloads.small_spec(f"l{seed}", seed, k_dtype, q_dtype, R=5, P=P, G=G,
                                init_blocks=init, local_blocks=local, topk=topk, len_range=lens,
                                pad_requests=pads)
    b = workloads.make_batch(spec)
    out = _gpu.run(b, block_score="lse")
    ref = oracle.index.index_step(**oracle_kwargs(b), block_score="lse")
    assert out.flags == 0
    _check_blockmax(b, out, ref)
    _check_all_rows(b, out, ref)


def test_lse_bounds_the_max_on_device():
    """On the same planes, max <= lse <= max + ln(tokens in the block) for
    every block both variants score."""
    spec = workloads.small_spec("lb", 121, "bf16", "bf16", R=4, len_range=(1, 6000), topk=16)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    mx = _gpu.run(b, planes=planes)
    ls = _gpu.run(b, planes=planes, block_score="lse")
    lens = b.row_lens.numpy().reshape(b.R, spec.packed_queries)
    for r in range(b.R):
        if not (0 <= int(b.slot_ids[r]) < b.page_table.shape[0]):
            continue
        for i in range(b.M):
            L = int(lens[r, i // spec.gqa])
            nb = (L + 127) // 128
            if nb == 0:
                continue
            m = mx.blockmax[r * b.M + i, :nb].astype(np.float64)
            l = ls.blockmax[r * b.M + i, :nb].astype(np.float64)
            n = np.minimum(128, L - 128 * np.arange(nb))
            assert np.all(l >= m - score_tol(m)), (r, i)
            assert np.all(l <= m + np.log(n) + score_tol(m)), (r, i)


@pytest.mark.parametrize("name", ["verify_bf16_4x32k", "verify_fp8_4x32k"])
def test_verify_rows_4x4_ending_32767(name):
    """4 requests x 4 draft rows ending at tokens 32767..32770: one tile mixes
    256- and 257-block rows with different local windows."""
    b = workloads.make_batch(workloads.WORKLOADS[name])
    out = _gpu.run(b)
    ref = oracle.index.index_step(**oracle_kwargs(b))
    _check_blockmax(b, out, ref)
    _check_all_rows(b, out, ref)


@pytest.mark.parametrize("k_dtype,q_dtype", [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"),
                                             ("nvfp4", "bf16")])
def test_packed_equals_perrow_bitwise(k_dtype, q_dtype):
    """Both variants run the same 16-row MMA, so the max scores are equal
    bit for bit and so are the selections."""
    spec = workloads.small_spec("pp", 201, k_dtype, q_dtype, R=5, len_range=(1, 7000), topk=32)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    a = _gpu.run(b, planes=planes)
    p = _gpu.run(b, planes=planes, perrow=True)
    assert np.array_equal(a.ids, p.ids)
    assert np.array_equal(a.scores.view(np.uint32), p.scores.view(np.uint32))


def test_nvfp4_store_bitexact():
    spec = workloads.small_spec("st", 301, "nvfp4", "bf16", R=4, len_range=(1, 5000))
    b = workloads.make_batch(spec)
    payload, scale = _gpu.device_planes(b)
    ref_payload, ref_scale = oracle_planes(b)
    assert np.array_equal(np_u8(payload.cpu()), ref_payload)
    assert np.array_equal(np_u8(scale.cpu()), ref_scale)


def test_nvfp4_store_golden_groups():
    import test_oracle_formats as F
    cases = F._read_golden()
    n = len(cases)
    src = torch.zeros((n * 8, 128), dtype=torch.bfloat16)
    for c, (x, sc, pay) in enumerate(cases):
        for g in range(8):
            src[c * 8 + g, 16 * g:16 * g + 16] = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)
    payload = torch.zeros((n * 8 + 64, 64), dtype=torch.uint8, device="cuda")
    scale = torch.zeros((n * 8 + 64, 8), dtype=torch.uint8, device="cuda")
    rows = torch.arange(n * 8, dtype=torch.int64) + 3   # rows shifted off the identity
    import sparse_attention_indexer_packed_gb300 as idx
    idx.idx_store_nvfp4(src.cuda(), rows.cuda(), (payload, scale))
    P = payload.cpu().numpy()
    S = scale.cpu().numpy()
    for c, (x, sc, pay) in enumerate(cases):
        for g in range(8):
            row = c * 8 + g + 3
            assert S[row, g] == sc, (c, g, hex(S[row, g]))
            assert P[row, 8 * g:8 * g + 8].tolist() == pay, (c, g, P[row].tolist())


def _every_midpoint_groups():
    """bf16 bit patterns [G, 16]: for every positive finite E4M3 scale s, groups
    whose amax is 6 s (so amax / 6 = s exactly) holding each e2m1 midpoint t * s
    (t in .25, .75, 1.25, 1.75, 2.5, 3.5, 5), its negation, its bf16 neighbours,
    -0 and -6 s: every tie of the rounding at every scale."""
    import oracle
    groups = []
    for code in range(1, 127):
        s = float(oracle.formats.E4M3_TABLE[code])
        bits = lambda v: int(np.array([v], np.float32).view(np.uint32)[0] >> 16)
        vals = []
        for t in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
            b = bits(t * s)
            assert np.array([t * s], np.float32)[0] == t * s
            vals += [b, b | 0x8000, b - 1, b + 1]
        six = bits(6 * s)
        vals += [0x8000, six | 0x8000]                 # -0 and -6 s
        for k in range(0, len(vals), 15):
            g = [six] + vals[k:k + 15]
            g += [0] * (16 - len(g))
            groups.append(g)
    return np.array(groups, dtype=np.uint16)


def test_nvfp4_store_every_midpoint_of_every_scale():
    """The store's codes at every tie of the e2m1 rounding, for all 126 scales,
    bit for bit against the oracle's quantiser (ROCm/ATOM #2745, Summary:
    half-to-even, saturating at 6; -0 and negatives that round to 0 keep the
    sign)."""
    import oracle
    g = _every_midpoint_groups()
    n_keys = -(-len(g) // 8)
    bits = np.zeros((n_keys * 8, 16), dtype=np.uint16)
    bits[:len(g)] = g
    bits = bits.reshape(n_keys, 128)
    want_pay, want_sc = oracle.formats.nvfp4_quantize(bits)
    assert (want_sc.reshape(-1)[:len(g)] == np.repeat(np.arange(1, 127), 2)[:len(g)]).all()
    src = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    rows = torch.arange(n_keys, dtype=torch.int64) + 5
    payload = torch.zeros((n_keys + 64, 64), dtype=torch.uint8, device="cuda")
    scale = torch.zeros((n_keys + 64, 8), dtype=torch.uint8, device="cuda")
    import sparse_attention_indexer_packed_gb300 as idx
    idx.idx_store_nvfp4(src, rows.cuda(), (payload, scale))
    P = payload.cpu().numpy()[5:5 + n_keys]
    S = scale.cpu().numpy()[5:5 + n_keys]
    assert np.array_equal(S, want_sc)
    bad = np.argwhere(P != want_pay)
    assert not len(bad), [(int(r), int(c), hex(P[r, c]), hex(want_pay[r, c])) for r, c in bad[:8]]


# Unit roundoff of one fp32 addition that truncates instead of rounding (the
# worst a tensor core's accumulation may do): 2^-23.
_U_TRUNC = 2.0 ** -23


def test_nvfp4_scores_match_bf16_scorer_on_dequantised_cache():
    """e2m1 x E4M3 values are exact in bf16 (ROCm/ATOM #2745, Validation), so the
    FP4 scorer and the bf16 scorer fed the dequantised keys sum the same 128 exact
    products per token.  They do not sum them in the same order: the NVFP4 path
    feeds the f16 MMA its k elements in the order the packed bytes arrive
    (32m + 8t + 4h + {0..3}) with the query scaled by a power of two, the bf16
    path in natural order, and fp32 addition is not associative, so bitwise
    equal scores cannot be promised.  What holds: each side is the exact sum
    after at most 127 fp32 additions, each off by at most one unit in the last
    place (2^-23 relative, even if the hardware truncates), so each differs from
    the exact sum by at most 127 * 2^-23 * sum_d |q_d k_d| to first order, and
    the two by twice that.  A block score is a max over tokens, so per block the
    bound takes the largest sum_d |q_d k_d| over the block's valid tokens.
    Every block score of every row is checked against that bound and the top-k
    ids must be equal except at a near tie within it."""
    spec = workloads.small_spec("eq", 401, "nvfp4", "bf16", R=5, len_range=(1, 8000), topk=32)
    b = workloads.make_batch(spec)
    payload, scale = _gpu.device_planes(b)
    out4 = _gpu.run(b, planes=(payload, scale))
    # dequantise the stored planes with the oracle, as bf16 keys
    deq = oracle.formats.nvfp4_dequantize(np_u8(payload.cpu()), np_u8(scale.cpu()))
    kb = torch.from_numpy(deq.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(kb.to(torch.float64), torch.from_numpy(deq))      # exact
    b16 = workloads.Batch(**{**b.__dict__})
    b16.spec = workloads.Spec(**{**spec.__dict__, "k_dtype": "bf16"})
    b16.payload = kb.view(torch.uint8).reshape(-1, 256)
    b16.scale = None
    out16 = _gpu.run(b16, planes=(b16.payload.cuda(), None))
    qf = b.q.to(torch.float64).numpy()
    pt, lens = b.page_table.numpy(), b.row_lens.numpy()
    worst, checked, bad = 0.0, 0, []
    for r in range(b.R):
        slot = int(b.slot_ids[r])
        if not 0 <= slot < b.n_slots:
            continue
        ext = int(lens[r].max())
        if ext <= 0:
            continue
        absk = np.abs(deq[oracle.index.key_rows(pt, slot, ext)])
        for i in range(b.M):
            j, h = divmod(i, spec.gqa)
            L = int(lens[r, j])
            nb = (L + 127) // 128
            if nb == 0:
                continue
            absdot = absk[:L] @ np.abs(qf[r, j, h])
            big = np.array([absdot[128 * x:min(128 * x + 128, L)].max() for x in range(nb)])
            bound = 2 * 127 * _U_TRUNC * big
            s4 = out4.blockmax[r * b.M + i, :nb].astype(np.float64)
            s16 = out16.blockmax[r * b.M + i, :nb].astype(np.float64)
            d = np.abs(s4 - s16)
            worst = max(worst, float((d / bound).max()))
            checked += nb
            if np.any(d > bound):
                bad.append((r, i, "block score"))
            got, want = set(out4.ids[r, i].tolist()) - {-1}, set(out16.ids[r, i].tolist()) - {-1}
            if got != want:
                forced = set(oracle.index.forced_blocks(nb, spec.init_blocks, spec.local_blocks))
                cands = [x for x in range(nb) if x not in forced]
                tol = lambda s, bd=float(bound.max()): bd
                err = near_tie_violation(s16, cands, len(want) - len(forced), got ^ want, tol)
                if err:
                    bad.append((r, i, err))
    assert checked > 0
    assert not bad, (bad[:10], f"worst |diff| / bound = {worst:.3g}")


def test_pad_requests_and_empty_rows():
    spec = workloads.small_spec("pad", 501, "bf16", "bf16", R=4, P=2, G=2,
                                explicit_lens=[[0, 0], [5, 300], [200, 200], [1, 1]],
                                pad_requests=(2, 3), topk=4)
    b = workloads.make_batch(spec)
    out = _gpu.run(b)
    ref = oracle.index.index_step(**oracle_kwargs(b))
    _check_all_rows(b, out, ref)
    for r in (0, 2, 3):
        assert np.all(out.ids[r] == -1) and np.all(np.isneginf(out.scores[r]))


def test_zero_requests():
    spec = workloads.small_spec("z", 502, "bf16", "bf16", R=1, len_range=(10, 20))
    b = workloads.make_batch(spec)
    import sparse_attention_indexer_packed_gb300 as idx
    q = b.q[:0].cuda()
    out_ids = torch.zeros((0, 16, 16), dtype=torch.int32, device="cuda")
    out_sc = torch.zeros((0, 16, 16), dtype=torch.float32, device="cuda")
    ws = idx.alloc_workspace(0, 4, 4, b.max_pages)
    idx.idx_score_topk(q, None, b.payload.cuda(), None, "bf16", b.page_table.cuda(),
                       b.slot_ids[:0].cuda(), b.row_lens[:0].cuda(), 4, 4, 1, 2, 16,
                       out_ids, out_sc, ws)
    torch.cuda.synchronize()


def test_most_requests_per_call():
    """IDX_MAX_REQUESTS (2048) requests of 16 packed rows in one call, short
    ragged contexts and a few pad requests: 32768 rows, so the warp-per-row
    top-k takes them."""
    spec = workloads.small_spec("mr", 504, "bf16", "bf16", R=2048, len_range=(1, 1200),
                                pad_requests=(0, 777, 2047), topk=12)
    b = workloads.make_batch(spec)
    out = _gpu.run(b)
    assert out.flags == 0
    ref = oracle.index.index_step(**oracle_kwargs(b))
    _check_blockmax(b, out, ref)
    _check_all_rows(b, out, ref)


@pytest.mark.parametrize("length,seed", [(300_000, 511), (600_000, 512)])
def test_long_rows_on_few_ctas(length, seed):
    """One request of ~300K / ~600K tokens packing 2 draft rows x 2 heads, so
    each row's selection runs on a 512-thread CTA and reads ~2300 / ~4700 block
    scores with eight / sixteen loads in flight per thread.  Every row and block
    score is checked against the oracle."""
    spec = workloads.small_spec(f"long{length}", seed, "bf16", "bf16", R=1, P=2, G=2,
                                len_range=(length - 1000, length), topk=64, local_blocks=4)
    b = workloads.make_batch(spec)
    out = _gpu.run(b)
    assert out.flags == 0
    ref = oracle.index.index_step(**oracle_kwargs(b))
    _check_blockmax(b, out, ref)
    _check_all_rows(b, out, ref)


def test_topk_edge_values():
    """topk = init + local (no free choice), topk = 256, all scores equal."""
    spec = workloads.small_spec("e", 503, "bf16", "bf16", R=3, len_range=(1, 40000), topk=6)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    kw = oracle_kwargs(b)
    for topk, init, local in [(3, 1, 2), (256, 1, 4), (1, 0, 0), (2, 2, 0)]:
        out = _gpu.run(b, planes=planes, topk=topk, init_blocks=init, local_blocks=local)
        ref = oracle.index.index_step(**dict(kw, topk=topk, init_blocks=init, local_blocks=local))
        _check_all_rows(b, out, ref, init, local)
    # all keys zero -> every block max is 0: ties resolve to the lowest ids
    zp = torch.zeros_like(b.payload).cuda()
    out = _gpu.run(b, planes=(zp, None), topk=8, init_blocks=1, local_blocks=1)
    zkw = dict(kw, payload=np.zeros_like(kw["payload"]), topk=8, init_blocks=1, local_blocks=1)
    ref = oracle.index.index_step(**zkw)
    assert np.array_equal(out.ids, ref.ids)


def test_warp_rows_with_all_scores_equal():
    """Enough short rows for the warp-per-row top-k (3200 rows of at most 157
    blocks) with every key zero, so every block score ties: each row must
    choose the lowest ids, in id order."""
    spec = workloads.small_spec("wz", 505, "bf16", "bf16", R=200, len_range=(1, 20000), topk=20)
    b = workloads.make_batch(spec)
    zp = torch.zeros_like(b.payload).cuda()
    out = _gpu.run(b, planes=(zp, None))
    zkw = dict(oracle_kwargs(b), payload=np.zeros_like(np_u8(b.payload)))
    ref = oracle.index.index_step(**zkw)
    assert np.array_equal(out.ids, ref.ids)


@pytest.mark.parametrize("P,G,grid", [(4, 4, 0), (40, 4, 0), (40, 4, 1)])
def test_bad_page_ids_are_flagged_not_read(P, G, grid):
    """Page ids outside the pool are flagged and not read, on the 16-row path
    and on the tensor-core path; with one CTA the late bad page sits in a later
    batch of the producer's page lookups than the first."""
    import sparse_attention_indexer_packed_gb300 as idx
    spec = workloads.small_spec("bp", 504, "fp8_e4m3", "fp8_e4m3", R=2, P=P, G=G,
                                len_range=(3000, 4000))
    b = workloads.make_batch(spec)
    pt = b.page_table.clone()
    pt[int(b.slot_ids[0]), 3] = b.num_pages + 5
    pt[int(b.slot_ids[1]), 0] = -7
    pt[int(b.slot_ids[1]), 45] = b.num_pages
    try:
        idx.idx_set_grid_limit(grid)
        out = _gpu.run(b, page_table=pt)
    finally:
        idx.idx_set_grid_limit(0)
    assert out.flags & 1


def test_rows_longer_than_the_page_table_are_clamped():
    spec = workloads.small_spec("cl", 505, "bf16", "bf16", R=2, explicit_lens=[[100, 200, 300, 400]] * 2)
    b = workloads.make_batch(spec)
    b.row_lens[1, 3] = b.max_pages * 64 + 500
    out = _gpu.run(b)
    assert out.flags & 4
    b.row_lens[1, 3] = b.max_pages * 64
    ref = oracle.index.index_step(**oracle_kwargs(b))
    _check_all_rows(b, out, ref)


@pytest.mark.parametrize("k_dtype,q_dtype", [("bf16", "bf16"), ("fp8_e4m3", "fp8_e4m3"),
                                             ("nvfp4", "bf16")])
def test_results_do_not_depend_on_the_grid(k_dtype, q_dtype):
    """Few CTAs force many blocks (and request boundaries) through each CTA's
    stage ring; the outputs must be bitwise the same as with one CTA per SM,
    and match the oracle."""
    import sparse_attention_indexer_packed_gb300 as idx
    spec = workloads.small_spec("grid", 601, k_dtype, q_dtype, R=7, len_range=(1, 30000), topk=24,
                                pad_requests=(2,))
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    base = _gpu.run(b, planes=planes)
    ref = oracle.index.index_step(**oracle_kwargs(b))
    _check_all_rows(b, base, ref)
    try:
        for lim in (1, 3, 13):
            idx.idx_set_grid_limit(lim)
            o = _gpu.run(b, planes=planes)
            assert o.flags == 0, (lim, hex(o.flags))
            assert np.array_equal(o.ids, base.ids), lim
            assert np.array_equal(o.scores.view(np.uint32), base.scores.view(np.uint32)), lim
    finally:
        idx.idx_set_grid_limit(0)


def test_batch_invariance_of_a_request():
    """A request's outputs are bitwise the same whatever the other requests in
    the batch are (reduction order never depends on the batch)."""
    spec = workloads.small_spec("bi", 602, "bf16", "bf16", R=6, len_range=(500, 20000), topk=16)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    a = _gpu.run(b, planes=planes)
    b2 = workloads.make_batch(spec)
    g = torch.Generator().manual_seed(5)
    b2.q[1:] = torch.randn(b2.q[1:].shape, generator=g).to(torch.bfloat16)
    b2.row_lens[2:] = torch.randint(1, 20000, b2.row_lens[2:].shape, generator=g, dtype=torch.int32)
    o = _gpu.run(b2, planes=planes)
    assert np.array_equal(a.ids[0], o.ids[0])
    assert np.array_equal(a.scores[0].view(np.uint32), o.scores[0].view(np.uint32))


@pytest.mark.parametrize("topk,max_len", [(16, 9000), (100, 20000)])
def test_topk_warp_rows_match_cta_rows(topk, max_len):
    """Many rows of at most 256 blocks (here 4 prefill-like requests of 256
    query tokens x 4 heads: 4096 rows) take the warp-per-row top-k; the same
    rows behind a page table wider than 512 pages take the CTA-per-row one.
    Both must give the oracle's selection and agree bit for bit, including rows
    whose scores are all equal (zero queries: every tie goes to the lower id).
    A budget of 16 blocks orders its chosen entries by the in-register sort
    (at most 64), one of 100 over rows of up to 157 blocks by the rank count."""
    spec = workloads.small_spec("tk", 501, "bf16", "bf16", R=4, P=256, G=4,
                                len_range=(300, max_len), topk=topk)
    b = workloads.make_batch(spec)
    b.q[1] = 0                      # request 1: every block score 0
    b.q[2, 7, 1] = 0                # one row of request 2
    planes = _gpu.device_planes(b)
    warp = _gpu.run(b, planes=planes)
    wide_pt = torch.cat([b.page_table, b.page_table[:, :1].repeat(1, 600)], dim=1)
    cta = _gpu.run(b, planes=planes, page_table=wide_pt)
    assert warp.flags == 0 and cta.flags == 0
    assert np.array_equal(warp.ids, cta.ids)
    assert np.array_equal(warp.scores.view(np.uint32), cta.scores.view(np.uint32))
    ref = oracle.index.index_step(**oracle_kwargs(b))
    _check_all_rows(b, warp, ref)


@pytest.mark.parametrize("k_dtype,q_dtype,P,G", [("bf16", "bf16", 4, 4), ("bf16", "bf16", 40, 4),
                                                 ("bf16", "bf16", 8, 8),
                                                 ("fp8_e4m3", "fp8_e4m3", 8, 8),
                                                 ("nvfp4", "bf16", 40, 4),
                                                 ("nvfp4", "bf16", 8, 8)])
def test_wait_timeout_is_reported_and_the_context_survives(k_dtype, q_dtype, P, G):
    """A wait that nothing completes (the stall test: one role per score CTA
    waits on a barrier no one arrives at, with a 20 ms limit) must end the call
    through the timeout path -- copies in flight waited for, TMEM freed,
    IDX_DEVERR_TIMEOUT in the workspace -- instead of hanging or faulting, and
    the next call must be exact again.  P x G = 40 x 4 takes the tensor-core
    path, whose other roles then also run out of their waits; 8 x 8 is one
    tile per request there, whose query slots alternate."""
    import sparse_attention_indexer_packed_gb300 as idx
    spec = workloads.small_spec("to", 701, k_dtype, q_dtype, R=4, P=P, G=G,
                                len_range=(2000, 9000), topk=16)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    try:
        idx.idx_set_wait_limit_ns(20_000_000)
        idx.idx_set_stall_test(True)
        bad = _gpu.run(b, planes=planes)
    finally:
        idx.idx_set_stall_test(False)
        idx.idx_set_wait_limit_ns(0)
    assert bad.flags & 2, f"expected IDX_DEVERR_TIMEOUT, flags {bad.flags:#x}"
    good = _gpu.run(b, planes=planes)
    assert good.flags == 0
    ref = oracle.index.index_step(**oracle_kwargs(b))
    _check_all_rows(b, good, ref)


def test_kernel_waits_order_a_pipelined_step():
    """idx_set_kernel_waits: inputs copied on another stream behind a long
    kernel.  Waited for before the score kernel, or before the previous call's
    top-k (the next call's score kernel reads its inputs only after that top-k),
    the results equal the plain call's bit for bit; the inputs' buffers hold
    zeros until the copies land, so a wait that is not honoured shows."""
    import sparse_attention_indexer_packed_gb300 as idx
    spec = workloads.small_spec("kw", 611, "bf16", "bf16", R=5, len_range=(2000, 12000), topk=24)
    b = workloads.make_batch(spec)
    planes = _gpu.device_planes(b)
    ref = _gpu.run(b, planes=planes)
    dev = "cuda"
    s = b.spec
    pt, sl, ln = b.page_table.to(dev), b.slot_ids.to(dev), b.row_lens.to(dev)
    q_host = b.q.pin_memory()
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()

    def out_bufs():
        return (torch.full((b.R, b.M, s.topk), 77, dtype=torch.int32, device=dev),
                torch.full((b.R, b.M, s.topk), 77.0, dtype=torch.float32, device=dev))

    def call(q, ids, sc, ws):
        idx.idx_score_topk(q, None, planes[0], planes[1], s.k_dtype, pt, sl, ln,
                           s.packed_queries, s.gqa, s.init_blocks, s.local_blocks, s.topk,
                           ids, sc, ws, main)

    def staged_copy(q_dev):
        ev = torch.cuda.Event()
        side.wait_stream(main)                  # after the buffer's zero fill
        with torch.cuda.stream(side):
            torch.cuda._sleep(20_000_000)       # ~10 ms of spinning before the copy
            q_dev.copy_(q_host, non_blocking=True)
            ev.record(side)
        return ev

    ws1 = idx.alloc_workspace(b.R, s.packed_queries, s.gqa, b.max_pages)
    ws2 = idx.alloc_workspace(b.R, s.packed_queries, s.gqa, b.max_pages)
    # before the score kernel
    q1 = torch.zeros_like(b.q, device=dev)
    ev1 = staged_copy(q1)
    ids1, sc1 = out_bufs()
    idx.idx_set_kernel_waits(ev1, None)
    call(q1, ids1, sc1, ws1)
    # before the previous call's top-k
    q2 = torch.zeros_like(b.q, device=dev)
    ev2 = staged_copy(q2)
    ids0, sc0 = out_bufs()
    idx.idx_set_kernel_waits(None, ev2)
    call(b.q.to(dev), ids0, sc0, ws1)
    ids2, sc2 = out_bufs()
    call(q2, ids2, sc2, ws2)
    torch.cuda.synchronize()
    for ids, sc in [(ids1, sc1), (ids0, sc0), (ids2, sc2)]:
        assert np.array_equal(ids.cpu().numpy(), ref.ids)
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), ref.scores.view(np.uint32))

"""The id-set rule the GPU parity tests apply (tests/_util.compare_row), checked
on hand-made rows: top-k ids must equal the oracle's except where the oracle's
k-th and (k+1)-th candidate scores lie within 1e-3 (1 + |s|), and then only in
candidates within that tolerance of the k-th."""
import numpy as np

from _util import compare_row, near_tie_violation


def _ref(bm, topk, init=0, local=0):
    import oracle
    return oracle.index.select_row(np.asarray(bm, dtype=np.float64), init, local, topk)


def _dev(ids, bm, topk):
    ids = list(ids) + [-1] * (topk - len(ids))
    sc = [bm[i] if i >= 0 else -np.inf for i in ids]
    return np.array(ids), np.array(sc)


def test_identical_selection_passes():
    bm = np.array([5.0, 4.0, 3.0, 2.0, 1.0])
    ri, rs = _ref(bm, 3)
    assert compare_row(ri, rs, ri, rs, bm, 0, 0) is None


def test_swap_at_a_near_tie_passes():
    bm = np.array([5.0, 4.0, 3.0005, 3.0, 1.0])
    ri, rs = _ref(bm, 3)
    di, ds = _dev([0, 1, 3], bm, 3)
    assert compare_row(di, ds, ri, rs, bm, 0, 0) is None


def test_swap_without_a_near_tie_fails():
    bm = np.array([5.0, 4.0, 3.1, 3.0, 1.0])
    ri, rs = _ref(bm, 3)
    di, ds = _dev([0, 1, 3], bm, 3)
    assert "not within tolerance" in compare_row(di, ds, ri, rs, bm, 0, 0)


def test_swap_past_the_band_fails_even_with_a_near_tie():
    # k-th 3.0 and (k+1)-th 2.997 are within 0.004, but block 4 (2.993) is 0.007
    # from the k-th: a rule of twice the tolerance would have let it through
    bm = np.array([5.0, 4.0, 3.0, 2.997, 2.993])
    ri, rs = _ref(bm, 3)
    di, ds = _dev([0, 1, 4], bm, 3)
    assert "beyond the near tie" in compare_row(di, ds, ri, rs, bm, 0, 0)


def test_far_block_swapped_in_fails():
    bm = np.array([5.0, 4.0, 3.0005, 3.0, 1.0])
    ri, rs = _ref(bm, 3)
    di, ds = _dev([0, 1, 4], bm, 3)
    assert compare_row(di, ds, ri, rs, bm, 0, 0) is not None


def test_forced_blocks_are_not_candidates():
    # block 4 is forced (local 1); the candidates' k-th / (k+1)-th tie is
    # between blocks 2 and 3
    bm = np.array([5.0, 4.0, 3.0005, 3.0, -9.0])
    ri, rs = _ref(bm, 3, local=1)
    assert set(ri[ri >= 0].tolist()) == {0, 1, 4}
    di, ds = _dev([4, 0, 2], bm, 3)
    assert compare_row(di, ds, ri, rs, bm, 0, 1) is not None   # 1 (4.0) is not near 3.0005
    bm2 = np.array([5.0, 3.0004, 3.0005, 3.0, -9.0])
    ri2, rs2 = _ref(bm2, 3, local=1)
    di2, ds2 = _dev([4, 0, 1], bm2, 3)
    assert compare_row(di2, ds2, ri2, rs2, bm2, 0, 1) is None


def test_no_unchosen_candidate_means_exact():
    bm = np.array([5.0, 4.0])
    assert near_tie_violation(bm, [0, 1], 2, {1}) is not None
    assert near_tie_violation(bm, [0, 1], 0, {1}) is not None
    assert near_tie_violation(bm, [0, 1], 1, set()) is None

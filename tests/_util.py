"""Shared test helpers: turn a synthetic batch into the oracle's numpy inputs
and compare CUDA-path outputs with the oracle's."""
import numpy as np

from oracle.inputs import np_bits16, np_u8  # noqa: F401  (re-exported for the tests)
from oracle.inputs import planes as _planes
from oracle.inputs import step_kwargs as _step_kwargs


def oracle_planes(batch, requests=None):
    """Pool planes as the oracle sees them (oracle.inputs.planes)."""
    return _planes(batch, requests=requests)


def oracle_kwargs(batch, planes=None):
    """index_step's arguments for the batch (oracle.inputs.step_kwargs)."""
    return _step_kwargs(batch, pool_planes=planes)


def score_tol(s):
    """|delta| <= 1e-3 * (1 + |s|), the block-score tolerance."""
    return 1e-3 * (1.0 + np.abs(s))


def near_tie_violation(bm, cands, c, diff, tol=score_tol):
    """The id-set rule for a selection of c blocks from ``cands``.

    cands: candidate block ids (forced blocks excluded); c: how many of them
    the oracle chose; diff: the ids on which the two selections differ.  The
    sets may differ only where the oracle's k-th and (k+1)-th candidates (its
    last chosen and its best unchosen one, ranked by score desc, id asc) lie
    within tolerance of each other, and then only in candidates whose oracle
    score lies within tolerance of the k-th's.  Returns an error string or
    None."""
    if not diff:
        return None
    order = sorted(cands, key=lambda b: (-bm[b], b))
    if c <= 0 or c >= len(order):
        return f"id sets differ with no unchosen candidate to tie with: {sorted(diff)}"
    s_k, s_k1 = float(bm[order[c - 1]]), float(bm[order[c]])
    t = float(tol(s_k))
    if abs(s_k - s_k1) > t:
        return (f"id sets differ {sorted(diff)} but the k-th and (k+1)-th scores "
                f"{s_k} and {s_k1} are not within tolerance")
    for b in diff:
        if abs(float(bm[b]) - s_k) > t:
            return f"id sets differ beyond the near tie at block {b}: {bm[b]} vs k-th {s_k}"
    return None


def compare_row(ids_dev, sc_dev, ids_ref, sc_ref, blockmax_ref, init_blocks, local_blocks):
    """Compare one row's top-k output against the oracle.

    IDs must be equal as sets, except where the oracle's k-th and (k+1)-th
    candidate scores lie within tolerance (near_tie_violation).  Every emitted
    id's score must be within tolerance of the oracle's block score for that
    id.  Returns an error string or None.
    """
    ids_dev = np.asarray(ids_dev, dtype=np.int64)
    sc_dev = np.asarray(sc_dev, dtype=np.float64)
    ids_ref = np.asarray(ids_ref, dtype=np.int64)
    n_ref = int((ids_ref >= 0).sum())
    n_dev = int((ids_dev >= 0).sum())
    if n_ref != n_dev:
        return f"count {n_dev} != {n_ref}"
    if np.any(ids_dev[n_dev:] != -1) or np.any(np.isfinite(sc_dev[n_dev:])):
        return "pad tail is not (-1, -inf)"
    if n_ref == 0:
        return None
    dev = ids_dev[:n_dev]
    if len(set(dev.tolist())) != n_dev:
        return "duplicate ids"
    bm = blockmax_ref
    nb = len(bm)
    if dev.min() < 0 or dev.max() >= nb:
        return "id out of range"
    err = np.abs(sc_dev[:n_dev] - bm[dev])
    if np.any(err > score_tol(bm[dev])):
        k = int(np.argmax(err - score_tol(bm[dev])))
        return f"score of block {dev[k]}: {sc_dev[k]} vs {bm[dev[k]]}"
    ref = set(ids_ref[:n_ref].tolist())
    got = set(dev.tolist())
    if ref == got:
        return None
    forced = set(range(min(init_blocks, nb))) | set(range(max(0, nb - local_blocks), nb))
    if not forced <= got:
        return "a forced block is missing"
    cands = [b for b in range(nb) if b not in forced]
    return near_tie_violation(bm, cands, n_ref - len(forced & ref), got ^ ref)

"""Shared test helpers: turn a synthetic batch into the oracle's numpy inputs
and compare CUDA-path outputs with the oracle's."""
import numpy as np
import torch


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy()


def np_bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_planes(batch, requests=None):
    """Pool planes as the oracle sees them.  For NVFP4 the oracle quantises the
    bf16 staging keys itself (never reading bytes the CUDA path wrote); with
    ``requests`` only those requests' keys are quantised."""
    import oracle
    payload = np_u8(batch.payload).copy()
    scale = None if batch.scale is None else np_u8(batch.scale).copy()
    if batch.spec.k_dtype == "nvfp4" and batch.staging is not None and batch.staging.numel():
        if requests is None:
            sel = slice(None)
            stage = batch.staging
            rows = batch.slot_mapping.numpy()
        else:
            lens = batch.group_lens()
            idx = [np.arange(batch.staging_offsets[r], batch.staging_offsets[r] + lens[r])
                   for r in requests if batch.staging_offsets[r] >= 0]
            sel = np.concatenate(idx) if idx else np.zeros(0, np.int64)
            stage = batch.staging[torch.from_numpy(sel)]
            rows = batch.slot_mapping.numpy()[sel]
        pay, sc = oracle.formats.nvfp4_quantize(np_bits16(stage))
        keep = rows >= 0
        payload[rows[keep]] = pay[keep]
        scale[rows[keep]] = sc[keep]
    return payload, scale


def oracle_kwargs(batch, planes=None):
    payload, scale = planes if planes is not None else oracle_planes(batch)
    if batch.spec.q_dtype == "bf16":
        q = np_bits16(batch.q)
    else:
        q = np_u8(batch.q)
    return dict(q=q, q_dtype=batch.spec.q_dtype,
                q_scale=None if batch.q_scale is None else batch.q_scale.numpy().astype(np.float64),
                payload=payload, scale=scale, k_dtype=batch.spec.k_dtype,
                page_table=batch.page_table.numpy(), slot_ids=batch.slot_ids.numpy(),
                row_lens=batch.row_lens.numpy(), packed_queries=batch.spec.packed_queries,
                gqa=batch.spec.gqa, init_blocks=batch.spec.init_blocks,
                local_blocks=batch.spec.local_blocks, topk=batch.spec.topk)


def score_tol(s):
    """|delta| <= 1e-3 * (1 + |s|), the block-max score tolerance."""
    return 1e-3 * (1.0 + np.abs(s))


def compare_row(ids_dev, sc_dev, ids_ref, sc_ref, blockmax_ref, init_blocks, local_blocks):
    """Compare one row's top-k output against the oracle.

    IDs must be equal as sets, except that where the oracle's last-chosen and
    best-unchosen candidate scores lie within tolerance, any choice among the
    near-tied candidates is accepted.  Every emitted id's score must be within
    tolerance of the oracle's block max for that id.  Returns an error string
    or None.
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
    # near-tie exemption: differing ids must all be candidates whose oracle score is
    # within tolerance of the selection threshold
    forced = set(range(min(init_blocks, nb))) | set(range(max(0, nb - local_blocks), nb))
    if not forced <= got:
        return "a forced block is missing"
    chosen = [b for b in ref if b not in forced]
    if not chosen:
        return f"id sets differ: {sorted(got ^ ref)}"
    thr = min(bm[b] for b in chosen)
    for b in got ^ ref:
        if abs(bm[b] - thr) > 2 * score_tol(thr):
            return f"id sets differ beyond a near tie at block {b}: {bm[b]} vs threshold {thr}"
    return None

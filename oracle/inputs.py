"""The oracle's view of a seeded synthetic batch.

TEST INFRASTRUCTURE ONLY (see the package docstring): the tests and the CPU
baseline / reference leg of the benchmark turn a ``workloads.Batch`` (torch
tensors on the host) into the plain numpy arguments of ``index.index_step``.

Nothing here is read from the CUDA path.  For NVFP4 keys the oracle quantises
the batch's bf16 staging keys with its own quantiser (``formats``) and places
them at their slots, so it never sees bytes the GPU store wrote.  torch is
imported lazily, only to view the batch's tensors as numpy arrays; importing
``oracle`` itself still needs numpy alone.
"""
from __future__ import annotations

import numpy as np

from . import formats

_QUANT_CHUNK = 1 << 16  # keys quantised at a time


def np_u8(t) -> np.ndarray:
    """A host tensor's bytes as uint8."""
    import torch
    return t.contiguous().view(torch.uint8).numpy()


def np_bits16(t) -> np.ndarray:
    """A host bf16 tensor's bit patterns as uint16."""
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def planes(batch, requests=None):
    """Pool planes (payload, scale) as the oracle sees them.  For NVFP4 the
    staged bf16 keys are quantised here by the oracle; with ``requests`` only
    those requests' keys are quantised (the rest of the plane keeps the batch's
    filler bytes)."""
    import torch
    payload = np_u8(batch.payload).copy()
    scale = None if batch.scale is None else np_u8(batch.scale).copy()
    if batch.spec.k_dtype == "nvfp4" and batch.staging is not None and batch.staging.numel():
        if requests is None:
            stage = batch.staging
            rows = batch.slot_mapping.numpy()
        else:
            lens = batch.group_lens()
            idx = [np.arange(batch.staging_offsets[r], batch.staging_offsets[r] + lens[r])
                   for r in requests if batch.staging_offsets[r] >= 0]
            sel = np.concatenate(idx) if idx else np.zeros(0, np.int64)
            stage = batch.staging[torch.from_numpy(sel)]
            rows = batch.slot_mapping.numpy()[sel]
        # in bounded chunks of keys: the quantiser works on float arrays
        bits = np_bits16(stage)
        for a in range(0, len(rows), _QUANT_CHUNK):
            pay, sc = formats.nvfp4_quantize(bits[a:a + _QUANT_CHUNK])
            rr = rows[a:a + _QUANT_CHUNK]
            keep = rr >= 0
            payload[rr[keep]] = pay[keep]
            scale[rr[keep]] = sc[keep]
    return payload, scale


def step_kwargs(batch, pool_planes=None) -> dict:
    """Keyword arguments of ``index.index_step`` for the whole batch."""
    payload, scale = pool_planes if pool_planes is not None else planes(batch)
    q = np_bits16(batch.q) if batch.spec.q_dtype == "bf16" else np_u8(batch.q)
    return dict(q=q, q_dtype=batch.spec.q_dtype,
                q_scale=None if batch.q_scale is None else batch.q_scale.numpy().astype(np.float64),
                payload=payload, scale=scale, k_dtype=batch.spec.k_dtype,
                page_table=batch.page_table.numpy(), slot_ids=batch.slot_ids.numpy(),
                row_lens=batch.row_lens.numpy(), packed_queries=batch.spec.packed_queries,
                gqa=batch.spec.gqa, init_blocks=batch.spec.init_blocks,
                local_blocks=batch.spec.local_blocks, topk=batch.spec.topk)

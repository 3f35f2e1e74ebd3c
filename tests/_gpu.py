"""Run the CUDA path (through the C ABI binding) on a synthetic batch."""
import dataclasses

import numpy as np
import torch

import sparse_attention_indexer_packed_gb300 as idx


@dataclasses.dataclass
class GpuOut:
    ids: np.ndarray
    scores: np.ndarray
    flags: int
    payload: torch.Tensor
    scale: torch.Tensor
    blockmax: np.ndarray    # [R*M, nb_cap] from the workspace (rows' own blocks only are defined)


def device_planes(batch, dev="cuda"):
    """Pool planes on the device; NVFP4 keys are written by the store kernel."""
    payload = batch.payload.to(dev)
    scale = None if batch.scale is None else batch.scale.to(dev)
    if batch.spec.k_dtype == "nvfp4" and batch.staging is not None and batch.staging.numel():
        idx.idx_store_nvfp4(batch.staging.to(dev), batch.slot_mapping.to(dev), (payload, scale))
    return payload, scale


def run(batch, perrow=False, planes=None, dev="cuda", topk=None, init_blocks=None,
        local_blocks=None, page_table=None, block_score="max", row_lens=None):
    s = batch.spec
    topk = s.topk if topk is None else topk
    init_blocks = s.init_blocks if init_blocks is None else init_blocks
    local_blocks = s.local_blocks if local_blocks is None else local_blocks
    payload, scale = planes if planes is not None else device_planes(batch, dev)
    q = batch.q.to(dev)
    q_scale = None if batch.q_scale is None else batch.q_scale.to(dev)
    pt = (batch.page_table if page_table is None else page_table).to(dev)
    R, M = batch.R, batch.M
    out_ids = torch.full((R, M, topk), 7777, dtype=torch.int32, device=dev)
    out_sc = torch.full((R, M, topk), 7777.0, dtype=torch.float32, device=dev)
    ws = idx.alloc_workspace(R, s.packed_queries, s.gqa, int(pt.shape[1]), device=dev)
    if block_score == "lse":
        assert not perrow
        fn = idx.idx_score_topk_lse
    else:
        fn = idx.idx_score_topk_perrow if perrow else idx.idx_score_topk
    lens = batch.row_lens.to(dev) if row_lens is None else row_lens
    fn(q, q_scale, payload, scale, s.k_dtype, pt, batch.slot_ids.to(dev), lens,
       s.packed_queries, s.gqa, init_blocks, local_blocks, topk, out_ids, out_sc, ws)
    flags = idx.idx_workspace_errors(ws)
    torch.cuda.synchronize()
    nb_cap = (int(pt.shape[1]) + 1) // 2
    bm = ws[1024:1024 + R * M * nb_cap * 4].view(torch.float32).reshape(R * M, nb_cap).cpu().numpy() \
        if R * M else np.zeros((0, nb_cap), np.float32)
    return GpuOut(ids=out_ids.cpu().numpy(), scores=out_sc.cpu().numpy(), flags=flags,
                  payload=payload, scale=scale, blockmax=bm)

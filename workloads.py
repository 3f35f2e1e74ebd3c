"""Seeded synthetic inputs for the packed index-score + block top-k step.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no scoring, no NVFP4 quantisation, no selection).  Both the
CPU oracle tests and the CUDA path's tests and benchmark take their inputs from
here, so the two sides always see the same bytes.

Workload shapes follow the pages' benchmarks: sglang #45451 "Speed Tests and
Profiling" (16 req x 131K and 32 req x 524K, bf16 and fp8 index K), the verify
test of sglang #42614 "[AMD] MiniMax-M3 indexer CP: packed scoring for EAGLE
verify rows" (Accuracy Tests: 4 requests x 4 draft rows ending at 32767..32770,
permuted gapped slots), and ROCm/ATOM #2745 "Validation" (NVFP4 index, bs64 at
~150K context).  The pages measure on serving traces and weights that are not
available; these generators stand in for them with N(0,1) keys and queries.

Layout conventions (shared with the C ABI header, restated here as data):
  * page size 64 tokens, head dim D = 128, block = 128 tokens;
  * payload plane: uint8 [num_pages * 64, row_bytes], row = page * 64 + t % 64,
    row_bytes = 256 (bf16), 128 (fp8 e4m3), 64 (NVFP4);
  * scale plane: uint8 [num_pages * 64, scale_bytes], scale_bytes = 0 (bf16),
    4 (fp8: one little-endian fp32 per key), 8 (NVFP4: one E4M3 byte per 16 dims);
  * q: [R, P, G, D] (bf16, or e4m3 codes as uint8) with q_scale fp32 [R, P*G]
    for e4m3 q; packed row i of a request is (draft row i // G, head i % G);
  * page_table int32 [n_slots, max_pages]; slot_ids int32 [R];
    row_lens int32 [R, P].
"""
from __future__ import annotations

import dataclasses
import math
import os
from typing import Optional

import torch

PAGE = 64
BLOCK = 128
DIM = 128

ROW_BYTES = {"bf16": 256, "fp8_e4m3": 128, "nvfp4": 64}
SCALE_BYTES = {"bf16": 0, "fp8_e4m3": 4, "nvfp4": 8}


@dataclasses.dataclass
class Spec:
    """Recipe for one synthetic batch (all sizes in tokens unless stated)."""

    name: str
    seed: int
    k_dtype: str                 # "bf16" | "fp8_e4m3" | "nvfp4"
    q_dtype: str                 # "bf16" | "fp8_e4m3"
    num_requests: int
    packed_queries: int          # P, draft rows per request
    gqa: int                     # G, heads per draft row
    init_blocks: int
    local_blocks: int
    topk: int
    # Row lengths: either explicit per-request lists, or a uniform range for the
    # request's longest row with row j of P having length L - (P - 1) + j.
    explicit_lens: Optional[list] = None
    len_range: Optional[tuple] = None
    junk_page_frac: float = 0.125    # extra physical pages holding garbage
    pad_requests: tuple = ()         # request indices given a pad (out of range) slot
    max_pages: Optional[int] = None  # page-table width; default = longest row's pages


@dataclasses.dataclass
class Batch:
    spec: Spec
    q: torch.Tensor                   # bf16 [R,P,G,D] or uint8 e4m3 codes
    q_scale: Optional[torch.Tensor]   # fp32 [R, P*G] (e4m3 q) else None
    num_pages: int
    payload: torch.Tensor             # uint8 [num_pages*64, row_bytes]
    scale: Optional[torch.Tensor]     # uint8 [num_pages*64, scale_bytes] or None
    staging: Optional[torch.Tensor]   # bf16 [T, D] keys to store (NVFP4 only)
    slot_mapping: Optional[torch.Tensor]  # int64 [T] physical row per staged key
    page_table: torch.Tensor          # int32 [n_slots, max_pages]
    slot_ids: torch.Tensor            # int32 [R]
    row_lens: torch.Tensor            # int32 [R, P]
    staging_offsets: Optional[list] = None  # first staged row of each request (-1: pad)

    @property
    def R(self) -> int:
        return self.spec.num_requests

    @property
    def M(self) -> int:
        return self.spec.packed_queries * self.spec.gqa

    @property
    def n_slots(self) -> int:
        return int(self.page_table.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    def group_lens(self) -> list:
        """Longest row of each request (0 for a pad request)."""
        out = []
        for r in range(self.R):
            s = int(self.slot_ids[r])
            if s < 0 or s >= self.n_slots:
                out.append(0)
            else:
                out.append(max(0, int(self.row_lens[r].max())))
        return out

    def k_bytes_read(self) -> int:
        """Index-K bytes a once-per-request read of every needed page moves."""
        per_tok = ROW_BYTES[self.spec.k_dtype] + SCALE_BYTES[self.spec.k_dtype]
        return sum(min(L, self.max_pages * PAGE) for L in self.group_lens()) * per_tok


_CHUNK = 1 << 16   # rows drawn by one chunk generator


def _chunked(gen: torch.Generator, n: int, fill) -> None:
    """Run fill(chunk_generator, a, b) over rows [a, b) in chunks of _CHUNK rows,
    on a thread pool.  Every chunk draws from its own generator, seeded from one
    number taken from `gen`, so the bytes do not depend on the thread count."""
    from concurrent.futures import ThreadPoolExecutor
    base = int(torch.randint(0, 2 ** 62, (1,), generator=gen))
    spans = [(c, a, min(n, a + _CHUNK)) for c, a in enumerate(range(0, n, _CHUNK))]

    def one(span):
        c, a, b = span
        fill(torch.Generator().manual_seed((base + 1000003 * c) % (2 ** 63)), a, b)

    if len(spans) <= 1:
        for sp in spans:
            one(sp)
        return
    with ThreadPoolExecutor(max_workers=min(len(spans), os.cpu_count() or 1)) as ex:
        list(ex.map(one, spans))


def _e4m3_rows(gen: torch.Generator, n: int):
    """n vectors v ~ N(0,1)^D, each scaled so its amax maps to 448.

    Returns (codes uint8 [n, D], scale fp32 [n]) with value = code * scale.
    The cast to e4m3 is torch's own float8_e4m3fn conversion.
    """
    codes = torch.empty((n, DIM), dtype=torch.uint8)
    scales = torch.empty((n,), dtype=torch.float32)

    def fill(g, a, b):
        v = torch.randn((b - a, DIM), generator=g, dtype=torch.float32)
        amax = v.abs().amax(dim=1).clamp_min(1e-30)
        x = (v * (448.0 / amax)[:, None]).clamp(-448.0, 448.0)
        codes[a:b] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        scales[a:b] = amax / 448.0

    _chunked(gen, n, fill)
    return codes, scales


def _bf16_rows(gen: torch.Generator, n: int) -> torch.Tensor:
    out = torch.empty((n, DIM), dtype=torch.bfloat16)

    def fill(g, a, b):
        out[a:b] = torch.randn((b - a, DIM), generator=g, dtype=torch.float32).to(torch.bfloat16)

    _chunked(gen, n, fill)
    return out


def _byte_rows(gen: torch.Generator, n: int, width: int, hi: int) -> torch.Tensor:
    """uint8 [n, width], each byte uniform in [0, hi)."""
    out = torch.empty((n, width), dtype=torch.uint8)

    def fill(g, a, b):
        out[a:b] = torch.randint(0, hi, (b - a, width), generator=g, dtype=torch.uint8)

    _chunked(gen, n, fill)
    return out


def make_batch(spec: Spec) -> Batch:
    gen = torch.Generator().manual_seed(spec.seed)
    R, P, G = spec.num_requests, spec.packed_queries, spec.gqa

    # ---- row lengths -------------------------------------------------------
    if spec.explicit_lens is not None:
        row_lens = torch.tensor(spec.explicit_lens, dtype=torch.int32).reshape(R, P)
    else:
        lo, hi = spec.len_range
        L = torch.randint(lo, hi + 1, (R,), generator=gen, dtype=torch.int64)
        j = torch.arange(P, dtype=torch.int64)
        row_lens = (L[:, None] - (P - 1) + j[None, :]).clamp_min(0).to(torch.int32)
    longest = [int(row_lens[r].max()) for r in range(R)]
    pages_needed = [max(0, math.ceil(x / PAGE)) for x in longest]
    max_pages = spec.max_pages or max(1, max(pages_needed))

    # ---- slots: permuted, gapped, never equal to the request index ---------
    n_slots = 2 * R + 2
    perm = torch.randperm(n_slots, generator=gen).tolist()
    slot_ids = []
    for r in range(R):
        pick = next(s for s in perm if s != r and s not in slot_ids)
        slot_ids.append(pick)
    for r in spec.pad_requests:
        slot_ids[r] = -1 if (r % 2 == 0) else n_slots + 3   # both kinds of pad
    slot_ids_t = torch.tensor(slot_ids, dtype=torch.int32)

    # ---- physical pages: one global random permutation ---------------------
    used = sum(pages_needed[r] for r in range(R) if r not in spec.pad_requests)
    junk = max(8, int(used * spec.junk_page_frac))
    num_pages = used + junk
    phys = torch.randperm(num_pages, generator=gen).to(torch.int32)
    junk_ids = phys[used:]
    page_table = junk_ids[torch.randint(0, junk, (n_slots, max_pages), generator=gen)].clone()
    cursor = 0
    for r in range(R):
        if r in spec.pad_requests:
            continue
        n = pages_needed[r]
        page_table[slot_ids[r], :n] = phys[cursor:cursor + n]
        cursor += n

    # ---- pool contents: every row random, so a misaddressed read shows -----
    rows = num_pages * PAGE
    staging = slot_mapping = None
    staging_offsets = None
    if spec.k_dtype == "bf16":
        payload = _bf16_rows(gen, rows).view(torch.uint8).reshape(rows, 256)
        scale = None
    elif spec.k_dtype == "fp8_e4m3":
        codes, sc = _e4m3_rows(gen, rows)
        payload = codes
        scale = sc.view(torch.uint8).reshape(rows, 4).clone()
    elif spec.k_dtype == "nvfp4":
        payload = _byte_rows(gen, rows, 64, 256)
        # junk scale bytes stay finite: 0x7F / 0xFF are the E4M3 NaN codes
        scale = _byte_rows(gen, rows, 8, 0x7F)
        # the step's keys arrive as bf16 token-major staging + a slot mapping
        maps = []
        staging_offsets = []
        pos = 0
        for r in range(R):
            if r in spec.pad_requests:
                staging_offsets.append(-1)
                continue
            staging_offsets.append(pos)
            pos += longest[r]
            t = torch.arange(longest[r], dtype=torch.int64)
            pg = page_table[slot_ids[r]].to(torch.int64)[t // PAGE]
            maps.append(pg * PAGE + t % PAGE)
        slot_mapping = torch.cat(maps) if maps else torch.zeros(0, dtype=torch.int64)
        staging = _bf16_rows(gen, int(slot_mapping.numel()))
    else:
        raise ValueError(spec.k_dtype)

    # ---- queries -----------------------------------------------------------
    if spec.q_dtype == "bf16":
        q = _bf16_rows(gen, R * P * G).reshape(R, P, G, DIM)
        q_scale = None
    elif spec.q_dtype == "fp8_e4m3":
        codes, sc = _e4m3_rows(gen, R * P * G)
        q = codes.reshape(R, P, G, DIM)
        q_scale = sc.reshape(R, P * G)
    else:
        raise ValueError(spec.q_dtype)

    return Batch(spec=spec, q=q, q_scale=q_scale, num_pages=num_pages, payload=payload,
                 scale=scale, staging=staging, slot_mapping=slot_mapping,
                 page_table=page_table, slot_ids=slot_ids_t, row_lens=row_lens,
                 staging_offsets=staging_offsets)


# ---------------------------------------------------------------------------
# Named workloads.  Seeds 1001..1006 are fixed per workload.
# ---------------------------------------------------------------------------
def _verify_rows(P: int, ends: list) -> list:
    return [e + 1 for e in ends]   # a row that ends at token t has length t + 1


WORKLOADS = {
    # 1 request, 4 draft rows x 4 heads, rows end at tokens 4095..4098 -> 32/33 blocks
    "tiny_bf16_1x4k": Spec("tiny_bf16_1x4k", 1001, "bf16", "bf16", 1, 4, 4, 1, 2, 8,
                           explicit_lens=[_verify_rows(4, [4095, 4096, 4097, 4098])],
                           junk_page_frac=1.0),
    # 16 requests x ~131K (uniform in [120000, 131072]), bf16 K and q
    "bf16_16x131k": Spec("bf16_16x131k", 1002, "bf16", "bf16", 16, 4, 4, 1, 4, 64,
                         len_range=(120000, 131072)),
    # same with fp8 e4m3 K and q (per-token fp32 scales)
    "fp8_16x131k": Spec("fp8_16x131k", 1003, "fp8_e4m3", "fp8_e4m3", 16, 4, 4, 1, 4, 64,
                        len_range=(120000, 131072)),
    "fp8_16x131k_local0": Spec("fp8_16x131k_local0", 1006, "fp8_e4m3", "fp8_e4m3", 16, 4, 4,
                               1, 0, 64, len_range=(120000, 131072)),
    # 32 requests x ~524K (uniform in [500000, 524288]), fp8
    "fp8_32x524k": Spec("fp8_32x524k", 1004, "fp8_e4m3", "fp8_e4m3", 32, 4, 4, 1, 4, 64,
                        len_range=(500000, 524288)),
    # 64 requests x ~150K (+-5%), NVFP4 K from bf16 keys via the store, bf16 q
    "nvfp4_64x150k": Spec("nvfp4_64x150k", 1005, "nvfp4", "bf16", 64, 4, 4, 1, 4, 64,
                          len_range=(142500, 157500)),
    # the verify-rows layout: 4 requests x 4 draft rows ending at 32767..32770
    "verify_bf16_4x32k": Spec("verify_bf16_4x32k", 1007, "bf16", "bf16", 4, 4, 4, 1, 4, 64,
                              explicit_lens=[_verify_rows(4, [32767, 32768, 32769, 32770])] * 4),
    "verify_fp8_4x32k": Spec("verify_fp8_4x32k", 1008, "fp8_e4m3", "fp8_e4m3", 4, 4, 4, 1, 4, 64,
                             explicit_lens=[_verify_rows(4, [32767, 32768, 32769, 32770])] * 4),
    # more than 16 packed rows (the 128-row tensor-core tiles): 8 draft rows x 8 heads
    "verify_bf16_16x32k_p8g8": Spec("verify_bf16_16x32k_p8g8", 1009, "bf16", "bf16", 16, 8, 8,
                                    1, 4, 64, len_range=(30000, 32768)),
    # prefill chunks: 512 query tokens x 4 heads per request, the chunk ending the
    # request's ~32K context (row j of the chunk has length L - 511 + j)
    "prefill_nvfp4_4x32k_c512": Spec("prefill_nvfp4_4x32k_c512", 1010, "nvfp4", "bf16", 4, 512, 4,
                                     1, 4, 64, len_range=(32000, 32768)),
    "prefill_bf16_4x32k_c512": Spec("prefill_bf16_4x32k_c512", 1011, "bf16", "bf16", 4, 512, 4,
                                    1, 4, 64, len_range=(32000, 32768)),
    "prefill_fp8_4x32k_c512": Spec("prefill_fp8_4x32k_c512", 1012, "fp8_e4m3", "fp8_e4m3", 4, 512,
                                   4, 1, 4, 64, len_range=(32000, 32768)),
}


def small_spec(name: str, seed: int, k_dtype: str, q_dtype: str, *, R: int = 5, P: int = 4,
               G: int = 4, init_blocks: int = 1, local_blocks: int = 2, topk: int = 16,
               len_range=(1, 9000), pad_requests=(), explicit_lens=None) -> Spec:
    """A batch the oracle finishes in well under a second: several tiles and
    ragged tails, optional pad requests."""
    return Spec(name, seed, k_dtype, q_dtype, R, P, G, init_blocks, local_blocks, topk,
                explicit_lens=explicit_lens, len_range=None if explicit_lens else len_range,
                pad_requests=tuple(pad_requests), junk_page_frac=0.5)

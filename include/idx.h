/*
 * libidx — packed sparse-attention index scoring + block top-k for GB300 (sm_103a).
 *
 * C ABI.  Every pointer named "device" must point to device memory of the current
 * CUDA device; "host" pointers are read before the call returns.  Streams are
 * cudaStream_t values passed as void* (NULL = legacy default stream).  No call
 * below synchronises the host with the device, except the ones marked "syncs".
 *
 * Constants of the format (the pages' workloads):
 *   page = 64 tokens, block = 128 tokens, head dim D = 128, at most 16 packed rows.
 *
 * Pool planes (one index-K pool per layer; ROCm/ATOM #2745, Summary, "Pool and
 * binding": payload and scale kept as separate uint8 planes):
 *   payload: uint8 [num_pages * 64][row_bytes], physical row = page * 64 + t % 64
 *            row_bytes = 256 (bf16 keys, little-endian), 128 (e4m3 codes),
 *            64 (NVFP4: two e2m1 codes per byte, even element in the low nibble)
 *   scale:   uint8 [num_pages * 64][scale_bytes]
 *            scale_bytes = 0 (bf16: no plane), 4 (fp8: one fp32 per key),
 *            8 (NVFP4: one E4M3 scale per 16 elements, unit outer scale)
 */
#ifndef LIBIDX_IDX_H_
#define LIBIDX_IDX_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define IDX_API __attribute__((visibility("default")))
#else
#define IDX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define IDX_ABI_VERSION 1
#define IDX_PAGE_SIZE 64
#define IDX_BLOCK_SIZE 128
#define IDX_DIM 128
#define IDX_MAX_PACKED_ROWS 16        /* rows of one warp-MMA tile (P*G up to this) */
#define IDX_WIDE_TILE_ROWS 128        /* rows of one tensor-core tile (P*G above 16) */
#define IDX_MAX_ROWS_PER_REQUEST 32768 /* packed_queries * gqa of one request */
#define IDX_MAX_CP_WORLD 8            /* context shards idx_topk_merge accepts */
#define IDX_MAX_TOPK 256
#define IDX_WORKSPACE_HEADER_BYTES 1024
#define IDX_MAX_REQUESTS 2048  /* per idx_score_topk call (draft rows per per-row call) */

typedef enum {
  IDX_BF16 = 0,      /* bfloat16 */
  IDX_FP8_E4M3 = 1,  /* OCP E4M3 ("fn": no infinities, max 448) with fp32 scales */
  IDX_NVFP4 = 2      /* e2m1 payload + E4M3 per-16 scales (keys only) */
} idx_dtype;

typedef enum {
  IDX_OK = 0,
  IDX_ERR_INVALID = -1,      /* an argument is out of range or a pointer is NULL */
  IDX_ERR_UNSUPPORTED = -2,  /* a dtype combination this library does not implement */
  IDX_ERR_CUDA = -3,         /* a CUDA runtime call or kernel launch failed */
  IDX_ERR_OOM = -4           /* device allocation failed */
} idx_status;

/* Device-side error flags of a call, kept in the workspace header (read them with
 * idx_workspace_errors). */
#define IDX_DEVERR_BAD_PAGE 1u      /* a page id outside [0, num_pages): page not read */
#define IDX_DEVERR_TIMEOUT 2u       /* a pipeline wait gave up (kernel ended early) */
#define IDX_DEVERR_LEN_CLAMPED 4u   /* a row longer than max_pages * 64 was clamped */

/* One index-K pool: payload + scale planes of a paged cache. */
typedef struct idx_pool {
  int32_t dtype;              /* idx_dtype of the keys */
  int32_t page_size;          /* tokens per page: 64 */
  int32_t dim;                /* head dim: 128 */
  int32_t reserved;
  int64_t num_pages;
  void* payload;              /* device, uint8 [num_pages*64][payload_row_bytes] */
  void* scale;                /* device, uint8 [num_pages*64][scale_row_bytes]; NULL for bf16 */
  int64_t payload_row_bytes;  /* 256 | 128 | 64 */
  int64_t scale_row_bytes;    /* 0 | 4 | 8 */
} idx_pool;

/* Library / status helpers. */
IDX_API int idx_abi_version(void);
IDX_API const char* idx_status_string(int status);
/* Text of the last error raised on the calling host thread ("" if none). */
IDX_API const char* idx_last_error(void);

/*
 * idx_pool_alloc — allocate the planes of a paged index-K pool on the current device.
 * The pool layout is the one the ATOM NVFP4 index cache page describes (ROCm/ATOM
 * #2745, Summary): 72 B per NVFP4 key (64 B payload + 8 B scales), 128 B + 4 B
 * per fp8 key, 256 B per bf16 key.  Contents are uninitialised.
 *   dtype: idx_dtype; num_pages >= 1; page_size must be 64; dim must be 128.
 *   out (host): filled on success; the library owns the planes until idx_pool_free.
 * Returns IDX_ERR_INVALID for bad arguments, IDX_ERR_OOM if cudaMalloc fails.
 */
IDX_API int idx_pool_alloc(int dtype, int64_t num_pages, int page_size, int dim, idx_pool* out);

/* idx_pool_free — release planes made by idx_pool_alloc (syncs with the device
 * through cudaFree).  Zeroes *pool.  A pool whose planes the caller allocated must
 * not be passed here. */
IDX_API int idx_pool_free(idx_pool* pool);

/*
 * idx_store_nvfp4 — quantise staged bf16 keys to NVFP4 and write them into the pool
 * at their real slots (ROCm/ATOM #2745, Summary: "Store" and "Write").  Per group of
 * 16 elements: amax in fp32; scale = E4M3(amax / 6) rounded half-to-even, saturating
 * at 448; codes = e2m1(x / scale) with a correctly rounded fp32 division, rounded
 * half-to-even, saturating at 6, sign kept (a negative value rounding to 0 is 0x8);
 * a scale of 0 writes all-zero codes; element 2b goes to the low nibble of byte b.
 *   src_bf16 (device):     bf16 [num_tokens][128], token-major staging buffer.
 *   slot_mapping (device): int64 [num_tokens], physical pool row of each key
 *                          (page * 64 + offset); a negative entry skips the key; an
 *                          entry >= num_pages*64 skips it too.
 *   pool (host):           an NVFP4 pool (caller- or library-allocated planes).
 * Asynchronous on stream.  IDX_ERR_INVALID if pool is not NVFP4 or a pointer is NULL
 * (num_tokens == 0 is a no-op).
 */
IDX_API int idx_store_nvfp4(const void* src_bf16, const int64_t* slot_mapping, int64_t num_tokens,
                    const idx_pool* pool, void* stream);

/*
 * idx_score_topk_workspace_bytes — device scratch idx_score_topk needs: a header of
 * IDX_WORKSPACE_HEADER_BYTES (device error flags) plus one fp32 block score per
 * (request, packed row, block): num_requests * packed_queries * gqa *
 * ceil(max_pages / 2) floats.  When packed_queries * gqa > IDX_MAX_PACKED_ROWS
 * (the 128-row tensor-core path) it adds, from the next 256-byte boundary, 260
 * bytes per packed row: the rows of q converted once per call to f16 (NVFP4
 * keys), and their scales.
 */
IDX_API size_t idx_score_topk_workspace_bytes(int num_requests, int packed_queries, int gqa,
                                      int max_pages);

/*
 * idx_score_topk — the packed index step of one sparse layer (sglang #45451,
 * Modifications; sglang #42614 "[AMD] MiniMax-M3 indexer CP: packed scoring for EAGLE
 * verify rows", Modifications 1).
 *
 * For request r, its P = packed_queries draft rows times G = gqa heads form its
 * packed rows; row i is (draft row i / G, head i % G).  With P*G <= 16 the rows are
 * one 16-row tile, dotted with the request's keys on the warp-level tensor-core MMA
 * with the keys read once per request up to the group's longest row.  With P*G > 16
 * (many draft rows, or a prefill chunk: P query tokens, each its own row length) the
 * rows are cut into tiles of IDX_WIDE_TILE_ROWS, each dotted on the 5th-generation
 * tensor cores (tcgen05) with the keys read once per tile up to the tile's longest
 * row.  Row i then keeps only tokens t < its own length, takes the max score of each
 * 128-token block, always keeps its first init_blocks and last local_blocks blocks
 * (from its own block count), and emits topk block ids with their scores.
 *
 *   q (device):          [R][P][G][128] bf16 (q_dtype IDX_BF16) or e4m3 codes (IDX_FP8_E4M3)
 *   q_scale (device):    fp32 [R][P*G], one scale per packed row; required for e4m3 q,
 *                        ignored (may be NULL) for bf16 q
 *   k_payload, k_scale (device): the pool planes; k_scale is ignored for bf16 keys
 *   k_dtype:             IDX_BF16 (with bf16 q), IDX_FP8_E4M3 (with e4m3 q) or
 *                        IDX_NVFP4 (with bf16 q); other pairs: IDX_ERR_UNSUPPORTED
 *   num_pages:           pages in the pool (page ids outside [0, num_pages) are not
 *                        read and set IDX_DEVERR_BAD_PAGE)
 *   page_table (device): int32 [n_slots][max_pages], page of token t of the request
 *                        in slot s = page_table[s][t / 64]
 *   slot_ids (device):   int32 [R]; a slot outside [0, n_slots) marks a pad request
 *                        (graph padding): nothing is read, all its rows are pads
 *   row_lens (device):   int32 [R][P], tokens of each draft row (its causal length);
 *                        <= 0 gives an all-pad row; > max_pages*64 is clamped
 *   init_blocks, local_blocks >= 0 with init_blocks + local_blocks <= topk
 *   topk:                1 ..IDX_MAX_TOPK
 *   out_ids (device):    int32 [R][P*G][topk]
 *   out_scores (device): fp32 [R][P*G][topk]
 *   workspace (device):  >= idx_score_topk_workspace_bytes(R, P, G, max_pages) bytes,
 *                        256-byte aligned; overwritten by every call (no clearing is
 *                        needed); its header holds the device error flags
 *                        (IDX_DEVERR_*) of the last call and the state of the
 *                        kernel's dynamic work counter, which every call leaves
 *                        ready for the next one (a fresh workspace simply runs
 *                        its first call with a static schedule).  Calls that may
 *                        overlap on the GPU (on different streams, or from
 *                        different host threads without ordering) must not share
 *                        a workspace: they race on its block scores, its error
 *                        flags and the work counter.
 * Output row i of request r: its forced blocks in ascending id order, then the chosen
 * blocks by descending score (ties to the lower id), then (-1, -inf) pads.  Scores are
 * raw q.k block maxima (fp8: code dot products times q_scale times the key's scale).
 * Asynchronous on stream; allocates nothing; capturable in a CUDA graph.
 * Host-side checks return IDX_ERR_INVALID (P*G outside [1, IDX_MAX_ROWS_PER_REQUEST],
 * topk out of range, init+local > topk, NULL pointers, R < 0 or > IDX_MAX_REQUESTS,
 * R * ceil(ceil(P*G / IDX_WIDE_TILE_ROWS) / 2) > IDX_MAX_REQUESTS when P*G > 16, n_slots or
 * max_pages < 1, workspace too
 * small or misaligned, num_pages < 1).  With R == 0 only the workspace is required
 * (its header is reset) and the per-request pointers may be NULL.
 */
IDX_API int idx_score_topk(const void* q, const float* q_scale, int q_dtype,
                   const void* k_payload, const void* k_scale, int k_dtype, int64_t num_pages,
                   const int32_t* page_table, int n_slots, int max_pages,
                   const int32_t* slot_ids, const int32_t* row_lens,
                   int num_requests, int packed_queries, int gqa,
                   int init_blocks, int local_blocks, int topk,
                   int32_t* out_ids, float* out_scores,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * idx_score_topk_lse — idx_score_topk with the log-sum-exp block score in place of the
 * block max (sglang #45451, Accuracy Tests: selected-block scores "max; lse"): a row's
 * score for block b is ln sum exp(q.k_t) over the tokens t of the block inside the row's
 * length (raw dot products, natural log).  Same arguments, outputs, selection rules and
 * workspace; out_scores holds the chosen blocks' log-sum-exp.
 */
IDX_API int idx_score_topk_lse(const void* q, const float* q_scale, int q_dtype,
                               const void* k_payload, const void* k_scale, int k_dtype,
                               int64_t num_pages, const int32_t* page_table, int n_slots,
                               int max_pages, const int32_t* slot_ids, const int32_t* row_lens,
                               int num_requests, int packed_queries, int gqa,
                               int init_blocks, int local_blocks, int topk,
                               int32_t* out_ids, float* out_scores,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * idx_score_local_blocks — the step over one context shard (indexer context
 * parallelism: sglang #42614 "[AMD] MiniMax-M3 indexer CP: packed scoring for EAGLE
 * verify rows", Motivation and Modifications 1, name the per-shard scorer
 * score_local_blocks).  The rank holding the shard calls it; idx_topk_merge then
 * combines every shard's list.
 *
 * The shard is global blocks [block_begin, block_begin + max_pages / 2) of every
 * request: page_table[s][p] is the page of the request's global tokens
 * (2 * block_begin + p) * 64 .. + 63, so max_pages must be even (whole 128-token
 * blocks; a block never straddles two shards).  row_lens, init_blocks,
 * local_blocks and topk are the row's global ones: the forced blocks and the number
 * c of candidates to choose come from the row's own global block count.  Row i of
 * request r gets the shard's forced blocks (ascending, global ids), then its best
 * min(c, candidates in the shard) candidates by score (ties to the lower id), then
 * (-1, -inf) pads.  Packed rows of one 16-row tile only (P*G <= 16).  Other
 * arguments, the workspace (sized for the shard's max_pages) and the error
 * behaviour are those of idx_score_topk; rows longer than the shard are not
 * flagged (IDX_DEVERR_LEN_CLAMPED is for whole-context calls).
 */
IDX_API int idx_score_local_blocks(const void* q, const float* q_scale, int q_dtype,
                                   const void* k_payload, const void* k_scale, int k_dtype,
                                   int64_t num_pages, const int32_t* page_table, int n_slots,
                                   int max_pages, int block_begin, const int32_t* slot_ids,
                                   const int32_t* row_lens, int num_requests,
                                   int packed_queries, int gqa, int init_blocks,
                                   int local_blocks, int topk, int32_t* out_ids,
                                   float* out_scores, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * idx_topk_merge — the exchange step's re-selection: combine the lists of `world`
 * context shards into each row's global selection.
 *
 *   cand_ids, cand_scores (device): int32 / fp32 [world][R][P*G][topk], shard w's
 *                        idx_score_local_blocks output (any order of shards); the
 *                        shards must partition every row's blocks
 *   slot_ids, row_lens (device): as for idx_score_topk (global lengths; a slot
 *                        outside [0, n_slots) makes the request's rows pads)
 *   out_ids, out_scores (device): int32 / fp32 [R][P*G][topk]
 * Row i gets its forced blocks ascending with the score their shard reported, then
 * the best c of all the shards' other entries (score desc, ties to the lower id),
 * then (-1, -inf) pads: the same as idx_score_topk over the whole context, since
 * each shard keeps its best c candidates.  Host checks return IDX_ERR_INVALID
 * (world outside [1, IDX_MAX_CP_WORLD], R outside [0, IDX_MAX_REQUESTS], P*G out of
 * range, topk or init/local out of range, n_slots < 1, NULL pointers).
 * Asynchronous on stream; allocates nothing.
 */
IDX_API int idx_topk_merge(const int32_t* cand_ids, const float* cand_scores, int world,
                           const int32_t* slot_ids, const int32_t* row_lens, int n_slots,
                           int num_requests, int packed_queries, int gqa, int init_blocks,
                           int local_blocks, int topk, int32_t* out_ids, float* out_scores,
                           void* stream);

/*
 * idx_score_topk_perrow — the same step with every draft row scored as its own decode
 * row (the per-row kernel the packed one replaces: sglang #45451, Motivation; sglang
 * #42614, Motivation): the tile holds G live rows and each request's keys are read
 * once per draft row.  Same arguments, same outputs, same workspace size; an internal
 * ablation of the packed kernel.
 */
IDX_API int idx_score_topk_perrow(const void* q, const float* q_scale, int q_dtype,
                          const void* k_payload, const void* k_scale, int k_dtype,
                          int64_t num_pages, const int32_t* page_table, int n_slots,
                          int max_pages, const int32_t* slot_ids, const int32_t* row_lens,
                          int num_requests, int packed_queries, int gqa,
                          int init_blocks, int local_blocks, int topk,
                          int32_t* out_ids, float* out_scores,
                          void* workspace, size_t workspace_bytes, void* stream);

/* idx_set_kernel_events — instrumentation for timing.  Arms, for the next
 * idx_score_topk / idx_score_topk_perrow call on the calling host thread only, up
 * to three cudaEvent_t (passed as void*, NULL to skip) that the call records on its
 * stream: before the score kernel, after the score kernel, after the top-k kernel.
 * The events are used once and then forgotten. */
IDX_API int idx_set_kernel_events(void* score_begin, void* score_end, void* topk_end);

/* idx_set_kernel_waits — ordering for pipelined callers.  Arms, for the next
 * idx_score_topk / _lse / _perrow / idx_score_local_blocks call on the calling
 * host thread only, up to two cudaEvent_t (passed as void*, NULL to skip) that
 * the call's stream waits for (cudaStreamWaitEvent): before_score before the
 * score kernel is launched, before_topk before the top-k kernel is launched.
 * The events are used once and then forgotten.  What it is for: the score
 * kernel is launched as a programmatic dependent of the kernel before it and
 * starts under it, but a wait placed right before it (a cross-stream event, a
 * captured graph's join) makes it start only after that kernel has finished.
 * A loop that copies step k + 1's inputs on another stream can hand that
 * copy's event to step k's call as before_topk: step k + 1's score kernel reads
 * its inputs only after step k's top-k has completed, which now comes after the
 * copy, and keeps its overlap with step k.  Always returns IDX_OK. */
IDX_API int idx_set_kernel_waits(void* before_score, void* before_topk);

/*
 * idx_score_topk_noalloc — idx_score_topk for callers that cannot allocate device
 * memory.  (The pages have no counterpart: it is an addition of this library.)
 *
 * Who needs it: a caller whose device memory is owned by someone else — a serving
 * engine whose memory pool must account for every byte, a plugin loaded into a host
 * framework with no allocator hook — or a caller that cannot afford the device-wide
 * synchronisation cudaMalloc / cudaFree may cause in the middle of a decode step,
 * has no way to hand idx_score_topk a workspace.  This variant keeps its block-score
 * scratch in a fixed array of IDX_NOALLOC_SCRATCH_BYTES inside the library instead;
 * every GPU that loads the library holds that array until the process exits.
 *
 * Same arguments and outputs as idx_score_topk without the workspace.  The call must
 * need at most IDX_NOALLOC_SCRATCH_BYTES of scratch, i.e.
 *   IDX_WORKSPACE_HEADER_BYTES + num_requests * packed_queries * gqa *
 *   ceil(max_pages / 2) * 4 bytes,
 * otherwise it returns IDX_ERR_INVALID before any device work.  It calls no
 * allocator.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call before
 * any stream capture.  All calls share the one array and it keeps the last call's
 * contents (each call rewrites what it reads): calls that overlap on
 * the GPU — on different streams, or from different host threads — race on it and
 * must be serialised by the caller.  The device error flags of the last call on
 * the current device are read with idx_noalloc_errors.  If the device's context
 * is torn down and made anew (cudaDeviceReset), the next call looks the address
 * up again.
 */
#define IDX_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)
IDX_API int idx_score_topk_noalloc(const void* q, const float* q_scale, int q_dtype,
                                   const void* k_payload, const void* k_scale, int k_dtype,
                                   int64_t num_pages, const int32_t* page_table, int n_slots,
                                   int max_pages, const int32_t* slot_ids,
                                   const int32_t* row_lens, int num_requests, int packed_queries,
                                   int gqa, int init_blocks, int local_blocks, int topk,
                                   int32_t* out_ids, float* out_scores, void* stream);

/* idx_noalloc_errors — the device error flags (IDX_DEVERR_*) of the last
 * idx_score_topk_noalloc call on the current device, read from the fixed scratch
 * array's header (syncs on stream; allocates nothing).  No counterpart on the
 * pages: it is the no-allocation variant's idx_workspace_errors.
 *   flags (host): receives the IDX_DEVERR_* bits. */
IDX_API int idx_noalloc_errors(void* stream, uint32_t* flags);

/* idx_set_wait_limit_ns — limit (nanoseconds, process-wide) of every pipeline wait in
 * the score kernels; 0 restores the default of 2 s.  A wait that runs past it ends
 * its role: the CTA waits for its own copies in flight, frees its tensor memory,
 * sets IDX_DEVERR_TIMEOUT in the workspace header and exits, so the context stays
 * usable.  The limit is read at each call (a captured graph keeps the one of its
 * capture).  Always returns IDX_OK. */
IDX_API int idx_set_wait_limit_ns(uint64_t ns);

/* idx_set_stall_test — diagnostic (process-wide, off by default): with on != 0, in
 * every score CTA one role's first pipeline wait goes to a barrier that nothing
 * completes (the 16-row kernel: warp 0, after issuing its first copies; the
 * tensor-core kernel: the MMA issuer), so it runs out after the wait limit and the
 * call ends through the timeout path described above, with IDX_DEVERR_TIMEOUT set.
 * Outputs of such a call are meaningless.  Lets a test exercise failure handling
 * on the GPU without a fault.  Always returns IDX_OK. */
IDX_API int idx_set_stall_test(int on);

/* idx_set_grid_limit — cap the number of CTAs the score kernel launches (process-
 * wide; 0 restores the default of one CTA per SM).  Results do not depend on it:
 * each block max is computed whole by one warp, so any split of the work gives the
 * same bits.  Meant for tests and tuning. */
IDX_API int idx_set_grid_limit(int max_ctas);

/* idx_workspace_errors — read the device error flags of the last call that used this
 * workspace (syncs on stream).  flags (host): receives the IDX_DEVERR_* bits. */
IDX_API int idx_workspace_errors(const void* workspace, void* stream, uint32_t* flags);

#ifdef __cplusplus
}
#endif

#endif /* LIBIDX_IDX_H_ */

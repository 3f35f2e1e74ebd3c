// C ABI of libidx: argument checks, tensor-map set-up and kernel launches.
// Every entry point returns an idx_status; the message of the last failure on
// the calling host thread is available from idx_last_error().
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>

#include "../../include/idx.h"
#include "idx_internal.cuh"

static_assert(idx::kHeaderBytes == IDX_WORKSPACE_HEADER_BYTES, "header size mismatch");

namespace {

thread_local std::string g_last_error;
thread_local cudaEvent_t g_ev[3] = {nullptr, nullptr, nullptr};
thread_local cudaEvent_t g_wait[2] = {nullptr, nullptr};

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(IDX_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Record a caller-supplied timing event on the stream; while the stream is being
// captured into a CUDA graph the record becomes an external event node, so the
// event still carries a timestamp each time the graph is replayed.
cudaError_t record_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  return cudaEventRecord(ev, st);
}

int64_t payload_row_bytes(int dtype) {
  switch (dtype) {
    case IDX_BF16: return 256;
    case IDX_FP8_E4M3: return 128;
    case IDX_NVFP4: return 64;
    default: return -1;
  }
}

int64_t scale_row_bytes(int dtype) {
  switch (dtype) {
    case IDX_BF16: return 0;
    case IDX_FP8_E4M3: return 4;
    case IDX_NVFP4: return 8;
    default: return -1;
  }
}

// cuTensorMapEncodeTiled, looked up once through the runtime so the library
// carries no link-time dependency on the driver library.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The last few tensor maps this host thread encoded, keyed by what they
// describe, so a caller that reuses its pool and query buffers (a serving loop)
// pays for the encoding once.
struct MapCache {
  struct Entry {
    int kind, dtype;
    const void* ptr;
    int64_t rows;
    CUtensorMap map;
  };
  static constexpr int kEntries = 8;
  Entry e[kEntries];
  int n = 0, next = 0;
  const CUtensorMap* find(int kind, int dtype, const void* ptr, int64_t rows) const {
    for (int i = 0; i < n; ++i)
      if (e[i].kind == kind && e[i].dtype == dtype && e[i].ptr == ptr && e[i].rows == rows)
        return &e[i].map;
    return nullptr;
  }
  void put(int kind, int dtype, const void* ptr, int64_t rows, const CUtensorMap& m) {
    Entry& x = e[next];
    x.kind = kind;
    x.dtype = dtype;
    x.ptr = ptr;
    x.rows = rows;
    x.map = m;
    next = (next + 1) % kEntries;
    if (n < kEntries) ++n;
  }
};
thread_local MapCache g_maps;

// Tensor map over the payload plane, one 64-row (one page) box per load:
//  bf16: 128 bf16 per row, box 64 x 64 (two boxes per page), 128-byte swizzle
//  fp8:  128 bytes per row, box 128 x 64, 128-byte swizzle
//  fp4:  64 bytes per row,  box 64 x 64,  64-byte swizzle
int make_payload_map(int dtype, const void* payload, int64_t num_pages, CUtensorMap* map) {
  if (const CUtensorMap* hit = g_maps.find(0, dtype, payload, num_pages)) {
    *map = *hit;
    return IDX_OK;
  }
  auto fn = encode_fn();
  if (!fn) return fail(IDX_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t rows = (cuuint64_t)num_pages * idx::kPage;
  cuuint64_t dims[2];
  cuuint64_t strides[1];
  cuuint32_t box[2];
  const cuuint32_t estride[2] = {1, 1};
  CUtensorMapDataType dt;
  CUtensorMapSwizzle sw;
  if (dtype == IDX_BF16) {
    dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    dims[0] = 128; strides[0] = 256; box[0] = 64; sw = CU_TENSOR_MAP_SWIZZLE_128B;
  } else if (dtype == IDX_FP8_E4M3) {
    dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    dims[0] = 128; strides[0] = 128; box[0] = 128; sw = CU_TENSOR_MAP_SWIZZLE_128B;
  } else {
    dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    dims[0] = 64; strides[0] = 64; box[0] = 64; sw = CU_TENSOR_MAP_SWIZZLE_64B;
  }
  dims[1] = rows;
  box[1] = idx::kPage;
  CUresult r = fn(map, dt, 2, const_cast<void*>(payload), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IDX_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  g_maps.put(0, dtype, payload, num_pages, *map);
  return IDX_OK;
}

// Tensor map over the query rows [rows][128] for the 128-row tiles of the
// tensor-core path: bf16 as two 64-column boxes, e4m3 as one 128-byte box, both
// 128 rows high with the 128-byte swizzle the MMA operand descriptors expect.
// Rows past the end read as zeros.
int make_q_map(int q_dtype, const void* q, int64_t rows, CUtensorMap* map) {
  if (const CUtensorMap* hit = g_maps.find(1, q_dtype, q, rows)) {
    *map = *hit;
    return IDX_OK;
  }
  auto fn = encode_fn();
  if (!fn) return fail(IDX_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1];
  cuuint32_t box[2] = {0, 128};
  const cuuint32_t estride[2] = {1, 1};
  CUtensorMapDataType dt;
  if (q_dtype == IDX_BF16) {
    dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    strides[0] = 256;
    box[0] = 64;
  } else {
    dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    strides[0] = 128;
    box[0] = 128;
  }
  CUresult r = fn(map, dt, 2, const_cast<void*>(q), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(IDX_ERR_CUDA, "cuTensorMapEncodeTiled (query rows) failed (%d)", (int)r);
  g_maps.put(1, q_dtype, q, rows, *map);
  return IDX_OK;
}

// block_begin < 0: the page table covers each request's whole context; >= 0:
// it covers one context shard starting at that global block.
int score_topk_impl(bool perrow, int block_score, int block_begin, const void* q,
                    const float* q_scale, int q_dtype,
                    const void* k_payload, const void* k_scale, int k_dtype, int64_t num_pages,
                    const int32_t* page_table, int n_slots, int max_pages, const int32_t* slot_ids,
                    const int32_t* row_lens, int R, int P, int G, int init_blocks,
                    int local_blocks, int topk, int32_t* out_ids, float* out_scores,
                    void* workspace, size_t workspace_bytes, void* stream) {
  if (R < 0) return fail(IDX_ERR_INVALID, "num_requests must be >= 0 (got %d)", R);
  if (P < 1 || G < 1 || (long long)P * G > IDX_MAX_ROWS_PER_REQUEST)
    return fail(IDX_ERR_INVALID, "packed_queries * gqa must be in [1, %d] (got %d x %d)",
                IDX_MAX_ROWS_PER_REQUEST, P, G);
  if (perrow && G > IDX_MAX_PACKED_ROWS)
    return fail(IDX_ERR_INVALID, "per-row scoring needs gqa <= %d (got %d)", IDX_MAX_PACKED_ROWS,
                G);
  const bool wide = !perrow && P * G > IDX_MAX_PACKED_ROWS;
  const bool shard = block_begin >= 0;
  if (shard && (perrow || wide))
    return fail(IDX_ERR_INVALID,
                "context-shard scoring takes packed rows of one 16-row tile (P*G <= 16)");
  if (shard && (max_pages % 2 != 0 || block_begin > (1 << 24)))
    return fail(IDX_ERR_INVALID,
                "a context shard holds whole 128-token blocks: max_pages must be even (got %d)",
                max_pages);
  const int tiles = (P * G + IDX_WIDE_TILE_ROWS - 1) / IDX_WIDE_TILE_ROWS;
  if (wide && (long long)R * ((tiles + 1) / 2) > idx::kMaxGroups)
    return fail(IDX_ERR_INVALID,
                "at most %d pairs of request tiles per call (num_requests * ceil(packed_queries "
                "* gqa / %d) / 2, rounded up per request, = %lld)",
                idx::kMaxGroups, IDX_WIDE_TILE_ROWS, (long long)R * ((tiles + 1) / 2));
  if (topk < 1 || topk > IDX_MAX_TOPK)
    return fail(IDX_ERR_INVALID, "topk must be in [1, %d] (got %d)", IDX_MAX_TOPK, topk);
  if (init_blocks < 0 || local_blocks < 0 || init_blocks + local_blocks > topk)
    return fail(IDX_ERR_INVALID,
                "need init_blocks, local_blocks >= 0 and init + local <= topk (got %d, %d, %d)",
                init_blocks, local_blocks, topk);
  const bool pair_ok = (k_dtype == IDX_BF16 && q_dtype == IDX_BF16) ||
                       (k_dtype == IDX_FP8_E4M3 && q_dtype == IDX_FP8_E4M3) ||
                       (k_dtype == IDX_NVFP4 && q_dtype == IDX_BF16);
  if (!pair_ok)
    return fail(IDX_ERR_UNSUPPORTED, "unsupported (k_dtype, q_dtype) = (%d, %d)", k_dtype, q_dtype);
  if ((perrow ? (long long)R * P : (long long)R) > idx::kMaxGroups)
    return fail(IDX_ERR_INVALID, "at most %d %s per call (got %lld)", idx::kMaxGroups,
                perrow ? "draft rows (num_requests * packed_queries)" : "requests",
                perrow ? (long long)R * P : (long long)R);
  if (n_slots < 1 || max_pages < 1 || max_pages > 65536)
    return fail(IDX_ERR_INVALID, "need n_slots >= 1 and 1 <= max_pages <= 65536 (got %d, %d)",
                n_slots, max_pages);
  if (num_pages < 1 || num_pages * idx::kPage > 0x7fffffffLL)
    return fail(IDX_ERR_INVALID, "num_pages must be in [1, 2^31 / 64) (got %lld)",
                (long long)num_pages);
  if (!workspace) return fail(IDX_ERR_INVALID, "workspace is NULL");
  if (R > 0 && (!q || !k_payload || !page_table || !slot_ids || !row_lens || !out_ids ||
                !out_scores))
    return fail(IDX_ERR_INVALID, "a required pointer is NULL");
  if (R > 0 && k_dtype != IDX_BF16 && !k_scale) return fail(IDX_ERR_INVALID, "k_scale is NULL");
  if (R > 0 && q_dtype == IDX_FP8_E4M3 && !q_scale)
    return fail(IDX_ERR_INVALID, "q_scale is NULL");
  if (!aligned(k_payload, 16) || (k_scale && !aligned(k_scale, 16)) || !aligned(q, 16))
    return fail(IDX_ERR_INVALID, "q, k_payload and k_scale must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(IDX_ERR_INVALID, "workspace must be 256-byte aligned");
  const size_t need = idx_score_topk_workspace_bytes(R, P, G, max_pages);
  if (workspace_bytes < need)
    return fail(IDX_ERR_INVALID, "workspace too small: %zu < %zu bytes", workspace_bytes, need);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (R == 0) {
    // no kernel runs: record "no CTA, no flags" for idx_workspace_errors
    e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace header");
    return IDX_OK;
  }

  CUtensorMap map;
  int rc = make_payload_map(k_dtype, k_payload, num_pages, &map);
  if (rc != IDX_OK) return rc;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  idx::ScoreArgs sa;
  sa.q = static_cast<const uint8_t*>(q);
  sa.q_scale = q_scale;
  sa.k_scale = static_cast<const uint8_t*>(k_scale);
  sa.page_table = page_table;
  sa.slot_ids = slot_ids;
  sa.row_lens = row_lens;
  sa.blockmax = reinterpret_cast<float*>(ws + IDX_WORKSPACE_HEADER_BYTES);
  sa.err_bytes = ws + idx::kFlagBytesOff;
  sa.err_count = reinterpret_cast<uint32_t*>(ws);
  sa.sched_counter = reinterpret_cast<uint32_t*>(ws + idx::kSchedOff);
  sa.sched_tag = reinterpret_cast<const unsigned long long*>(ws + idx::kTagOff);
  sa.num_pages = num_pages;
  sa.n_slots = n_slots;
  sa.max_pages = max_pages;
  sa.nb_cap = (max_pages + 1) / 2;
  sa.R = R;
  sa.P = P;
  sa.G = G;
  sa.M = P * G;
  sa.perrow = perrow ? 1 : 0;
  sa.tiles = tiles;
  sa.block_off = shard ? block_begin : 0;
  sa.shard = shard ? 1 : 0;
  sa.wait_ns = idx::wait_limit_ns();
  sa.stall_test = idx::stall_test();
  sa.q16 = nullptr;
  sa.qpost = nullptr;
  CUtensorMap qmap = map;
  if (wide && k_dtype != IDX_NVFP4) {
    rc = make_q_map(q_dtype, q, (int64_t)R * P * G, &qmap);
    if (rc != IDX_OK) return rc;
  } else if (wide) {
    // NVFP4 keys: the query rows are converted to f16 once per call into the
    // workspace (a small kernel before the score kernel), and the tiles load
    // from there like bf16 ones (TMA copies bits: the bf16 map describes them)
    const long long rows = (long long)R * P * G;
    sa.q16 = reinterpret_cast<uint16_t*>(ws + idx::ws_q16_offset(rows, max_pages));
    sa.qpost = reinterpret_cast<float*>(ws + idx::ws_q16_offset(rows, max_pages) + rows * 256);
    rc = make_q_map(IDX_BF16, sa.q16, rows, &qmap);
    if (rc != IDX_OK) return rc;
  }
  cudaEvent_t ev[3] = {g_ev[0], g_ev[1], g_ev[2]};
  g_ev[0] = g_ev[1] = g_ev[2] = nullptr;
  const cudaEvent_t wait_score = g_wait[0], wait_topk = g_wait[1];
  g_wait[0] = g_wait[1] = nullptr;

  idx::TopkArgs ta;
  ta.blockmax = sa.blockmax;
  ta.slot_ids = slot_ids;
  ta.row_lens = row_lens;
  ta.out_ids = out_ids;
  ta.out_scores = out_scores;
  ta.sched_counter = sa.sched_counter;
  ta.sched_tag = reinterpret_cast<unsigned long long*>(ws + idx::kTagOff);
  ta.n_slots = n_slots;
  ta.max_pages = max_pages;
  ta.nb_cap = sa.nb_cap;
  ta.R = R;
  ta.P = P;
  ta.G = G;
  ta.M = P * G;
  ta.init_blocks = init_blocks;
  ta.local_blocks = local_blocks;
  ta.topk = topk;
  ta.block_off = sa.block_off;
  ta.shard = sa.shard;
#if IDX_FUSED_TOPK
  const bool fused = !wide && !shard && !perrow;
  sa.fused = fused ? 1 : 0;
  if (fused) {
    sa.topk = ta;
    sa.arrive = reinterpret_cast<uint32_t*>(ws + idx::kArriveOff);
    sa.depart = reinterpret_cast<uint32_t*>(ws + idx::kDepartOff);
    // the grid barrier's counters must start at zero whatever the workspace
    // held before (the dynamic schedule's tag is dropped with them)
    e = cudaMemsetAsync(ws + idx::kSchedOff, 0, idx::kFlagBytesOff - idx::kSchedOff, st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace counters");
  }
#else
  const bool fused = false;
#endif
  if (wait_score && (e = cudaStreamWaitEvent(st, wait_score, 0)) != cudaSuccess)
    return cuda_fail(e, "waiting for the score kernel's event");
  if (ev[0] && (e = record_event(ev[0], st)) != cudaSuccess) return cuda_fail(e, "event");
  if (sa.q16 && (e = idx::launch_q16(sa, st)) != cudaSuccess)
    return cuda_fail(e, "launching the query conversion kernel");
  e = wide ? idx::launch_wide(k_dtype, block_score, sa, map, qmap, st)
           : idx::launch_score(k_dtype, block_score, sa, map, st);
  if (e != cudaSuccess) return cuda_fail(e, "launching the score kernel");
  if (ev[1] && (e = record_event(ev[1], st)) != cudaSuccess) return cuda_fail(e, "event");
  if (fused) {
    if (wait_topk && (e = cudaStreamWaitEvent(st, wait_topk, 0)) != cudaSuccess)
      return cuda_fail(e, "waiting for the top-k kernel's event");
    if (ev[2] && (e = record_event(ev[2], st)) != cudaSuccess) return cuda_fail(e, "event");
    return IDX_OK;
  }
  if (wait_topk && (e = cudaStreamWaitEvent(st, wait_topk, 0)) != cudaSuccess)
    return cuda_fail(e, "waiting for the top-k kernel's event");
  e = idx::launch_topk(ta, st);
  if (e != cudaSuccess) {
    // the top-k kernel is what leaves the dynamic-schedule counter at zero and
    // tags it so; without it the counter may be left nonzero, so drop the tag
    // and the next call on this workspace schedules statically
    cudaGetLastError();
    (void)cudaMemsetAsync(ws + idx::kTagOff, 0, sizeof(unsigned long long), st);
    return cuda_fail(e, "launching the top-k kernel");
  }
  if (ev[2] && (e = record_event(ev[2], st)) != cudaSuccess) return cuda_fail(e, "event");
  return IDX_OK;
}

}  // namespace

namespace idx {
int record_error(int status, const char* message) { return fail(status, "%s", message); }
}  // namespace idx

extern "C" {

int idx_abi_version(void) { return IDX_ABI_VERSION; }

const char* idx_status_string(int status) {
  switch (status) {
    case IDX_OK: return "IDX_OK";
    case IDX_ERR_INVALID: return "IDX_ERR_INVALID";
    case IDX_ERR_UNSUPPORTED: return "IDX_ERR_UNSUPPORTED";
    case IDX_ERR_CUDA: return "IDX_ERR_CUDA";
    case IDX_ERR_OOM: return "IDX_ERR_OOM";
    default: return "IDX_ERR_UNKNOWN";
  }
}

const char* idx_last_error(void) { return g_last_error.c_str(); }

int idx_pool_alloc(int dtype, int64_t num_pages, int page_size, int dim, idx_pool* out) {
  if (!out) return fail(IDX_ERR_INVALID, "out is NULL");
  if (payload_row_bytes(dtype) < 0) return fail(IDX_ERR_INVALID, "unknown dtype %d", dtype);
  if (page_size != IDX_PAGE_SIZE || dim != IDX_DIM)
    return fail(IDX_ERR_INVALID, "page_size must be 64 and dim 128 (got %d, %d)", page_size, dim);
  if (num_pages < 1 || num_pages * idx::kPage > 0x7fffffffLL)
    return fail(IDX_ERR_INVALID, "num_pages must be in [1, 2^31 / 64) (got %lld)",
                (long long)num_pages);
  memset(out, 0, sizeof(*out));
  const int64_t rows = num_pages * IDX_PAGE_SIZE;
  void* payload = nullptr;
  void* scale = nullptr;
  cudaError_t e = cudaMalloc(&payload, (size_t)(rows * payload_row_bytes(dtype)));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(IDX_ERR_OOM, "cudaMalloc of the payload plane failed: %s", cudaGetErrorString(e));
  }
  if (scale_row_bytes(dtype) > 0) {
    e = cudaMalloc(&scale, (size_t)(rows * scale_row_bytes(dtype)));
    if (e != cudaSuccess) {
      cudaGetLastError();
      cudaFree(payload);
      return fail(IDX_ERR_OOM, "cudaMalloc of the scale plane failed: %s", cudaGetErrorString(e));
    }
  }
  out->dtype = dtype;
  out->page_size = page_size;
  out->dim = dim;
  out->num_pages = num_pages;
  out->payload = payload;
  out->scale = scale;
  out->payload_row_bytes = payload_row_bytes(dtype);
  out->scale_row_bytes = scale_row_bytes(dtype);
  return IDX_OK;
}

int idx_pool_free(idx_pool* pool) {
  if (!pool) return fail(IDX_ERR_INVALID, "pool is NULL");
  cudaError_t e1 = pool->payload ? cudaFree(pool->payload) : cudaSuccess;
  cudaError_t e2 = pool->scale ? cudaFree(pool->scale) : cudaSuccess;
  memset(pool, 0, sizeof(*pool));
  if (e1 != cudaSuccess) return cuda_fail(e1, "cudaFree of the payload plane");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFree of the scale plane");
  return IDX_OK;
}

int idx_store_nvfp4(const void* src_bf16, const int64_t* slot_mapping, int64_t num_tokens,
                    const idx_pool* pool, void* stream) {
  if (!pool) return fail(IDX_ERR_INVALID, "pool is NULL");
  if (pool->dtype != IDX_NVFP4 || pool->payload_row_bytes != 64 || pool->scale_row_bytes != 8 ||
      pool->page_size != IDX_PAGE_SIZE || pool->dim != IDX_DIM)
    return fail(IDX_ERR_INVALID, "pool is not an NVFP4 pool with 64-token pages of dim 128");
  if (num_tokens < 0) return fail(IDX_ERR_INVALID, "num_tokens must be >= 0");
  if (num_tokens == 0) return IDX_OK;
  if (!src_bf16 || !slot_mapping || !pool->payload || !pool->scale)
    return fail(IDX_ERR_INVALID, "a required pointer is NULL");
  if (!aligned(src_bf16, 16) || !aligned(pool->payload, 8))
    return fail(IDX_ERR_INVALID, "src_bf16 must be 16-byte and the payload 8-byte aligned");
  if (num_tokens > (int64_t)0x7fffffff * 32)
    return fail(IDX_ERR_INVALID, "num_tokens too large");
  cudaError_t e = idx::launch_store_nvfp4(
      static_cast<const uint16_t*>(src_bf16), slot_mapping, num_tokens,
      static_cast<uint8_t*>(pool->payload), static_cast<uint8_t*>(pool->scale),
      pool->num_pages * IDX_PAGE_SIZE, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the NVFP4 store kernel");
  return IDX_OK;
}

size_t idx_score_topk_workspace_bytes(int num_requests, int packed_queries, int gqa,
                                      int max_pages) {
  if (num_requests < 0 || packed_queries < 1 || gqa < 1 || max_pages < 1) return 0;
  const long long rows = (long long)num_requests * packed_queries * gqa;
  if ((long long)packed_queries * gqa > IDX_MAX_PACKED_ROWS)
    return idx::ws_q16_offset(rows, max_pages) + idx::ws_wide_bytes(rows);
  return IDX_WORKSPACE_HEADER_BYTES + idx::ws_blockmax_bytes(rows, max_pages);
}

int idx_score_topk(const void* q, const float* q_scale, int q_dtype, const void* k_payload,
                   const void* k_scale, int k_dtype, int64_t num_pages, const int32_t* page_table,
                   int n_slots, int max_pages, const int32_t* slot_ids, const int32_t* row_lens,
                   int num_requests, int packed_queries, int gqa, int init_blocks,
                   int local_blocks, int topk, int32_t* out_ids, float* out_scores,
                   void* workspace, size_t workspace_bytes, void* stream) {
  return score_topk_impl(false, idx::kBlockMax, -1, q, q_scale, q_dtype, k_payload, k_scale, k_dtype, num_pages,
                         page_table, n_slots, max_pages, slot_ids, row_lens, num_requests,
                         packed_queries, gqa, init_blocks, local_blocks, topk, out_ids,
                         out_scores, workspace, workspace_bytes, stream);
}

int idx_score_topk_lse(const void* q, const float* q_scale, int q_dtype, const void* k_payload,
                       const void* k_scale, int k_dtype, int64_t num_pages,
                       const int32_t* page_table, int n_slots, int max_pages,
                       const int32_t* slot_ids, const int32_t* row_lens, int num_requests,
                       int packed_queries, int gqa, int init_blocks, int local_blocks, int topk,
                       int32_t* out_ids, float* out_scores, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return score_topk_impl(false, idx::kBlockLse, -1, q, q_scale, q_dtype, k_payload, k_scale, k_dtype,
                         num_pages, page_table, n_slots, max_pages, slot_ids, row_lens,
                         num_requests, packed_queries, gqa, init_blocks, local_blocks, topk,
                         out_ids, out_scores, workspace, workspace_bytes, stream);
}

int idx_score_topk_perrow(const void* q, const float* q_scale, int q_dtype, const void* k_payload,
                          const void* k_scale, int k_dtype, int64_t num_pages,
                          const int32_t* page_table, int n_slots, int max_pages,
                          const int32_t* slot_ids, const int32_t* row_lens, int num_requests,
                          int packed_queries, int gqa, int init_blocks, int local_blocks,
                          int topk, int32_t* out_ids, float* out_scores, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return score_topk_impl(true, idx::kBlockMax, -1, q, q_scale, q_dtype, k_payload, k_scale, k_dtype, num_pages,
                         page_table, n_slots, max_pages, slot_ids, row_lens, num_requests,
                         packed_queries, gqa, init_blocks, local_blocks, topk, out_ids,
                         out_scores, workspace, workspace_bytes, stream);
}

int idx_set_wait_limit_ns(uint64_t ns) {
  idx::set_wait_limit_ns(ns);
  return IDX_OK;
}

int idx_set_stall_test(int on) {
  idx::set_stall_test(on);
  return IDX_OK;
}

int idx_set_grid_limit(int max_ctas) {
  if (max_ctas < 0) return fail(IDX_ERR_INVALID, "max_ctas must be >= 0");
  idx::set_grid_limit(max_ctas);
  return IDX_OK;
}

int idx_set_kernel_events(void* score_begin, void* score_end, void* topk_end) {
  g_ev[0] = static_cast<cudaEvent_t>(score_begin);
  g_ev[1] = static_cast<cudaEvent_t>(score_end);
  g_ev[2] = static_cast<cudaEvent_t>(topk_end);
  return IDX_OK;
}

int idx_set_kernel_waits(void* before_score, void* before_topk) {
  g_wait[0] = static_cast<cudaEvent_t>(before_score);
  g_wait[1] = static_cast<cudaEvent_t>(before_topk);
  return IDX_OK;
}

int idx_workspace_errors(const void* workspace, void* stream, uint32_t* flags) {
  if (!workspace || !flags) return fail(IDX_ERR_INVALID, "a required pointer is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t header[IDX_WORKSPACE_HEADER_BYTES];
  cudaError_t e = cudaMemcpyAsync(header, workspace, sizeof(header), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace header");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "synchronising the stream");
  uint32_t n = 0;
  memcpy(&n, header, sizeof(n));
  if (n > (uint32_t)idx::kMaxScoreCtas) n = idx::kMaxScoreCtas;
  uint32_t f = 0;
  for (uint32_t c = 0; c < n; ++c) f |= header[idx::kFlagBytesOff + c];
  *flags = f;
  return IDX_OK;
}

int idx_score_local_blocks(const void* q, const float* q_scale, int q_dtype,
                           const void* k_payload, const void* k_scale, int k_dtype,
                           int64_t num_pages, const int32_t* page_table, int n_slots,
                           int max_pages, int block_begin, const int32_t* slot_ids,
                           const int32_t* row_lens, int num_requests, int packed_queries, int gqa,
                           int init_blocks, int local_blocks, int topk, int32_t* out_ids,
                           float* out_scores, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (block_begin < 0)
    return fail(IDX_ERR_INVALID, "block_begin must be >= 0 (got %d)", block_begin);
  return score_topk_impl(false, idx::kBlockMax, block_begin, q, q_scale, q_dtype, k_payload,
                         k_scale, k_dtype, num_pages, page_table, n_slots, max_pages, slot_ids,
                         row_lens, num_requests, packed_queries, gqa, init_blocks, local_blocks,
                         topk, out_ids, out_scores, workspace, workspace_bytes, stream);
}

int idx_topk_merge(const int32_t* cand_ids, const float* cand_scores, int world,
                   const int32_t* slot_ids, const int32_t* row_lens, int n_slots,
                   int num_requests, int packed_queries, int gqa, int init_blocks,
                   int local_blocks, int topk, int32_t* out_ids, float* out_scores,
                   void* stream) {
  const int R = num_requests, P = packed_queries, G = gqa;
  if (world < 1 || world > IDX_MAX_CP_WORLD)
    return fail(IDX_ERR_INVALID, "world must be in [1, %d] (got %d)", IDX_MAX_CP_WORLD, world);
  if (R < 0 || R > IDX_MAX_REQUESTS)
    return fail(IDX_ERR_INVALID, "num_requests must be in [0, %d] (got %d)", IDX_MAX_REQUESTS, R);
  if (P < 1 || G < 1 || (long long)P * G > IDX_MAX_ROWS_PER_REQUEST)
    return fail(IDX_ERR_INVALID, "packed_queries * gqa must be in [1, %d] (got %d x %d)",
                IDX_MAX_ROWS_PER_REQUEST, P, G);
  if (topk < 1 || topk > IDX_MAX_TOPK)
    return fail(IDX_ERR_INVALID, "topk must be in [1, %d] (got %d)", IDX_MAX_TOPK, topk);
  if (init_blocks < 0 || local_blocks < 0 || init_blocks + local_blocks > topk)
    return fail(IDX_ERR_INVALID,
                "need init_blocks, local_blocks >= 0 and init + local <= topk (got %d, %d, %d)",
                init_blocks, local_blocks, topk);
  if (n_slots < 1) return fail(IDX_ERR_INVALID, "n_slots must be >= 1 (got %d)", n_slots);
  if (R > 0 && (!cand_ids || !cand_scores || !slot_ids || !row_lens || !out_ids || !out_scores))
    return fail(IDX_ERR_INVALID, "a required pointer is NULL");
  if (R == 0) return IDX_OK;
  idx::MergeArgs m;
  m.cand_ids = cand_ids;
  m.cand_scores = cand_scores;
  m.slot_ids = slot_ids;
  m.row_lens = row_lens;
  m.out_ids = out_ids;
  m.out_scores = out_scores;
  m.world = world;
  m.n_slots = n_slots;
  m.R = R;
  m.P = P;
  m.G = G;
  m.M = P * G;
  m.init_blocks = init_blocks;
  m.local_blocks = local_blocks;
  m.topk = topk;
  cudaError_t e = idx::launch_merge(m, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the merge kernel");
  return IDX_OK;
}

}  // extern "C"

// idx_score_topk_noalloc: the packed index step for callers that cannot allocate
// device memory.  The block-score scratch lives in a fixed, file-scope device
// array instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/idx.h"
#include "idx_internal.cuh"

namespace {

// Scratch shared by every call in this process, on every device that loads the
// library: it is resident from module load until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[IDX_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's name
// is only a host-side stand-in, so the address comes from cudaGetSymbolAddress,
// once per device, with that device current.
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int idx_score_topk_noalloc(const void* q, const float* q_scale, int q_dtype,
                                      const void* k_payload, const void* k_scale, int k_dtype,
                                      int64_t num_pages, const int32_t* page_table, int n_slots,
                                      int max_pages, const int32_t* slot_ids,
                                      const int32_t* row_lens, int num_requests,
                                      int packed_queries, int gqa, int init_blocks,
                                      int local_blocks, int topk, int32_t* out_ids,
                                      float* out_scores, void* stream) {
  const size_t need =
      idx_score_topk_workspace_bytes(num_requests, packed_queries, gqa, max_pages);
  if (need == 0)
    return idx::record_error(IDX_ERR_INVALID,
                             "idx_score_topk_noalloc: num_requests must be >= 0 and "
                             "packed_queries, gqa, max_pages >= 1");
  if (need > (size_t)IDX_NOALLOC_SCRATCH_BYTES)
    return idx::record_error(IDX_ERR_INVALID,
                             "idx_score_topk_noalloc: this call needs more scratch than the "
                             "fixed array holds (num_requests * packed_queries * gqa * "
                             "ceil(max_pages / 2) * 4 + IDX_WORKSPACE_HEADER_BYTES must be <= "
                             "IDX_NOALLOC_SCRATCH_BYTES); use idx_score_topk with a workspace");
  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess)
    return idx::record_error(IDX_ERR_CUDA,
                             "idx_score_topk_noalloc: cudaGetSymbolAddress of the scratch array "
                             "failed");
  return idx_score_topk(q, q_scale, q_dtype, k_payload, k_scale, k_dtype, num_pages, page_table,
                        n_slots, max_pages, slot_ids, row_lens, num_requests, packed_queries, gqa,
                        init_blocks, local_blocks, topk, out_ids, out_scores, scratch,
                        IDX_NOALLOC_SCRATCH_BYTES, stream);
}

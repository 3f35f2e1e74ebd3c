// idx_score_topk_noalloc: the packed index step for callers that cannot allocate
// device memory.  The block-score scratch lives in a fixed, file-scope device
// array instead of a caller-provided workspace.
#include <cuda.h>
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
// Per device: the array's device address and the context it was looked up in.
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// cuCtxGetCurrent through the runtime's driver entry point (no link-time
// dependency on the driver library); null if the driver does not offer it.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch array on the current device.  The array's name
// is only a host-side stand-in, so the address comes from cudaGetSymbolAddress,
// with that device current, once per device -- and again if the device's
// context has been torn down and made anew since (cudaDeviceReset), when the
// module holding the array is loaded again at another address.
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrentFn get_ctx = ctx_get_current();
  CUcontext ctx = nullptr;  // stays null until the runtime has made the context
  if (get_ctx) get_ctx(&ctx);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev] || !ctx || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the context if needed
    if (e != cudaSuccess) return e;
    ctx = nullptr;
    if (get_ctx) get_ctx(&ctx);
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
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

extern "C" int idx_noalloc_errors(void* stream, uint32_t* flags) {
  if (!flags) return idx::record_error(IDX_ERR_INVALID, "idx_noalloc_errors: flags is NULL");
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess)
    return idx::record_error(IDX_ERR_CUDA,
                             "idx_noalloc_errors: cudaGetSymbolAddress of the scratch array "
                             "failed");
  return idx_workspace_errors(scratch, stream, flags);
}

// Shared declarations between the kernel translation units and the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace idx {

constexpr int kPage = 64;     // tokens per page
constexpr int kBlock = 128;   // tokens per scored block
constexpr int kDim = 128;     // head dim
constexpr int kTileRows = 16; // packed rows per dot tile
constexpr int kMaxTopk = 256; // largest topk a call may ask for
// Workspace header: word 0 = number of score CTAs of the last call; bytes
// [kSchedOff, kSchedOff + 4) = the block counter of the dynamic schedule and
// [kTagOff, kTagOff + 8) = kSchedTag once a call has left that counter at zero;
// bytes [kFlagBytesOff, kFlagBytesOff + CTAs) = each CTA's device error flags.
constexpr int kHeaderBytes = 1024;
constexpr int kSchedOff = 8;
constexpr int kTagOff = 16;
constexpr int kArriveOff = 24;  // in-kernel selection only: grid barrier counters
constexpr int kDepartOff = 28;
constexpr int kFlagBytesOff = 64;
constexpr int kMaxScoreCtas = kHeaderBytes - kFlagBytesOff;
constexpr unsigned long long kSchedTag = 0x5CEDC0DE1DC0FFEEull;
// Scoring groups a call may have (requests when packed, draft rows when per-row):
// the score kernel keeps one prefix-sum entry and one slot per group in shared
// memory.
constexpr int kMaxGroups = 2048;

// Key formats, matching idx_dtype.
enum KeyFormat : int { kBf16 = 0, kFp8 = 1, kNvfp4 = 2 };
// Block scores: the block's largest score, or the log-sum-exp of its scores.
enum BlockScore : int { kBlockMax = 0, kBlockLse = 1 };

struct TopkArgs {
  const float* blockmax;       // [R*M][nb_cap]
  const int32_t* slot_ids;
  const int32_t* row_lens;
  int32_t* out_ids;            // [R*M][topk]
  float* out_scores;
  uint32_t* sched_counter;     // reset to zero for the next call
  unsigned long long* sched_tag;
  int n_slots, max_pages, nb_cap;
  int R, P, G, M;
  int init_blocks, local_blocks, topk;
  int block_off;               // first global block the workspace's block 0 stands for
  int shard;                   // 1: select within the shard [block_off, block_off + nb_cap)
};

// Selection inside the score kernel instead of the separate top-k kernel: one
// launch per step, the score CTAs meet at a grid barrier (bounded wait) and
// then select the rows, CTA k taking rows k, k + grid, ...  Off: measured
// slower on every decode workload (one GB300, graph replays: bf16 16 x 131K
// 83.2 -> 90.3 us a step, fp8 16 x 131K 54.2 -> 61.2, NVFP4 64 x 150K
// 157.8 -> 182.4, fp8 32 x 524K 330.9 -> 353.8, before the per-call counter
// reset this build also needs), since each SM then selects its rows in turn
// with one score CTA and the next step cannot start under the selection.
// Build with -DIDX_FUSED_TOPK=1 to try it.
#ifndef IDX_FUSED_TOPK
#define IDX_FUSED_TOPK 0
#endif

// Arguments of one scoring pass.  A "group" is the set of tile rows that share
// one read of the keys: a whole request when packed, one draft row when per-row.
// Workspace layout: the header, the block scores, and for the wide path (more
// than 16 packed rows) the f16 query rows and their scales from the next
// 256-byte boundary.
inline size_t ws_blockmax_bytes(long long rows, int max_pages) {
  return (size_t)rows * (size_t)((max_pages + 1) / 2) * sizeof(float);
}
inline size_t ws_q16_offset(long long rows, int max_pages) {
  return (kHeaderBytes + ws_blockmax_bytes(rows, max_pages) + 255) & ~(size_t)255;
}
inline size_t ws_wide_bytes(long long rows) { return (size_t)rows * (256 + sizeof(float)); }

struct ScoreArgs {
  const uint8_t* q;            // [R][P][G][128] bf16 or e4m3
  const float* q_scale;        // [R][P*G] (e4m3 q) or nullptr
  const uint8_t* k_scale;      // scale plane (fp8: 4 B / key, NVFP4: 8 B / key)
  const int32_t* page_table;   // [n_slots][max_pages]
  const int32_t* slot_ids;     // [R]
  const int32_t* row_lens;     // [R][P]
  float* blockmax;             // [R*P*G][nb_cap]
  uint16_t* q16;               // wide path, NVFP4 keys: f16 query rows [R*P*G][128]
  float* qpost;                // and the factor undoing each row's power-of-two scale
  uint8_t* err_bytes;          // one flag byte per CTA
  uint32_t* err_count;         // CTAs that wrote a flag byte
  uint32_t* sched_counter;     // dynamic-schedule block counter (zero at entry)
  const unsigned long long* sched_tag;  // kSchedTag when the counter is valid
  int64_t num_pages;
  int n_slots, max_pages, nb_cap;
  int R, P, G, M;
  int perrow;                  // 0: groups are requests; 1: groups are draft rows
  int tiles;                   // wide path: 128-row tiles per request (groups = R * tiles)
  int block_off;               // global block of local block 0 (a context shard); 0 otherwise
  int shard;                   // 1: the page table holds one context shard of each request
  unsigned long long wait_ns;  // limit of each pipeline wait before IDX_DEVERR_TIMEOUT
  int stall_test;              // diagnostic: one role per CTA waits on a barrier nothing completes
#if IDX_FUSED_TOPK
  int fused;                   // 1: select in this kernel (16-row packed whole-context calls)
  TopkArgs topk;               // the selection the CTAs run after a grid barrier
  uint32_t* arrive;            // grid barrier: CTAs arrived (zero between calls)
  uint32_t* depart;            // CTAs done selecting; the last resets both counters
#endif
};


// Merge of context shards' candidate lists: cand_* are [world][R*M][topk].
struct MergeArgs {
  const int32_t* cand_ids;
  const float* cand_scores;
  const int32_t* slot_ids;
  const int32_t* row_lens;
  int32_t* out_ids;
  float* out_scores;
  int world, n_slots;
  int R, P, G, M;
  int init_blocks, local_blocks, topk;
};

// ---- host-side launch helpers: keep a call's CPU cost to its launches -------
// Streaming multiprocessors of device `dev`, looked up once per device.
inline int cached_sm_count(int dev) {
  static std::atomic<int> cache[64];
  int n = 0;
  if (dev >= 0 && dev < 64) n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Once per device (`done` is a per-kernel bit mask of the devices already set):
// raise a kernel's dynamic shared-memory limit to `bytes` (when > 0) and ask for
// the largest shared-memory carveout.  Every kernel of the step prefers the same
// carveout, so a programmatic dependent can become resident on an SM beside the
// grid it follows instead of waiting for that SM to be reconfigured.
template <class Kernel>
inline cudaError_t smem_limit_once(Kernel kernel, int bytes, int dev,
                                   std::atomic<unsigned long long>& done) {
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  if (bytes > 0)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launch as a programmatic dependent of the previous kernel on the stream: the
// grid may become resident while that kernel finishes (once all its CTAs have
// signalled griddepcontrol.launch_dependents or exited) and must execute
// griddepcontrol.wait before it touches memory the earlier work writes.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int threads, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Record an error message for idx_last_error() on this host thread; returns status.
int record_error(int status, const char* message);

// Process-wide limit of the score kernels' pipeline waits (default 2 s).
void set_wait_limit_ns(unsigned long long ns);
unsigned long long wait_limit_ns();
void set_stall_test(int on);
int stall_test();

// Process-wide cap on the score kernel's grid (0 = one CTA per SM).
void set_grid_limit(int max_ctas);
int grid_limit();

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_score(int key_format, int block_score, const ScoreArgs& args,
                         const CUtensorMap& payload_map, cudaStream_t stream);
// Requests of more than 16 packed rows: 128-row tiles on tcgen05 (q_map: the
// query rows [R*M][128] as bf16 or e4m3, or for NVFP4 keys the f16 rows
// launch_q16 writes to args.q16).
// Wide path with NVFP4 keys: the query rows to f16 (args.q16, args.qpost),
// launched before the wide kernel.
cudaError_t launch_q16(const ScoreArgs& args, cudaStream_t stream);
cudaError_t launch_wide(int key_format, int block_score, const ScoreArgs& args,
                        const CUtensorMap& payload_map, const CUtensorMap& q_map,
                        cudaStream_t stream);
cudaError_t launch_topk(const TopkArgs& args, cudaStream_t stream);
cudaError_t launch_merge(const MergeArgs& args, cudaStream_t stream);
cudaError_t launch_store_nvfp4(const uint16_t* src, const int64_t* slot_mapping, int64_t num_tokens,
                               uint8_t* payload, uint8_t* scale, int64_t num_rows,
                               cudaStream_t stream);

}  // namespace idx

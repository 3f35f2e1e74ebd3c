// Block top-k select and the context-shard merge.  Three kernels: one CTA
// (eight warps) per packed output row for long rows or few rows; one warp per
// row for many rows of at most 256 blocks; one warp per row merging the lists
// of context shards.
//
// What it computes (sglang #42614 "[AMD] MiniMax-M3 indexer CP: packed scoring
// for EAGLE verify rows", Modifications 1 and Accuracy Tests; sglang #45451,
// Accuracy Tests): the row always keeps its first init_blocks and last
// local_blocks blocks, counted from its own length, and fills the rest of topk
// with the best remaining blocks by block max; selection is exact.  Ties go to
// the lower block id.  Output: forced blocks ascending, chosen blocks by
// descending score, then (-1, -inf) pads.
//
// How (CTA per row): the non-forced candidates form one contiguous id range.
// Their block maxima are read from L2 with as many loads in flight per thread
// as the row needs and kept in shared memory as order-preserving 32-bit keys.
// When there are many candidates, most-significant-digit radix passes (8-bit
// digits starting below the bits every candidate shares, one shared 256-bin
// histogram per digit) narrow them to the keys at or above the threshold's
// bin, usually after one pass.  Each remaining (key, id) entry is then placed
// by its rank among them, ties going to the lower id; entries ranked c or later
// are dropped.  (A second pass, one warp sorting the entries with a bitonic
// network, and several threads sharing each entry's count all measured slower
// in the step.)  The score written out is recovered from the key, so nothing
// is read back from memory.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "idx_internal.cuh"
#include "idx_select.cuh"

namespace idx {

namespace {

using sel::kBatch;
using sel::kCap;
using sel::key_value;
using sel::order_key;
using sel::pack;
using sel::row_plan;
using sel::RowPlan;

constexpr int kThreads = 256;
constexpr int kMaxWorld = 8;  // context shards a merge accepts

// Descending bitonic sort of 32 E values (32- or 64-bit) held by one warp,
// element e = lane + 32 h in x[h] (E a power of two).  Partners closer than 32
// are exchanged by shuffles, farther ones inside the lane's registers.
template <int E, class T>
__device__ __forceinline__ void warp_sort_desc(T (&x)[E], int lane) {
#pragma unroll
  for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        const int hj = j >> 5;
#pragma unroll
        for (int h = 0; h < E; ++h) {
          if ((h & hj) == 0) {
            // pair (e, e + j), e = lane + 32 h; (e & k) depends on h alone
            const bool desc = ((32 * h) & k) == 0;
            const T a = x[h], b = x[h | hj];
            const bool swap = desc ? a < b : a > b;
            x[h] = swap ? b : a;
            x[h | hj] = swap ? a : b;
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < E; ++h) {
          const int e = lane + 32 * h;
          const T y = __shfl_xor_sync(0xffffffffu, x[h], j);
          // the lower index of a descending run keeps the larger value
          const bool take_max = ((e & j) == 0) == ((e & k) == 0);
          x[h] = take_max ? (x[h] > y ? x[h] : y) : (x[h] > y ? y : x[h]);
        }
      }
    }
  }
}

// Sorts list[0, n) (n <= 32 E) in one warp and writes entries of rank < c to
// the outputs at nf + rank.  Unused slots hold 0, below every (key, id) entry.
template <int E>
__device__ __forceinline__ void warp_place_sorted(const unsigned long long* list, int n, int c,
                                                  int nf, int lane, int32_t* out_ids,
                                                  float* out_sc) {
  unsigned long long x[E];
#pragma unroll
  for (int h = 0; h < E; ++h) x[h] = lane + 32 * h < n ? list[lane + 32 * h] : 0ull;
  warp_sort_desc<E>(x, lane);
#pragma unroll
  for (int h = 0; h < E; ++h) {
    const int e = lane + 32 * h;
    if (e < n && e < c) {
      out_ids[nf + e] = 0x7fffffff - (int)(uint32_t)(x[h] & 0xffffffffull);
      out_sc[nf + e] = key_value((uint32_t)(x[h] >> 32));
    }
  }
}


// kMinCtas = 8 caps registers at 32 so that eight rows share an SM (more than
// six rows per SM: one wave instead of two); 0 (no minimum) leaves the
// compiler the registers that keep a long row's loads in flight, measured
// faster for a few hundred rows of ~1000 blocks.  NT is the row's threads.
template <int kMinCtas, int NT>
__global__ void __launch_bounds__(NT, kMinCtas) topk_kernel(const TopkArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int tid = threadIdx.x;
  // the next call's score kernel may become resident as soon as every row of
  // this grid has started (it waits for this grid to finish before it reads)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int row = blockIdx.x;
  const int r = row / a.M;
  const RowPlan pl = row_plan(a, r, row - r * a.M);
  // pads need no block maxima: write them before waiting on the score kernel
  sel::row_pads<NT>(a, row, pl, tid);
  // launched as a programmatic dependent of the score kernel: wait for its
  // completion before touching the block maxima
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the score kernel is done: leave its block counter at zero for the next call
  if (row == 0 && tid == 0) {
    *reinterpret_cast<volatile uint32_t*>(a.sched_counter) = 0u;
    *reinterpret_cast<volatile unsigned long long*>(a.sched_tag) = kSchedTag;
  }
  sel::row_select<NT, false>(a, row, pl, smem_raw, tid);
}

// ---------------------------------------------------------------------------
// Rows of at most 32 * R blocks (short contexts, many rows: prefill chunks, wide
// verify): one warp per row, four rows per CTA, no block-wide barrier.  The
// row's candidate keys live in registers (element e = lane + 32 r is block
// fi + e); radix passes of up to 8 bits over a warp-private 256-bin histogram,
// starting below the bits every candidate shares, narrow to the threshold's
// bin: when that bin is taken whole they stop; otherwise they end at the exact
// c-th largest key T, keys above T are taken, and of the keys equal to T the
// lowest ids, counted with ballots in id order.  The chosen entries are
// compacted in id order and ordered by (key desc, id asc): up to 64 of them by
// a bitonic sort in registers, more by each one's rank among them.
// Same selection, outputs and score recovery as topk_kernel.
// ---------------------------------------------------------------------------
// Four rows per CTA and one 2 KB slot per warp (histogram while the threshold
// is found, then the chosen list): 8 KB, small enough to sit beside a score CTA
// on the same SM, so the programmatic launch still overlaps the score's tail.
constexpr int kRowsPerCta = 4;

union WarpSlot {
  uint32_t hist[256];
  unsigned long long list[256];
};

template <int R>
__global__ void __launch_bounds__(32 * kRowsPerCta) topk_warp_kernel(const TopkArgs a) {
  __shared__ WarpSlot sh[kRowsPerCta];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x * kRowsPerCta + warp;
  if (row >= a.R * a.M) return;
  uint32_t* hist = sh[warp].hist;
  unsigned long long* list = sh[warp].list;
  const int r = row / a.M;
  const int i = row - r * a.M;
  int32_t* out_ids = a.out_ids + (size_t)row * a.topk;
  float* out_sc = a.out_scores + (size_t)row * a.topk;
  const float* bm = a.blockmax + (size_t)row * a.nb_cap;

  const RowPlan pl = row_plan(a, r, i);
  const int nf = pl.nf, ncand = pl.ncand, c = pl.c;
  const int fi = pl.cb;  // global id of the first candidate
  // the workspace holds this row's blocks from s0 on: block g at g - s0
  const float* bmg = bm - pl.s0;

  for (int t = nf + max(c, 0) + lane; t < a.topk; t += 32) {
    out_ids[t] = -1;
    out_sc[t] = -INFINITY;
  }
  // the block scores are written by the score kernel this grid depends on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (row == 0 && lane == 0) {
    *reinterpret_cast<volatile uint32_t*>(a.sched_counter) = 0u;
    *reinterpret_cast<volatile unsigned long long*>(a.sched_tag) = kSchedTag;
  }
  for (int t = lane; t < nf; t += 32) {
    const int id = pl.forced_id(t);
    out_ids[t] = id;
    out_sc[t] = bmg[id];
  }
  if (c <= 0) return;

  uint32_t key[R];
  bool act[R];
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const int e = lane + 32 * q;
    act[q] = e < ncand;
    key[q] = act[q] ? order_key(bmg[fi + e]) : 0u;
  }
  bool sel[R];
#pragma unroll
  for (int q = 0; q < R; ++q) sel[q] = act[q];
  if (ncand > c) {
    // ---- threshold: radix passes of up to 8 bits, starting below the bits
    // all candidates share, until the threshold's bin is taken whole or the
    // exact c-th largest key T is known --------------------------------------
    uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
    for (int q = 0; q < R; ++q)
      if (act[q]) {
        kmin = min(kmin, key[q]);
        kmax = max(kmax, key[q]);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    int hi = 32 - __clz(kmin ^ kmax);  // bits [hi, 32) are common to all candidates
    uint32_t pmask = hi >= 32 ? 0u : (0xffffffffu << hi);
    uint32_t prefix = kmax & pmask, need = (uint32_t)c;
    bool whole_bin = false;
#pragma unroll 1
    while (hi > 0) {
      const int lo = max(hi - 8, 0);
      const uint32_t dmask = (1u << (hi - lo)) - 1u;
#pragma unroll
      for (int k = 0; k < 8; ++k) hist[lane * 8 + k] = 0u;
      __syncwarp();
#pragma unroll
      for (int q = 0; q < R; ++q)
        if (act[q] && (key[q] & pmask) == prefix) atomicAdd(&hist[(key[q] >> lo) & dmask], 1u);
      __syncwarp();
      // lane l owns bins 255 - 8 l - e, e = 0..7 (highest digits first)
      uint32_t loc[8];
      uint32_t sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        loc[e] = hist[255 - 8 * lane - e];
        sum += loc[e];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - sum;
      const bool mine = excl < need && need <= incl;
      uint32_t digit = 0, left = 0, inbin = 0;
      if (mine) {
        uint32_t above = excl;
        bool found = false;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (!found && above + loc[e] >= need) {
            digit = (uint32_t)(255 - 8 * lane - e);
            left = need - above;
            inbin = loc[e];
            found = true;
          }
          above += loc[e];
        }
      }
      const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
      digit = __shfl_sync(0xffffffffu, digit, src);
      need = __shfl_sync(0xffffffffu, left, src);
      inbin = __shfl_sync(0xffffffffu, inbin, src);
      prefix |= digit << lo;
      pmask |= dmask << lo;
      hi = lo;
      __syncwarp();  // every lane has read the histogram before it is reused
      if (need == inbin) {  // the whole threshold bin is chosen
        whole_bin = true;
        break;
      }
    }
    if (whole_bin) {
#pragma unroll
      for (int q = 0; q < R; ++q) sel[q] = act[q] && (key[q] & pmask) >= prefix;
    } else {
      // T = prefix exactly: keys above it, then the `need` lowest ids equal to it
      uint32_t base = 0;
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const bool eq = act[q] && key[q] == prefix;
        const unsigned m = __ballot_sync(0xffffffffu, eq);
        const uint32_t rk = base + __popc(m & ((1u << lane) - 1u));
        sel[q] = act[q] && (key[q] > prefix || (eq && rk < need));
        base += __popc(m);
      }
    }
  }
  // ---- compact the chosen entries in id order, then place each by rank -----
  int n = 0;
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const unsigned m = __ballot_sync(0xffffffffu, sel[q]);
    if (sel[q]) list[n + __popc(m & ((1u << lane) - 1u))] = pack(key[q], fi + lane + 32 * q);
    n += __popc(m);
  }
  __syncwarp();
  if (n <= 64) {
    // When the chosen keys differ only in their low 26 bits or fewer, each
    // entry sorts as one 32-bit word: those bits, then 63 - its position in
    // the list (the list is in id order, so equal keys keep the lower id
    // first); otherwise as (key, id) pairs.
    uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = lane + 32 * h;
      if (e < n) {
        const uint32_t k = (uint32_t)(list[e] >> 32);
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    const int vbits = 32 - __clz(kmin ^ kmax);  // 0 when every key is equal
    if (vbits > 26) {
      warp_place_sorted<2>(list, n, n, nf, lane, out_ids, out_sc);
      return;
    }
    const uint32_t vmask = (1u << vbits) - 1u;
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = lane + 32 * h;
      // unused slots sort last: a used one is at least 63 - (n - 1) >= 1
      w[h] = e < n ? ((((uint32_t)(list[e] >> 32)) & vmask) << 6) | (uint32_t)(63 - e) : 0u;
    }
    warp_sort_desc<2>(w, lane);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = lane + 32 * h;  // rank
      if (r < n) {
        const unsigned long long x = list[63 - (int)(w[h] & 63u)];
        out_ids[nf + r] = 0x7fffffff - (int)(uint32_t)(x & 0xffffffffull);
        out_sc[nf + r] = key_value((uint32_t)(x >> 32));
      }
    }
    return;
  }
  for (int j = lane; j < n; j += 32) {
    const unsigned long long x = list[j];
    int rank = 0;
#pragma unroll 8
    for (int k = 0; k < n; ++k) rank += list[k] > x ? 1 : 0;
    out_ids[nf + rank] = 0x7fffffff - (int)(uint32_t)(x & 0xffffffffull);
    out_sc[nf + rank] = key_value((uint32_t)(x >> 32));
  }
}

template <int R>
cudaError_t launch_topk_warp(const TopkArgs& a, int rows, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = smem_limit_once(topk_warp_kernel<R>, 0, dev, attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(topk_warp_kernel<R>, (rows + kRowsPerCta - 1) / kRowsPerCta,
                    32 * kRowsPerCta, 0, stream, a);
}

// ---------------------------------------------------------------------------
// Merge of context shards' lists (indexer context parallelism, the exchange
// step after each rank scored its shard; sglang #42614 names the per-shard
// scorer score_local_blocks).  One warp per row, four rows per CTA.  Each
// shard's list is its forced blocks, then its chosen candidates in (score desc,
// id asc) order, then pads; a forced block goes straight to its slot in the
// row's forced order, and a candidate's place among all shards' candidates is
// its place in its own list plus, for every other shard, how many of that
// shard's candidates rank above it (binary search, the lists being sorted).
// Candidates placed c or later are dropped.  The shards must partition the
// row's blocks, so each forced block appears in exactly one list.
// ---------------------------------------------------------------------------
constexpr int kMergeRowsPerCta = 4;

__global__ void __launch_bounds__(32 * kMergeRowsPerCta) merge_kernel(const MergeArgs a) {
  __shared__ int sh_nf[kMergeRowsPerCta][kMaxWorld];
  __shared__ int sh_nc[kMergeRowsPerCta][kMaxWorld];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = a.R * a.M;
  const int row = blockIdx.x * kMergeRowsPerCta + warp;
  if (row >= rows) return;
  const int r = row / a.M;
  const int i = row - r * a.M;
  const int slot = __ldg(a.slot_ids + r);
  const int L = (slot >= 0 && slot < a.n_slots) ? __ldg(a.row_lens + r * a.P + i / a.G) : 0;
  const int nb = L > 0 ? (L + kBlock - 1) / kBlock : 0;
  const int fi = min(a.init_blocks, nb);
  const int ls = max(fi, nb - a.local_blocks);
  const int nf = fi + (nb - ls);
  const int c = min(a.topk, nb) - nf;
  int32_t* out_ids = a.out_ids + (size_t)row * a.topk;
  float* out_sc = a.out_scores + (size_t)row * a.topk;
  for (int t = lane; t < a.topk; t += 32) {
    out_ids[t] = -1;
    out_sc[t] = -INFINITY;
  }
  // the lists are written by the shards' top-k (or copied in by the exchange)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  auto ids_of = [&](int w) { return a.cand_ids + ((size_t)w * rows + row) * a.topk; };
  auto sc_of = [&](int w) { return a.cand_scores + ((size_t)w * rows + row) * a.topk; };
  auto forced = [&](int id) { return id < fi || (id >= ls && id < nb); };
  for (int w = 0; w < a.world; ++w) {
    const int32_t* ids = ids_of(w);
    int nfw = 0, ncw = 0;
    for (int p = lane; p < a.topk; p += 32) {
      const int id = ids[p];
      if (id >= 0) {
        if (forced(id)) ++nfw;
        else ++ncw;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      nfw += __shfl_xor_sync(0xffffffffu, nfw, o);
      ncw += __shfl_xor_sync(0xffffffffu, ncw, o);
    }
    if (lane == 0) {
      sh_nf[warp][w] = nfw;
      sh_nc[warp][w] = ncw;
    }
  }
  __syncwarp();  // the pads above are written, the list sizes visible
  for (int e = lane; e < a.world * a.topk; e += 32) {
    const int w = e / a.topk, p = e - w * a.topk;
    const int id = ids_of(w)[p];
    if (id < 0) continue;
    const float v = sc_of(w)[p];
    if (forced(id)) {
      const int pos = id < fi ? id : fi + (id - ls);
      out_ids[pos] = id;
      out_sc[pos] = v;
      continue;
    }
    const unsigned long long x = pack(order_key(v), id);
    int rank = p - sh_nf[warp][w];
    for (int w2 = 0; w2 < a.world; ++w2) {
      if (w2 == w) continue;
      const int32_t* ids2 = ids_of(w2);
      const float* sc2 = sc_of(w2);
      int lo = sh_nf[warp][w2], hi = lo + sh_nc[warp][w2];
      const int base = lo;
      while (lo < hi) {  // first entry not above x (the list is descending)
        const int mid = (lo + hi) >> 1;
        if (pack(order_key(sc2[mid]), ids2[mid]) > x) lo = mid + 1;
        else hi = mid;
      }
      rank += lo - base;
    }
    if (rank < c) {
      out_ids[nf + rank] = id;
      out_sc[nf + rank] = v;
    }
  }
}

}  // namespace

template <int kMinCtas, int NT>
cudaError_t launch_topk_cta(const TopkArgs& a, int rows, cudaStream_t stream) {
  const size_t smem = sel::smem_bytes<NT>(a.nb_cap);
  // the limit is raised once per device to what the largest page table
  // (65536 pages: 32768 blocks) can need; each launch asks for its own size
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = smem_limit_once(topk_kernel<kMinCtas, NT>, (int)sel::smem_bytes<NT>(32768), dev,
                      attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, topk_kernel<kMinCtas, NT>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  const int rows = a.R * a.M;
  if (rows == 0) return cudaSuccess;
  // many short rows: a warp per row (measured: below about 16 rows per SM the
  // CTA-per-row kernel's shorter per-row latency wins)
  int cur = 0;
  if (cudaGetDevice(&cur) == cudaSuccess && rows >= 16 * cached_sm_count(cur)) {
    if (a.nb_cap <= 64) return launch_topk_warp<2>(a, rows, stream);
    if (a.nb_cap <= 128) return launch_topk_warp<4>(a, rows, stream);
    if (a.nb_cap <= 256) return launch_topk_warp<8>(a, rows, stream);
  }
  if (rows > 6 * cached_sm_count(cur)) return launch_topk_cta<8, kThreads>(a, rows, stream);
  // at most two rows per SM: 512 threads a row (measured 0.6 us off a 16 x
  // 131K bf16 step; more rows per SM were slower with them)
  if (rows <= 2 * cached_sm_count(cur)) return launch_topk_cta<0, 2 * kThreads>(a, rows, stream);
  return launch_topk_cta<0, kThreads>(a, rows, stream);
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int rows = a.R * a.M;
  if (rows == 0) return cudaSuccess;
  if (a.world < 1 || a.world > kMaxWorld) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(merge_kernel, (rows + kMergeRowsPerCta - 1) / kMergeRowsPerCta,
                             32 * kMergeRowsPerCta, 0, stream, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace idx

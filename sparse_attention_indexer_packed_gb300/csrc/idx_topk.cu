// Block top-k select: one CTA per packed output row.
//
// What it computes (sglang #42614 "[AMD] MiniMax-M3 indexer CP: packed scoring
// for EAGLE verify rows", Modifications 1 and Accuracy Tests; sglang #45451,
// Accuracy Tests): the row always keeps its first init_blocks and last
// local_blocks blocks, counted from its own length, and fills the rest of topk
// with the best remaining blocks by block max; selection is exact.  Ties go to
// the lower block id.  Output: forced blocks ascending, chosen blocks by
// descending score, then (-1, -inf) pads.
//
// How: the non-forced candidates form one contiguous id range.  Their scores are
// mapped to order-preserving 32-bit keys in shared memory; a most-significant-
// digit radix select (8-bit digits, starting below the bits all candidates
// share) finds the k-th largest key with one shared-memory histogram per digit;
// the chosen ids are gathered and sorted by (key desc, id asc) with a bitonic
// network.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "idx_internal.cuh"

namespace idx {

namespace {

constexpr int kTopkThreads = 256;
constexpr uint32_t kErrLenClamped = 4u;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t block_reduce_u32(uint32_t v, bool is_max, uint32_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t y = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? max(v, y) : min(v, y);
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
  for (int w = 1; w < kTopkThreads / 32; ++w) v = is_max ? max(v, red[w]) : min(v, red[w]);
  return v;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkArgs a) {
  extern __shared__ uint32_t keys[];  // [nb_cap] candidate keys
  __shared__ uint32_t hist[256];
  __shared__ uint32_t red[kTopkThreads / 32];
  __shared__ unsigned long long sel[kMaxTopk];
  __shared__ int sel_count;
  __shared__ uint32_t s_digit, s_need, s_taken_all;

  const int row = blockIdx.x;
  const int r = row / a.M;
  const int i = row - r * a.M;
  const int tid = threadIdx.x;
  int32_t* out_ids = a.out_ids + (size_t)row * a.topk;
  float* out_sc = a.out_scores + (size_t)row * a.topk;
  const float* bm = a.blockmax + (size_t)row * a.nb_cap;

  const int slot = __ldg(a.slot_ids + r);
  int L = 0;
  if (slot >= 0 && slot < a.n_slots) {
    L = __ldg(a.row_lens + r * a.P + i / a.G);
    if (L > a.max_pages * kPage) {
      L = a.max_pages * kPage;
      if (tid == 0) atomicOr(a.err, kErrLenClamped);
    }
  }
  const int nb = L > 0 ? (L + kBlock - 1) / kBlock : 0;
  const int fi = min(a.init_blocks, nb);               // forced init: [0, fi)
  const int ls = max(fi, nb - a.local_blocks);          // forced local: [ls, nb)
  const int nf = fi + (nb - ls);
  const int ncand = ls - fi;                            // candidates: [fi, ls)
  const int c = min(a.topk, nb) - nf;                   // candidates to choose

  // forced blocks first, ascending
  for (int t = tid; t < nf; t += kTopkThreads) {
    const int id = t < fi ? t : ls + (t - fi);
    out_ids[t] = id;
    out_sc[t] = bm[id];
  }
  // pads after the selection
  for (int t = nf + max(c, 0) + tid; t < a.topk; t += kTopkThreads) {
    out_ids[t] = -1;
    out_sc[t] = -INFINITY;
  }
  if (c <= 0) return;

  // ---- candidate keys ----------------------------------------------------
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int t = tid; t < ncand; t += kTopkThreads) {
    const uint32_t k = order_key(bm[fi + t]);
    keys[t] = k;
    kmin = min(kmin, k);
    kmax = max(kmax, k);
  }
  if (tid == 0) sel_count = 0;
  kmin = block_reduce_u32(kmin, false, red);
  kmax = block_reduce_u32(kmax, true, red);

  uint32_t fixed_mask = 0, fixed_val = 0;
  bool take_all_prefix = false;
  uint32_t need = (uint32_t)c;
  if (c == ncand) {
    take_all_prefix = true;  // every candidate is chosen
  } else if (kmin == kmax) {
    fixed_mask = 0xffffffffu;  // all equal: ties resolved by id below
    fixed_val = kmax;
  } else {
    const uint32_t diff = kmin ^ kmax;
    int hi = 32 - __clz(diff);  // bits [hi, 32) are common to all candidates
    fixed_mask = hi >= 32 ? 0u : (0xffffffffu << hi);
    fixed_val = kmax & fixed_mask;
    while (hi > 0) {
      const int lo = max(hi - 8, 0);
      const uint32_t dmask = (1u << (hi - lo)) - 1u;
      for (int d = tid; d < 256; d += kTopkThreads) hist[d] = 0;
      __syncthreads();
      for (int t = tid; t < ncand; t += kTopkThreads) {
        const uint32_t k = keys[t];
        if ((k & fixed_mask) == fixed_val) atomicAdd(&hist[(k >> lo) & dmask], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // bins from the top: lane l owns bins [255 - 8l - 7, 255 - 8l]
        uint32_t loc[8];
        uint32_t sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          loc[e] = hist[255 - 8 * tid - e];
          sum += loc[e];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += y;
        }
        const uint32_t excl = incl - sum;
        const bool has = excl < need && need <= incl;
        const unsigned hit = __ballot_sync(0xffffffffu, has);
        if (has) {
          uint32_t above = excl;
          for (int e = 0; e < 8; ++e) {
            if (above + loc[e] >= need) {
              s_digit = 255 - 8 * tid - e;
              s_need = need - above;
              s_taken_all = (loc[e] == need - above) ? 1u : 0u;
              break;
            }
            above += loc[e];
          }
        }
        (void)hit;
      }
      __syncthreads();
      const uint32_t d = s_digit;
      need = s_need;
      fixed_mask |= dmask << lo;
      fixed_val |= d << lo;
      if (s_taken_all) {
        take_all_prefix = true;
        break;
      }
      hi = lo;
    }
  }

  // ---- gather the chosen ids ---------------------------------------------
  // above: (k & mask) > val, or every key matching the prefix when take_all_prefix
  for (int t = tid; t < ncand; t += kTopkThreads) {
    const uint32_t k = keys[t];
    const uint32_t km = k & fixed_mask;
    const bool pick = take_all_prefix ? (km >= fixed_val) : (km > fixed_val);
    if (pick) {
      const int pos = atomicAdd(&sel_count, 1);
      if (pos < kMaxTopk) sel[pos] = ((unsigned long long)k << 32) | (uint32_t)(0x7fffffff - (fi + t));
    }
  }
  __syncthreads();
  if (!take_all_prefix && tid < 32) {
    // ties at the threshold: the `need` lowest ids among keys equal to fixed_val
    uint32_t left = need;
    int base = sel_count;
    for (int t0 = 0; t0 < ncand && left > 0; t0 += 32) {
      const int t = t0 + tid;
      const bool eq = t < ncand && (keys[t] & fixed_mask) == fixed_val;
      const unsigned m = __ballot_sync(0xffffffffu, eq);
      const int rank = __popc(m & ((1u << tid) - 1u));
      if (eq && (uint32_t)rank < left && base + rank < kMaxTopk)
        sel[base + rank] = ((unsigned long long)keys[t] << 32) | (uint32_t)(0x7fffffff - (fi + t));
      const uint32_t took = min((uint32_t)__popc(m), left);
      base += took;
      left -= took;
    }
    if (tid == 0) sel_count = base;
  }
  __syncthreads();

  // ---- sort (key desc, id asc) and write --------------------------------
  int n2 = 1;
  while (n2 < c) n2 <<= 1;
  for (int t = c + tid; t < n2; t += kTopkThreads) sel[t] = 0ull;
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = tid; t < n2; t += kTopkThreads) {
        const int p = t ^ j;
        if (p > t) {
          const unsigned long long x = sel[t], y = sel[p];
          const bool desc = (t & k) == 0;
          if (desc ? (x < y) : (x > y)) {
            sel[t] = y;
            sel[p] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int t = tid; t < c; t += kTopkThreads) {
    const int id = 0x7fffffff - (int)(uint32_t)(sel[t] & 0xffffffffull);
    out_ids[nf + t] = id;
    out_sc[nf + t] = bm[id];
  }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  const int rows = a.R * a.M;
  if (rows == 0) return cudaSuccess;
  const size_t smem = (size_t)a.nb_cap * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  topk_kernel<<<rows, kTopkThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace idx

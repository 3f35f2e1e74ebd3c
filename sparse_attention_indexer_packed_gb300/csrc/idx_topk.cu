// Block top-k select: one warp per packed output row.
//
// What it computes (sglang #42614 "[AMD] MiniMax-M3 indexer CP: packed scoring
// for EAGLE verify rows", Modifications 1 and Accuracy Tests; sglang #45451,
// Accuracy Tests): the row always keeps its first init_blocks and last
// local_blocks blocks, counted from its own length, and fills the rest of topk
// with the best remaining blocks by block max; selection is exact.  Ties go to
// the lower block id.  Output: forced blocks ascending, chosen blocks by
// descending score, then (-1, -inf) pads.
//
// How: the non-forced candidates form one contiguous id range.  A warp copies
// their scores into its own shared-memory slice as order-preserving 32-bit keys,
// finds the k-th largest key with a most-significant-digit radix select (8-bit
// digits starting below the bits every candidate shares, one warp-private
// 256-bin histogram per digit), gathers the chosen ids with ballots, resolves
// ties at the threshold to the lowest ids, and sorts the chosen (key desc, id
// asc) with a bitonic network.  No block-wide barrier is involved; a CTA holds
// up to eight rows.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "idx_internal.cuh"

namespace idx {

namespace {

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct WarpSmem {
  uint32_t hist[256];
  unsigned long long sel[kMaxTopk];
};

__global__ void topk_kernel(const TopkArgs a, int warps_per_cta) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * warps_per_cta + warp;
  if (row >= a.R * a.M) return;
  WarpSmem& ws = reinterpret_cast<WarpSmem*>(smem)[warp];
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + (size_t)warps_per_cta * sizeof(WarpSmem)) +
                   (size_t)warp * a.nb_cap;

  const int r = row / a.M;
  const int i = row - r * a.M;
  int32_t* out_ids = a.out_ids + (size_t)row * a.topk;
  float* out_sc = a.out_scores + (size_t)row * a.topk;
  const float* bm = a.blockmax + (size_t)row * a.nb_cap;

  const int slot = __ldg(a.slot_ids + r);
  int L = 0;
  if (slot >= 0 && slot < a.n_slots) L = min(__ldg(a.row_lens + r * a.P + i / a.G), a.max_pages * kPage);
  // launched as a programmatic dependent of the score kernel: wait for its
  // completion before touching the block maxima
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int nb = L > 0 ? (L + kBlock - 1) / kBlock : 0;
  const int fi = min(a.init_blocks, nb);       // forced init: [0, fi)
  const int ls = max(fi, nb - a.local_blocks);  // forced local: [ls, nb)
  const int nf = fi + (nb - ls);
  const int ncand = ls - fi;                    // candidates: [fi, ls)
  const int c = min(a.topk, nb) - nf;           // candidates to choose

  for (int t = lane; t < nf; t += 32) {
    const int id = t < fi ? t : ls + (t - fi);
    out_ids[t] = id;
    out_sc[t] = bm[id];
  }
  for (int t = nf + max(c, 0) + lane; t < a.topk; t += 32) {
    out_ids[t] = -1;
    out_sc[t] = -INFINITY;
  }
  if (c <= 0) return;

  // ---- candidate keys ----------------------------------------------------
  // 16 loads in flight per lane: the block maxima sit in L2, so the copy costs
  // a couple of round trips rather than one per 32 candidates
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  constexpr int kBatch = 16;
  for (int t0 = 0; t0 < ncand; t0 += 32 * kBatch) {
    float v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int t = t0 + u * 32 + lane;
      v[u] = t < ncand ? bm[fi + t] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int t = t0 + u * 32 + lane;
      if (t < ncand) {
        const uint32_t k = order_key(v[u]);
        keys[t] = k;
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  __syncwarp();

  uint32_t fixed_mask = 0, fixed_val = 0;
  bool take_all_prefix = false;
  uint32_t need = (uint32_t)c;
  if (c == ncand) {
    take_all_prefix = true;  // every candidate is chosen
  } else if (kmin == kmax) {
    fixed_mask = 0xffffffffu;  // all equal: ties resolved by id below
    fixed_val = kmax;
  } else {
    int hi = 32 - __clz(kmin ^ kmax);  // bits [hi, 32) are common to all candidates
    fixed_mask = hi >= 32 ? 0u : (0xffffffffu << hi);
    fixed_val = kmax & fixed_mask;
    while (hi > 0) {
      const int lo = max(hi - 8, 0);
      const uint32_t dmask = (1u << (hi - lo)) - 1u;
#pragma unroll
      for (int e = 0; e < 8; ++e) ws.hist[lane * 8 + e] = 0u;
      __syncwarp();
      for (int t = lane; t < ncand; t += 32) {
        const uint32_t k = keys[t];
        if ((k & fixed_mask) == fixed_val) atomicAdd(&ws.hist[(k >> lo) & dmask], 1u);
      }
      __syncwarp();
      // bins from the top: lane l owns bins 255 - 8l - e, e = 0..7
      uint32_t loc[8];
      uint32_t sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        loc[e] = ws.hist[255 - 8 * lane - e];
        sum += loc[e];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - sum;
      const bool has = excl < need && need <= incl;
      uint32_t digit = 0, rem = 0, all = 0;
      if (has) {
        uint32_t above = excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (!digit && above + loc[e] >= need) {
            digit = (uint32_t)(255 - 8 * lane - e) | 0x100u;  // bit 8 marks "found"
            rem = need - above;
            all = (loc[e] == need - above) ? 1u : 0u;
          }
          above += loc[e];
        }
      }
      const int src = __ffs(__ballot_sync(0xffffffffu, has)) - 1;
      digit = __shfl_sync(0xffffffffu, digit, src) & 0xffu;
      need = __shfl_sync(0xffffffffu, rem, src);
      all = __shfl_sync(0xffffffffu, all, src);
      fixed_mask |= dmask << lo;
      fixed_val |= digit << lo;
      __syncwarp();
      if (all) {
        take_all_prefix = true;
        break;
      }
      hi = lo;
    }
  }

  // ---- gather the chosen ids ---------------------------------------------
  // above the threshold: (k & mask) > val; with take_all_prefix also == val
  int count = 0;
  for (int t0 = 0; t0 < ncand; t0 += 32) {
    const int t = t0 + lane;
    bool pick = false;
    uint32_t k = 0;
    if (t < ncand) {
      k = keys[t];
      const uint32_t km = k & fixed_mask;
      pick = take_all_prefix ? (km >= fixed_val) : (km > fixed_val);
    }
    const unsigned m = __ballot_sync(0xffffffffu, pick);
    const int pos = count + __popc(m & ((1u << lane) - 1u));
    if (pick && pos < kMaxTopk)
      ws.sel[pos] = ((unsigned long long)k << 32) | (uint32_t)(0x7fffffff - (fi + t));
    count += __popc(m);
  }
  if (!take_all_prefix) {
    // ties at the threshold: the `need` lowest ids among keys equal to it
    uint32_t left = need;
    for (int t0 = 0; t0 < ncand && left > 0; t0 += 32) {
      const int t = t0 + lane;
      const bool eq = t < ncand && (keys[t] & fixed_mask) == fixed_val;
      const unsigned m = __ballot_sync(0xffffffffu, eq);
      const int rank = __popc(m & ((1u << lane) - 1u));
      if (eq && (uint32_t)rank < left && count + rank < kMaxTopk)
        ws.sel[count + rank] =
            ((unsigned long long)keys[t] << 32) | (uint32_t)(0x7fffffff - (fi + t));
      const uint32_t took = min((uint32_t)__popc(m), left);
      count += (int)took;
      left -= took;
    }
  }

  // ---- sort (key desc, id asc) and write --------------------------------
  int n2 = 1;
  while (n2 < c) n2 <<= 1;
  for (int t = c + lane; t < n2; t += 32) ws.sel[t] = 0ull;
  __syncwarp();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = lane; t < n2; t += 32) {
        const int p = t ^ j;
        if (p > t) {
          const unsigned long long x = ws.sel[t], y = ws.sel[p];
          const bool desc = (t & k) == 0;
          if (desc ? (x < y) : (x > y)) {
            ws.sel[t] = y;
            ws.sel[p] = x;
          }
        }
      }
      __syncwarp();
    }
  }
  for (int t = lane; t < c; t += 32) {
    const int id = 0x7fffffff - (int)(uint32_t)(ws.sel[t] & 0xffffffffull);
    out_ids[nf + t] = id;
    out_sc[nf + t] = bm[id];
  }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  const int rows = a.R * a.M;
  if (rows == 0) return cudaSuccess;
  // as many rows per CTA (one warp each) as fit in ~96 KB of shared memory
  const size_t per_warp = sizeof(WarpSmem) + (size_t)a.nb_cap * sizeof(uint32_t);
  int wpc = (int)((96 * 1024) / per_warp);
  wpc = wpc < 1 ? 1 : (wpc > 8 ? 8 : wpc);
  const size_t smem = per_warp * wpc;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = (rows + wpc - 1) / wpc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)(32 * wpc));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, topk_kernel, a, wpc);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace idx

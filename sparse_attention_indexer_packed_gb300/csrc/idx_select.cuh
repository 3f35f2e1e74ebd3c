// Block top-k selection of one packed row by a whole CTA: shared by the top-k
// kernel (one CTA per row) and the score kernel's in-kernel selection.
//
// What it computes (sglang #42614 "[AMD] MiniMax-M3 indexer CP: packed scoring
// for EAGLE verify rows", Modifications 1 and Accuracy Tests; sglang #45451,
// Accuracy Tests): the row always keeps its first init_blocks and last
// local_blocks blocks, counted from its own length, and fills the rest of topk
// with the best remaining blocks by block score; selection is exact, ties go to
// the lower block id.  Output: forced blocks ascending, chosen blocks by
// descending score, then (-1, -inf) pads.
//
// How: the non-forced candidates form one contiguous id range.  Their scores
// are read from L2 with as many loads in flight per thread as the row needs and
// kept in shared memory as order-preserving 32-bit keys.  When there are many
// candidates, most-significant-digit radix passes (8-bit digits starting below
// the bits every candidate shares, one shared 256-bin histogram per digit)
// narrow them to the keys at or above the threshold's bin, usually after one
// pass.  Each remaining (key, id) entry is then placed by its rank among them,
// ties going to the lower id; entries ranked c or later are dropped.  The score
// written out is recovered from the key, so nothing is read back from memory.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "idx_internal.cuh"

namespace idx {
namespace sel {

constexpr int kBatch = 16;  // independent loads in flight per thread (long rows)
// The exact step ranks at most kCap entries (kCap >= the largest topk).
constexpr int kCap = 1024;
static_assert(kCap >= kMaxTopk, "the exact step must hold a whole selection");

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// composite sort key: larger score first, then lower id first
__device__ __forceinline__ unsigned long long pack(uint32_t key, int id) {
  return ((unsigned long long)key << 32) | (uint32_t)(0x7fffffff - id);
}

// What a row selects: forced blocks [0, fi) and [ls, nb) and c more from the
// candidates [fi, ls), all counted from the row's own global block count nb.
// A context shard holds global blocks [s0, s1); it emits the forced blocks it
// holds (nf of them, ascending: the part of [0, fi) it holds, then of
// [ls, nb)), then its best min(c, its candidates) candidates from [cb,
// cb + ncand).  The whole context is the shard [0, nb).
struct RowPlan {
  int nb, fi, ls, s0, s1, nf, cb, ncand, c;
  __device__ int forced_id(int t) const {  // t < nf
    const int n0 = max(0, min(fi, s1) - s0);
    return t < n0 ? s0 + t : max(ls, s0) + (t - n0);
  }
};

__device__ __forceinline__ RowPlan row_plan(const TopkArgs& a, int r, int i) {
  RowPlan p;
  const int slot = __ldg(a.slot_ids + r);
  int L = 0;
  if (slot >= 0 && slot < a.n_slots) {
    L = __ldg(a.row_lens + r * a.P + i / a.G);
    if (!a.shard) L = min(L, a.max_pages * kPage);  // a whole-context table caps the row
  }
  p.nb = L > 0 ? (L + kBlock - 1) / kBlock : 0;
  p.fi = min(a.init_blocks, p.nb);
  p.ls = max(p.fi, p.nb - a.local_blocks);
  const int nf_all = p.fi + (p.nb - p.ls);
  const int c_all = min(a.topk, p.nb) - nf_all;
  p.s0 = a.shard ? a.block_off : 0;
  p.s1 = a.shard ? min(p.nb, a.block_off + a.nb_cap) : p.nb;
  p.nf = max(0, min(p.fi, p.s1) - p.s0) + max(0, p.s1 - max(p.ls, p.s0));
  p.cb = max(p.fi, p.s0);
  p.ncand = max(0, min(p.ls, p.s1) - p.cb);
  p.c = min(c_all, p.ncand);
  return p;
}

// Keys of candidates [0, ncand) (block maxima bm[0..)) into keys[], with B
// loads in flight per thread of NT (through L2 only with kCg); returns this
// thread's smallest and largest key.
template <int B, int NT, bool kCg>
__device__ __forceinline__ void load_keys(const float* bm, int ncand, uint32_t* keys, int tid,
                                          uint32_t& kmin, uint32_t& kmax) {
  for (int t0 = 0; t0 < ncand; t0 += NT * B) {
    float v[B];
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int t = t0 + u * NT + tid;
      v[u] = t < ncand ? (kCg ? __ldcg(bm + t) : bm[t]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int t = t0 + u * NT + tid;
      if (t < ncand) {
        const uint32_t k = order_key(v[u]);
        keys[t] = k;
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
    }
  }
}


// Shared memory of a CTA selecting one row (NW warps), followed by the row's
// keys (nb_cap 32-bit words).
template <int NW>
struct Shared {
  uint32_t hist[256];
  unsigned long long sel[kCap];
  uint32_t red_min[NW], red_max[NW];
  int count;
  uint32_t digit, need, bin;
};

template <int NT>
__host__ __device__ constexpr size_t smem_bytes(int nb_cap) {
  return sizeof(Shared<NT / 32>) + (size_t)nb_cap * sizeof(uint32_t);
}

// The row's pads: needs no block scores, so it may run before the dependency
// wait.
template <int NT>
__device__ __forceinline__ void row_pads(const TopkArgs& a, int row, const RowPlan& pl, int tid) {
  int32_t* out_ids = a.out_ids + (size_t)row * a.topk;
  float* out_sc = a.out_scores + (size_t)row * a.topk;
  for (int t = pl.nf + max(pl.c, 0) + tid; t < a.topk; t += NT) {
    out_ids[t] = -1;
    out_sc[t] = -INFINITY;
  }
}

// The row's forced and chosen blocks, once its block scores are complete and
// visible.  Every thread of the CTA calls it (it holds block barriers); smem is
// the 16-byte aligned Shared<NT / 32> plus the keys.  kCg: read the block
// scores through L2 only.
template <int NT, bool kCg>
__device__ void row_select(const TopkArgs& a, int row, const RowPlan& pl, uint8_t* smem_raw,
                           int tid) {
  Shared<NT / 32>& sh = *reinterpret_cast<Shared<NT / 32>*>(smem_raw);
  unsigned long long* sel = sh.sel;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + sizeof(Shared<NT / 32>));
  const int lane = tid & 31, warp = tid >> 5;
  int32_t* out_ids = a.out_ids + (size_t)row * a.topk;
  float* out_sc = a.out_scores + (size_t)row * a.topk;
  const float* bm = a.blockmax + (size_t)row * a.nb_cap;
  const int nf = pl.nf, ncand = pl.ncand, c = pl.c;
  const int fi = pl.cb;  // global id of the first candidate
  // the workspace holds this row's blocks from s0 on: block g at g - s0
  const float* bmg = bm - pl.s0;
  for (int t = tid; t < nf; t += NT) {
    const int id = pl.forced_id(t);
    out_ids[t] = id;
    out_sc[t] = kCg ? __ldcg(bmg + id) : bmg[id];
  }
  if (c <= 0) return;

  // ---- candidate keys ----------------------------------------------------
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  // as many loads in flight as the row needs, up to kBatch (predicated-off
  // loads still cost issue slots; the 8-load tier took 1.2 us off the NVFP4
  // 64 x 150K step, whose rows hold ~1170 candidates)
  if (ncand <= NT) load_keys<1, NT, kCg>(bmg + fi, ncand, keys, tid, kmin, kmax);
  else if (ncand <= 4 * NT) load_keys<4, NT, kCg>(bmg + fi, ncand, keys, tid, kmin, kmax);
  else if (ncand <= 8 * NT) load_keys<8, NT, kCg>(bmg + fi, ncand, keys, tid, kmin, kmax);
  else load_keys<kBatch, NT, kCg>(bmg + fi, ncand, keys, tid, kmin, kmax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    sh.red_min[warp] = kmin;
    sh.red_max[warp] = kmax;
  }
  // the first radix pass's histogram and the gather's counter start at zero
  for (int h = tid; h < 256; h += NT) sh.hist[h] = 0u;
  if (tid == 0) sh.count = 0;
  __syncthreads();
  kmin = sh.red_min[0];
  kmax = sh.red_max[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) {
    kmin = min(kmin, sh.red_min[w]);
    kmax = max(kmax, sh.red_max[w]);
  }

  // ---- narrow the candidates: radix passes on the threshold bin ----------
  // After each pass the keys above the threshold bin are certainly chosen and
  // the bin holds the rest; stop once "above + bin" is small enough to rank.
  uint32_t fixed_mask = 0, fixed_val = 0, need = (uint32_t)c;
  uint32_t ksize = (uint32_t)ncand;  // keys whose prefix is >= fixed_val
  const uint32_t stop = max(2u * (uint32_t)c, (uint32_t)c + 64u);  // <= 512
  if (ksize > stop && kmin != kmax) {
    int hi = 32 - __clz(kmin ^ kmax);  // bits [hi, 32) are common to all candidates
    fixed_mask = hi >= 32 ? 0u : (0xffffffffu << hi);
    fixed_val = kmax & fixed_mask;
    bool first = true;
    while (hi > 0 && ksize > stop) {
      const int lo = max(hi - 8, 0);
      const uint32_t dmask = (1u << (hi - lo)) - 1u;
      if (!first) {  // the previous pass's scan has read its histogram
        for (int h = tid; h < 256; h += NT) sh.hist[h] = 0u;
        __syncthreads();
      }
      first = false;
      for (int t = tid; t < ncand; t += NT) {
        const uint32_t k = keys[t];
        if ((k & fixed_mask) == fixed_val) atomicAdd(&sh.hist[(k >> lo) & dmask], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // bins from the top: lane l owns bins 255 - 8l - e, e = 0..7
        uint32_t loc[8];
        uint32_t sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          loc[e] = sh.hist[255 - 8 * lane - e];
          sum += loc[e];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - sum;
        if (excl < need && need <= incl) {
          uint32_t above = excl;
          for (int e = 0; e < 8; ++e) {
            if (above + loc[e] >= need) {
              sh.digit = (uint32_t)(255 - 8 * lane - e);
              sh.need = need - above;
              sh.bin = loc[e];
              break;
            }
            above += loc[e];
          }
        }
      }
      __syncthreads();
      ksize = (uint32_t)c - sh.need + sh.bin;  // above the bin + in the bin
      need = sh.need;
      fixed_mask |= dmask << lo;
      fixed_val |= sh.digit << lo;
      hi = lo;
    }
  }

  // ---- gather the final candidate set -------------------------------------
  // small enough: every key with prefix >= fixed_val; otherwise (many keys equal
  // to the exact threshold) the keys above it plus the `need` lowest ids equal
  // to it.  Either way each entry is then placed by its rank.
  const bool small = ksize <= (uint32_t)kCap;
  // each warp appends its entries at a shared counter (one atomic per warp and
  // round); their order is irrelevant, the ranks place them
  for (int t0 = 0; t0 < ncand; t0 += NT) {
    const int t = t0 + tid;
    uint32_t k = 0;
    bool take = false;
    if (t < ncand) {
      k = keys[t];
      const uint32_t km = k & fixed_mask;
      take = small ? (km >= fixed_val) : (km > fixed_val);
    }
    const unsigned m = __ballot_sync(0xffffffffu, take);
    if (m) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&sh.count, __popc(m));
      base = __shfl_sync(0xffffffffu, base, 0);
      const int at = base + __popc(m & ((1u << lane) - 1u));
      if (take && at < kCap) sel[at] = pack(k, fi + t);
    }
  }
  __syncthreads();
  if (!small && warp == 0) {
    // ties at the threshold: the `need` lowest ids among keys equal to it
    uint32_t left = need;
    int b = sh.count;
    for (int t0 = 0; t0 < ncand && left > 0; t0 += 32) {
      const int t = t0 + lane;
      const bool eq = t < ncand && (keys[t] & fixed_mask) == fixed_val;
      const unsigned m = __ballot_sync(0xffffffffu, eq);
      const int rk = __popc(m & ((1u << lane) - 1u));
      if (eq && (uint32_t)rk < left && b + rk < kCap) sel[b + rk] = pack(keys[t], fi + t);
      const uint32_t took = min((uint32_t)__popc(m), left);
      b += (int)took;
      left -= took;
    }
    if (lane == 0) sh.count = b;
  }
  if (!small) __syncthreads();

  // ---- place each entry by its rank (key desc, id asc); keep ranks < c ----
  const int n = min(sh.count, kCap);
  for (int e = tid; e < n; e += NT) {
    const unsigned long long x = sel[e];
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < n; ++j) rank += sel[j] > x ? 1 : 0;
    if (rank < c) {
      out_ids[nf + rank] = 0x7fffffff - (int)(uint32_t)(x & 0xffffffffull);
      out_sc[nf + rank] = key_value((uint32_t)(x >> 32));
    }
  }
}

}  // namespace sel
}  // namespace idx

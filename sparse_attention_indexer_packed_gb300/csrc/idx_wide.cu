// Block scores of wide requests -- more than 16 packed rows, e.g. many EAGLE
// draft rows x heads, or a prefill chunk whose query tokens each end at their own
// position -- on the 5th-generation tensor cores.
//
// The rows of a request are cut into tiles of up to 128 (tile tau holds rows
// [128 tau, 128 tau + 128)), and tiles 2p and 2p + 1 form one "group" that
// streams the request's keys once for both.  A 128-row x 128-token x 128-dim
// product is one tcgen05.mma chain (M = 128, N = 128) accumulating in fp32 in
// tensor memory, so the pages' per-request dot tile (sglang #45451,
// Modifications: the draft rows of a request share one dot tile against its
// index K) covers 128 rows at a time instead of 16.  Each row keeps its own
// length mask and its block max (or log-sum-exp), exactly as the 16-row path
// does; the oracle's per-row definition is the same for both.
//
// Roles inside a CTA (one CTA per SM, persistent over a contiguous range of
// blocks of the flattened (group, block) list):
//   warp 0      TMA producer: the group's query tiles (bf16, e4m3, or for
//               NVFP4 keys the f16 rows q16_kernel made) and each block's two
//               key pages (+ their scales) into a ring of stages;
//   warp 1      allocates 512 TMEM columns (one 128-column fp32 accumulator
//               per tile of a pair, two blocks in flight); as a whole warp it
//               waits for the operands and one elected lane issues both tiles'
//               MMAs of a block against the same staged keys and commits them
//               to mbarriers;
//   warps 2..9  epilogue, group g (four warps) owning tile g of the pair:
//               thread = tile row; tcgen05.ld of its 128 scores, the row's mask
//               and block score, one workspace write per row;
//   warps 10..13 (NVFP4 keys) decode a block's e2m1 codes x E4M3 group scales
//               into an f16 operand tile (ROCm/ATOM #2745: the products are
//               exact); the query rows are scaled by a power of two per row
//               into f16 range by q16_kernel, undone on the result.
// Every wait is bounded; a timeout sets IDX_DEVERR_TIMEOUT and the CTA winds down
// (copies in flight are waited for, TMEM is freed).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "idx_internal.cuh"
#include "idx_ptx.cuh"
#include "idx_tc.cuh"

namespace idx {
namespace {

constexpr int kWRows = 128;     // tile rows (MMA M)
constexpr int kPair = 2;         // tiles of one request that share a key block
constexpr int kUnits = 2;        // blocks in flight in tensor memory
constexpr int kTmemCols = 128 * kPair * kUnits;  // one 128-column fp32 accumulator per tile
constexpr unsigned int kErrBadPage = 1u;  // IDX_DEVERR_BAD_PAGE
constexpr unsigned int kErrTimeout = 2u;  // IDX_DEVERR_TIMEOUT
constexpr unsigned int kErrLenClamped = 4u;  // IDX_DEVERR_LEN_CLAMPED

template <int KF>
struct WCfg;
template <>
struct WCfg<kBf16> {
  static constexpr int kQBytes = 32768;     // one tile: 128 rows x 256 B, two 16 KB K-halves
  static constexpr int kStageBytes = 32768; // 128 tokens x 256 B: two 16 KB K-halves
  static constexpr int kPagePayload = 16384;
  static constexpr int kPageScale = 0;
  static constexpr int kStages = 4;
  static constexpr int kDecStages = 0;
  static constexpr int kDecWarps = 0;
  static constexpr uint32_t kIdesc = instr_desc(1u, 128, 128);  // bf16 x bf16
};
template <>
struct WCfg<kFp8> {
  static constexpr int kQBytes = 16384;     // one tile: 128 rows x 128 B
  static constexpr int kStageBytes = 16384; // 128 tokens x 128 B
  static constexpr int kPagePayload = 8192;
  static constexpr int kPageScale = 256;    // 64 fp32
  static constexpr int kStages = 10;
  static constexpr int kDecStages = 0;
  static constexpr int kDecWarps = 0;
  static constexpr uint32_t kIdesc = instr_desc(0u, 128, 128);  // e4m3 x e4m3
};
template <>
struct WCfg<kNvfp4> {
  static constexpr int kQBytes = 32768;     // one f16 query tile
  static constexpr int kStageBytes = 8192;  // raw codes of 128 tokens (64 B each)
  static constexpr int kPagePayload = 4096;
  static constexpr int kPageScale = 512;    // 64 x 8 E4M3 bytes
  static constexpr int kStages = 4;
  static constexpr int kDecStages = 3;      // decoded f16 tiles, 32 KB each
  static constexpr int kDecWarps = 4;
  static constexpr uint32_t kIdesc = instr_desc(0u, 128, 128);  // f16 x f16
};

template <int KF>
struct WLayout {
  using C = WCfg<KF>;
  static constexpr int S = C::kStages;
  static constexpr int SD = C::kDecStages;
  static constexpr int kQOff = 0;  // kPair query tiles
  static constexpr int kStageOff = kQOff + kPair * C::kQBytes;
  static constexpr int kDecOff = kStageOff + S * C::kStageBytes;
  static constexpr int kScaleOff = kDecOff + SD * 32768;
  static constexpr int kBarOff = kScaleOff + S * 2 * C::kPageScale;
  // full[S] empty[S] dfull[SD] dempty[SD] afull[kUnits] aempty[kUnits] qfull[2]
  // qempty[2] done
  static constexpr int kNumBars = 2 * S + 2 * SD + 2 * kUnits + 5;
  static constexpr int kCtlOff = (kBarOff + kNumBars * 8 + 15) / 16 * 16;
  static constexpr int kGroupOff = kCtlOff + 64;
  static constexpr int kBytes = kGroupOff + (2 * kMaxGroups + 1) * 4;
  static constexpr int kSmemBytes = kBytes + 1024;
  // producer, MMA issuer, two epilogue groups of four warps, decoders
  static constexpr int kEpiWarps = 8;
  static constexpr int kDecWarp0 = 2 + kEpiWarps;
  static constexpr int kWarps = kDecWarp0 + C::kDecWarps;
  static constexpr int kThreads = 32 * kWarps;
  static_assert(kStageOff % 1024 == 0 && kDecOff % 1024 == 0, "operand tiles 1024-aligned");
  static_assert(C::kStageBytes % 1024 == 0, "stages 1024-aligned");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

  __device__ static uint32_t full(uint32_t sb, int s) { return sb + kBarOff + 8 * s; }
  __device__ static uint32_t empty(uint32_t sb, int s) { return sb + kBarOff + 8 * (S + s); }
  __device__ static uint32_t dfull(uint32_t sb, int d) { return sb + kBarOff + 8 * (2 * S + d); }
  __device__ static uint32_t dempty(uint32_t sb, int d) {
    return sb + kBarOff + 8 * (2 * S + SD + d);
  }
  __device__ static uint32_t afull(uint32_t sb, int j) {
    return sb + kBarOff + 8 * (2 * S + 2 * SD + j);
  }
  __device__ static uint32_t aempty(uint32_t sb, int j) {
    return sb + kBarOff + 8 * (2 * S + 2 * SD + kUnits + j);
  }
  // query slot k's barriers (k = 0 only, unless every group is one tile)
  __device__ static uint32_t qfull(uint32_t sb, int k) {
    return sb + kBarOff + 8 * (2 * S + 2 * SD + 2 * kUnits + k);
  }
  __device__ static uint32_t qempty(uint32_t sb, int k) {
    return sb + kBarOff + 8 * (2 * S + 2 * SD + 2 * kUnits + 2 + k);
  }
  __device__ static uint32_t done(uint32_t sb) {
    return sb + kBarOff + 8 * (2 * S + 2 * SD + 2 * kUnits + 4);
  }
};

// Scores are finite, so the max needs no NaN rule of its own: fmaxf is a single
// FMNMX instruction (a compare-and-select pair would cost two).
__device__ __forceinline__ float fmax_finite(float a, float b) { return fmaxf(a, b); }

__device__ __forceinline__ void wlocate(const int* gpre, int V, int u, int& v, int& b) {
  int lo = 0, hi = V - 1;  // largest v with gpre[v] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (gpre[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  v = lo;
  b = u - gpre[lo];
}

// The unit after (v, b) in the flattened list (groups without blocks skipped).
__device__ __forceinline__ void wnext(const int* gpre, int V, int& v, int& b) {
  ++b;
  while (v < V - 1 && b >= gpre[v + 1] - gpre[v]) {
    ++v;
    b = 0;
  }
}

// Page `which` (0, 1) of block b of group v: -1 when the group's last block needs
// only one page, -2 for a page id outside the pool (flagged, not read).
__device__ __forceinline__ int wpage(const ScoreArgs& a, const int* gpre, const int* gslot, int v,
                                     int b, int which, unsigned int* flags) {
  const int word = gslot[v];
  const int slot = word & 0x7fffffff;
  const bool last = b == gpre[v + 1] - gpre[v] - 1;
  if (which == 1 && last && word < 0) return -1;
  const int p = __ldg(a.page_table + (size_t)slot * a.max_pages + 2 * b + which);
  if (p < 0 || p >= a.num_pages) {
    atomicOr(flags, kErrBadPage);
    return -2;
  }
  return p;
}

// Step (1) of the group table: gpre[v] = the longest draft row (clamped to the
// page table) among those with a row in group v, by atomicMax over all threads,
// B rows per thread per round with their loads in flight together.  Returns
// whether this thread saw a live request's row clamped (CTA 0 only).
template <int B>
__device__ __forceinline__ bool group_extents(const ScoreArgs& a, int* gpre, int TP, int RP) {
  bool clamped = false;
  const int cap = a.max_pages * kPage;
  for (int x0 = 0; x0 < RP; x0 += B * (int)blockDim.x) {
    int len[B];
#pragma unroll
    for (int e = 0; e < B; ++e) {
      const int x = x0 + e * (int)blockDim.x + (int)threadIdx.x;
      len[e] = x < RP ? __ldg(a.row_lens + x) : 0;
    }
#pragma unroll
    for (int e = 0; e < B; ++e) {
      const int x = x0 + e * (int)blockDim.x + (int)threadIdx.x;
      const int L = len[e];
      if (L <= 0) continue;
      const int r = x / a.P, j = x - r * a.P;
      const int t0 = (j * a.G) / kWRows, t1 = (j * a.G + a.G - 1) / kWRows;
      for (int t = t0 / 2; t <= t1 / 2; ++t) atomicMax(&gpre[r * TP + t], min(L, cap));
      if (blockIdx.x == 0 && L > cap) {
        const int slot = __ldg(a.slot_ids + r);
        clamped |= slot >= 0 && slot < a.n_slots;
      }
    }
  }
  return clamped;
}

// Per-thread row scores over one block, fed 32 columns at a time.
struct RowMax {
  float m = -INFINITY;
  float post;
  __device__ __forceinline__ explicit RowMax(float post_scale) : post(post_scale) {}
  template <bool kMask>
  __device__ __forceinline__ void add32(const float (&x)[32], int t0, int L) {
    float p = -INFINITY, q = -INFINITY;
    if constexpr (!kMask) {
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        p = fmax3_finite(p, x[k], x[k + 1]);
        q = fmax3_finite(q, x[k + 2], x[k + 3]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        if (t0 + k < L) p = fmax_finite(p, x[k]);
        if (t0 + k + 1 < L) q = fmax_finite(q, x[k + 1]);
      }
    }
    m = fmax3_finite(m, p, q);
  }
  __device__ __forceinline__ float out() const { return m * post; }
};

// ln sum exp over the row's valid tokens of the block, kept as the running max
// m of the raw sums and sum 2^((x - m) c), c = post * log2(e).
struct RowLse {
  float m = -INFINITY, s = 0.f;
  float c;
  __device__ __forceinline__ explicit RowLse(float post_scale)
      : c(post_scale * 1.4426950408889634f) {}
  template <bool kMask>
  __device__ __forceinline__ void add32(const float (&x)[32], int t0, int L) {
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (!kMask || t0 + k < L) mx = fmax_finite(mx, x[k]);
    const float mn = fmax_finite(m, mx);
    const float r = mn == -INFINITY ? 0.f : mn * c;
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
      if (!kMask || t0 + k < L) acc0 += ex2_approx(fmaf(x[k], c, -r));
      if (!kMask || t0 + k + 1 < L) acc1 += ex2_approx(fmaf(x[k + 1], c, -r));
    }
    s = fmaf(s, ex2_approx(fmaf(m, c, -r)), acc0 + acc1);
    m = mn;
  }
  __device__ __forceinline__ float out() const {
    return m == -INFINITY ? m : (m * c + log2f(s)) * 0.6931471805599453f;
  }
};

// Byte address of 16-byte chunk c (0..15) of row i in a 128-row x 256-byte
// operand tile stored as two 128-byte-swizzled K-halves of 16 KB.
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t tile, int i, int c) {
  const int h = c >> 3, cc = c & 7;
  return tile + (uint32_t)(h * 16384 + (i >> 3) * 1024 + (i & 7) * 128 + ((cc ^ (i & 7)) << 4));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// f16 query rows for NVFP4 keys (the MMA takes f16 on both sides, and the
// decoded keys are exact in f16): row i is rescaled by 2^qexp so its largest
// magnitude lies in [2^14, 2^15) and stored as f16, every element within 2^-24
// of that maximum exactly; qpost[i] = 2^-qexp undoes it on the scores.  One
// thread a row, all its loads in flight together; run once per call before the
// score kernel, which loads the f16 tiles by TMA.
__global__ void __launch_bounds__(128) q16_kernel(const ScoreArgs a) {
  // the score kernel may be scheduled at once; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the query rows may be written by the work before this call
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= (long long)a.R * a.M) return;
  const uint4* src = reinterpret_cast<const uint4*>(a.q + row * 256);
  uint4 u[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) u[c] = __ldg(src + c);
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[e] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[e] & 0xffff0000u)));
    }
  }
  int qexp = 0;
  if (amax > 0.f) qexp = 14 - (((__float_as_uint(amax) >> 23) & 0xff) - 127);
  qexp = max(-100, min(100, qexp));
  const float up = ldexpf(1.f, qexp);
  uint4* dst = reinterpret_cast<uint4*>(a.q16 + row * 128);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint32_t w[4] = {u[c].x, u[c].y, u[c].z, u[c].w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __half2 hh = __floats2half2_rn(__uint_as_float(w[e] << 16) * up,
                                     __uint_as_float(w[e] & 0xffff0000u) * up);
      o[e] = *reinterpret_cast<uint32_t*>(&hh);
    }
    dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  a.qpost[row] = ldexpf(1.f, -qexp);
}

// Decode token n (0..127) of a raw NVFP4 stage into the f16 operand tile.
// Raw payload: page pp = n / 64 at pp * 4096, row n % 64 at 64 B with the TMA
// 64-byte swizzle (16-byte chunk m stored at m ^ ((row >> 1) & 3)); scales: page
// pp at pp * 512, 8 bytes per token.
__device__ __forceinline__ void decode_token(uint32_t raw, uint32_t rscale, uint32_t dec, int n) {
  const int pp = n >> 6, nn = n & 63;
  uint32_t s_lo, s_hi;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
               : "=r"(s_lo), "=r"(s_hi)
               : "r"(rscale + (uint32_t)(pp * 512 + nn * 8)));
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    uint32_t w[4];
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(raw + (uint32_t)(pp * 4096 + nn * 64 + (((m ^ ((nn >> 1) & 3)) & 3) << 4))));
    // elements 32m .. 32m+31: groups 2m (words 0, 1) and 2m+1 (words 2, 3)
#pragma unroll
    for (int hg = 0; hg < 2; ++hg) {
      const int grp = 2 * m + hg;
      const uint32_t sb = ((grp < 4 ? s_lo : s_hi) >> (8 * (grp & 3))) & 0xffu;
      uint32_t sc, unused;
      e4m3x4_to_f16x2x2(sb | (sb << 8), sc, unused);  // {scale, scale}
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int e = 2 * hg + e2;
        uint32_t f[4];
        e2m1x8_to_f16x2x4(w[e], f);
        st_shared_v4(sw128_chunk(dec, n, 4 * m + e), hmul2_f16(f[0], sc), hmul2_f16(f[1], sc),
                     hmul2_f16(f[2], sc), hmul2_f16(f[3], sc));
      }
    }
  }
}

template <int KF, class RowScore>
__global__ void __launch_bounds__(WLayout<KF>::kThreads, 1)
    wide_kernel(const ScoreArgs a, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap qmap) {
  using L = WLayout<KF>;
  using C = WCfg<KF>;
  constexpr int S = L::S;
  constexpr int SD = L::SD;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + L::kCtlOff);
  // ctl[0] = units of the call, ctl[1] = TMEM base, ctl[4] = device error flags
  unsigned int* cta_flags = reinterpret_cast<unsigned int*>(smem + L::kCtlOff) + 4;
  int* gpre = reinterpret_cast<int*>(smem + L::kGroupOff);
  int* gslot = gpre + kMaxGroups + 1;
  const uint32_t qtile = sb + L::kQOff;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(L::full(sb, s), 1);
      // who frees a raw stage: the MMA (bf16), the MMA and the eight epilogue
      // warps that read its key scales (fp8), the four decoder warps (NVFP4)
      mbar_init(L::empty(sb, s), KF == kBf16 ? 1 : (KF == kFp8 ? 9 : 4));
    }
    for (int d = 0; d < SD; ++d) {
      mbar_init(L::dfull(sb, d), C::kDecWarps);
      mbar_init(L::dempty(sb, d), 1);
    }
    for (int j = 0; j < kUnits; ++j) {
      mbar_init(L::afull(sb, j), 1);
      mbar_init(L::aempty(sb, j), 8);  // both epilogue groups, every block
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(L::qfull(sb, k), 1);
      mbar_init(L::qempty(sb, k), 1);
    }
    mbar_init(L::done(sb), 1);
    mbar_init(sb + L::kCtlOff + 32, 1);  // the stall test's barrier
    fence_barrier_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&qmap);
  }
  if (warp == 1) {
    tmem_alloc(sb + L::kCtlOff + 4, kTmemCols);
    tmem_relinquish();
  }

  // launched as a programmatic dependent of whatever ran before on the stream:
  // everything above touches only this CTA; from here on inputs are read and
  // the workspace written, so wait for that work to complete
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- group table: block prefix sums and slots of every (request, tile pair)
  // group v = (request v / TP, tiles 2 (v % TP) and 2 (v % TP) + 1): TP pairs
  // per request, the last a single tile when a request has an odd count
  // (1) every thread takes draft rows: a tile's extent is the longest of the
  // draft rows any of its rows belongs to; (2) warp 0 turns extents into block
  // counts and prefix sums.
  const int TP = (a.tiles + 1) / 2;
  const int V = a.R * TP;
  for (int v = threadIdx.x; v < V; v += blockDim.x) gpre[v] = 0;
  if (threadIdx.x == 0) *cta_flags = 0u;
  // the first 32 groups' slots, read while the extents are gathered (one
  // round trip fewer before the first key copy)
  const int slot_pre = (warp == 0 && lane < V) ? __ldg(a.slot_ids + lane / TP) : 0;
  __syncthreads();
  {
    const int RP = a.R * a.P;
    // a prefill chunk has thousands of draft rows: eight loads in flight per
    // thread (one round trip instead of one per row); a verify pack's few
    // rows take one each (the batched loop measured slower there)
    const bool clamped = RP > (int)blockDim.x ? group_extents<8>(a, gpre, TP, RP)
                                              : group_extents<1>(a, gpre, TP, RP);
    if (clamped) atomicOr(cta_flags, kErrLenClamped);
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int v0 = 0; v0 < V; v0 += 32) {
      const int v = v0 + lane;
      int nbk = 0, word = 0;
      if (v < V) {
        const int ext = gpre[v];
        const int slot = v0 == 0 ? slot_pre : __ldg(a.slot_ids + v / TP);
        const bool pad = slot < 0 || slot >= a.n_slots;
        nbk = (pad || ext <= 0) ? 0 : (ext + kBlock - 1) / kBlock;
        const int rem = ext - (nbk - 1) * kBlock;  // tokens in the last block
        word = (nbk > 0 ? slot : 0) | ((nbk > 0 && rem <= kPage) ? (int)0x80000000 : 0);
      }
      int incl = nbk;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      __syncwarp();  // every lane has read its extent before any prefix is written
      if (v < V) {
        gpre[v] = run + incl - nbk;
        gslot[v] = word;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      gpre[V] = run;
      ctl[0] = run;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int U = ctl[0];
  const uint32_t tmem = (uint32_t)ctl[1];
  const int u0 = (int)((long long)U * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)U * (blockIdx.x + 1) / gridDim.x);
  // Query tiles: a group's tiles go to the two slots of shared memory, and
  // the next group's are loaded once the MMAs of this one are done with them.
  // When every group is a single tile (up to 128 rows a request, a verify
  // pack) the groups alternate between the slots instead: the n-th group's
  // tile goes to slot n % 2, so the next group's rows load while the MMAs
  // still read the other slot and a CTA whose range crosses a group boundary
  // does not drain its MMAs there.
  const bool alt = a.tiles == 1;

  if (warp == 0) {
    // ======================= producer =======================
    int prev_v = -1, nq = 0, i = 0;
    bool ok = true;
    int v = 0, b = 0, wpg = -1;
    if (u0 < u1) wlocate(gpre, V, u0, v, b);
    for (int u = u0; u < u1 && ok; ++u, ++i) {
      const int k = (u - u0) & 15;
      if (k == 0) {
        // page ids of the next 16 blocks in one round trip: lane l looks up
        // page l & 1 of block u + l / 2
        const int uu = u + (lane >> 1);
        wpg = -1;
        if (uu < u1) {
          int pv, pb;
          wlocate(gpre, V, uu, pv, pb);
          wpg = wpage(a, gpre, gslot, pv, pb, lane & 1, cta_flags);
        }
      }
      const int p0 = __shfl_sync(0xffffffffu, wpg, 2 * k);
      const int p1 = __shfl_sync(0xffffffffu, wpg, 2 * k + 1);
      if (v != prev_v) {
        if (lane == 0) {
          // the MMAs of the slot's previous group must be done with it
          const int k = alt ? (nq & 1) : 0;
          const int prev = alt ? nq - 2 : nq - 1;  // the slot's previous load
          if (prev >= 0 &&
              !mbar_wait_bounded(L::qempty(sb, k), (alt ? prev >> 1 : prev) & 1, a.wait_ns))
            ok = false;
          if (ok) {
            const int r = v / TP;
            const int tile0 = 2 * (v - r * TP);
            const int nt = min(kPair, a.tiles - tile0);
            const uint32_t qb = L::qfull(sb, k);
            mbar_arrive_expect_tx(qb, nt * C::kQBytes);
            for (int t = 0; t < nt; ++t) {
              const int base_row = r * a.M + (tile0 + t) * kWRows;
              const uint32_t qt = qtile + (k + t) * C::kQBytes;
              if (KF != kFp8) {  // bf16 rows, or the f16 rows made for NVFP4 keys
                tma_load_2d(qt, &qmap, 0, base_row, qb);
                tma_load_2d(qt + 16384, &qmap, 64, base_row, qb);
              } else {
                tma_load_2d(qt, &qmap, 0, base_row, qb);
              }
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        ++nq;
        prev_v = v;
      }
      const int s = i % S;
      if (lane == 0 && i >= S && !mbar_wait_bounded(L::empty(sb, s), ((i / S) - 1) & 1, a.wait_ns)) ok = false;
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if (lane == 0) {
        uint32_t tx = 0;
        if (p0 >= 0) tx += C::kPagePayload + C::kPageScale;
        if (p1 >= 0) tx += C::kPagePayload + C::kPageScale;
        const uint32_t fb = L::full(sb, s);
        mbar_arrive_expect_tx(fb, tx);
        const uint32_t dst = sb + L::kStageOff + s * C::kStageBytes;
        const uint32_t sdst = sb + L::kScaleOff + s * 2 * C::kPageScale;
        const int pgs[2] = {p0, p1};
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          if (pgs[pp] < 0) continue;
          const int y = pgs[pp] * kPage;
          if (KF == kBf16) {
            tma_load_2d(dst + pp * 8192, &kmap, 0, y, fb);
            tma_load_2d(dst + 16384 + pp * 8192, &kmap, 64, y, fb);
          } else {
            tma_load_2d(dst + pp * C::kPagePayload, &kmap, 0, y, fb);
            bulk_load(sdst + pp * C::kPageScale, a.k_scale + (size_t)pgs[pp] * C::kPageScale,
                      C::kPageScale, fb);
          }
        }
      }
      wnext(gpre, V, v, b);
    }
    if (lane == 0) {
      if (!ok) atomicOr(cta_flags, kErrTimeout);
      // every copy this warp issued has landed before the CTA can exit, also
      // when another role gave up early (instant when they were all consumed)
      for (int k = max(0, i - S); k < i; ++k)
        (void)mbar_wait_bounded(L::full(sb, k % S), (k / S) & 1, 200000000ull);
      // (the last load of each slot used)
      for (int n = max(0, nq - (alt ? 2 : 1)); n < nq; ++n)
        (void)mbar_wait_bounded(L::qfull(sb, alt ? (n & 1) : 0), (alt ? n >> 1 : n) & 1,
                                200000000ull);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    // The whole warp runs the loop with warp-uniform values; one elected lane
    // issues each MMA and commit (tc_*_warp).  Every wait is taken by all lanes
    // and its outcome agreed with a vote, so the warp stays converged.
    {
      int prev_v = -1, nq = 0, i = 0, nt = 1, qk = 0;
      uint32_t qbase = qtile;  // the group's query slot
      bool ok = true;
      int v = 0, b = 0;
      if (u0 < u1) wlocate(gpre, V, u0, v, b);
      for (int u = u0; u < u1; ++u, ++i) {
        if (v != prev_v) {
          // stall test: the first wait goes to a barrier nothing completes
          const bool stall = a.stall_test && nq == 0;
          qk = alt ? (nq & 1) : 0;
          qbase = qtile + qk * C::kQBytes;
          if (!__all_sync(0xffffffffu,
                          mbar_wait_bounded(stall ? sb + L::kCtlOff + 32 : L::qfull(sb, qk),
                                            stall ? 0u : (alt ? nq >> 1 : nq) & 1,
                                            a.wait_ns))) {
            ok = false;
            break;
          }
          ++nq;
          prev_v = v;
          nt = min(kPair, a.tiles - 2 * (v % TP));
        }
        const int s = i % S;
        uint32_t opnd;
        if constexpr (KF == kNvfp4) {
          const int d = i % SD;
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(L::dfull(sb, d), (i / SD) & 1, a.wait_ns))) {
            ok = false;
            break;
          }
          opnd = sb + L::kDecOff + d * 32768;
        } else {
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(L::full(sb, s), (i / S) & 1, a.wait_ns))) {
            ok = false;
            break;
          }
          opnd = sb + L::kStageOff + s * C::kStageBytes;
        }
        const int j = i % kUnits;
        if (i >= kUnits &&
            !__all_sync(0xffffffffu,
                        mbar_wait_bounded(L::aempty(sb, j), ((i / kUnits) - 1) & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // both tiles of the pair against the same staged keys
        for (int t = 0; t < nt; ++t) {
          const uint32_t d_tmem = tmem + (uint32_t)((j * kPair + t) * 128);
          const uint32_t qt = qbase + t * C::kQBytes;
          if (KF == kFp8) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma_f8_warp(d_tmem, desc_kmajor_sw128(qt + ks * 32),
                             desc_kmajor_sw128(opnd + ks * 32), C::kIdesc, ks > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off = (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32);
              tc_mma_f16_warp(d_tmem, desc_kmajor_sw128(qt + off), desc_kmajor_sw128(opnd + off),
                              C::kIdesc, ks > 0 ? 1u : 0u);
            }
          }
        }
        if constexpr (KF == kNvfp4) tc_commit_warp(L::dempty(sb, i % SD));
        else tc_commit_warp(L::empty(sb, s));
        tc_commit_warp(L::afull(sb, j));
        int vn = v, bn = b;
        if (u + 1 < u1) wnext(gpre, V, vn, bn);
        else vn = -1;
        if (vn != v) tc_commit_warp(L::qempty(sb, qk));  // last block of this group
        v = vn;
        b = bn;
      }
      if (!ok && lane == 0) atomicOr(cta_flags, kErrTimeout);
      // every MMA issued has completed before TMEM is released
      tc_commit_warp(L::done(sb));
      (void)mbar_wait_bounded(L::done(sb), 0, 200000000ull);
    }
    __syncwarp();
  } else if (warp < L::kDecWarp0) {
    // ======================= epilogue =======================
    // group eg owns tile eg of each pair (accumulator j * kPair + eg of block i,
    // j = i % kUnits); it waits for and frees every block's accumulators, also
    // when its pair has a single tile, so the barrier phases stay in step
    const int eg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int ti = quarter * 32 + lane;  // tile row of this thread
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    int prev_v = -1, nq = 0, i = 0;
    int Lrow = 0, out_row = -1;
    bool mine = false;  // the current pair has a tile eg
    float post = 1.f, qs = 0.f;
    bool ok = true;
    int v = 0, b = 0;
    if (u0 < u1) wlocate(gpre, V, u0, v, b);
    for (int u = u0; u < u1; ++u, ++i, wnext(gpre, V, v, b)) {
      if (v != prev_v) {
        const int r = v / TP;
        const int tile = 2 * (v - r * TP) + eg;
        mine = tile < a.tiles;
        const int row0 = tile * kWRows;
        const int nrows = mine ? min(kWRows, a.M - row0) : 0;
        const bool live = ti < nrows && gpre[v + 1] > gpre[v];
        out_row = live ? r * a.M + row0 + ti : -1;
        Lrow = live ? min(__ldg(a.row_lens + r * a.P + (row0 + ti) / a.G), a.max_pages * kPage) : 0;
        if (KF == kFp8) qs = live ? __ldg(a.q_scale + out_row) : 0.f;
        if (KF == kNvfp4) post = live ? __ldg(a.qpost + out_row) : 1.f;
        ++nq;
        prev_v = v;
      }
      const int j = i % kUnits;
      if (!mbar_wait_bounded(L::afull(sb, j), (i / kUnits) & 1, a.wait_ns)) ok = false;
      // the key scales this warp reads were written by the copy engine: observe
      // their arrival itself (already complete, since the MMA waited for it)
      if (KF == kFp8 && ok && !mbar_wait_bounded(L::full(sb, i % S), (i / S) & 1, a.wait_ns)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const int tbase = b * kBlock;
      RowScore sc(post);
      if (mine) {
        const float* ks = reinterpret_cast<const float*>(smem + L::kScaleOff + (i % S) * 2 * C::kPageScale);
        const uint32_t acc = trow + (uint32_t)((j * kPair + eg) * 128);
        const bool whole = tbase + kBlock <= Lrow;
        // kLd 32-column loads in flight per wait: for bf16 all four of the
        // block's (one TMEM round trip); two for e4m3, whose per-column key
        // scales need the registers (measured slower with four), and for
        // NVFP4, whose decoder warps leave fewer registers per thread
        constexpr int kLd = KF == kBf16 ? 4 : 2;
#pragma unroll 1
        for (int h = 0; h < 4 / kLd; ++h) {
          uint32_t raw[kLd][32];
          __syncwarp();
#pragma unroll
          for (int hh = 0; hh < kLd; ++hh) tc_ld_32cols(acc + (uint32_t)((h * kLd + hh) * 32), raw[hh]);
          tc_wait_ld();
#pragma unroll
          for (int hh = 0; hh < kLd; ++hh) {
            const int c0 = (h * kLd + hh) * 32;
            float x[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(raw[hh][k]);
            if constexpr (KF == kFp8) {
              // (dot * q scale) * key scale, two columns per packed multiply
              const float2 q2 = make_float2(qs, qs);
#pragma unroll
              for (int k = 0; k < 32; k += 2) {
                const float2 kk = *reinterpret_cast<const float2*>(ks + c0 + k);
                const float2 y = fmul2_rn(fmul2_rn(make_float2(x[k], x[k + 1]), q2), kk);
                x[k] = y.x;
                x[k + 1] = y.y;
              }
            }
            if (whole) sc.template add32<false>(x, tbase + c0, Lrow);
            else sc.template add32<true>(x, tbase + c0, Lrow);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(L::aempty(sb, j));
        if (KF == kFp8) mbar_arrive(L::empty(sb, i % S));
      }
      if (out_row >= 0 && tbase < Lrow) a.blockmax[(size_t)out_row * a.nb_cap + b] = sc.out();
    }
    if (!ok && lane == 0) atomicOr(cta_flags, kErrTimeout);
  } else if constexpr (KF == kNvfp4) {
    // ======================= NVFP4 decoders =======================
    const int n = (warp - L::kDecWarp0) * 32 + lane;  // token of the block
    bool ok = true;
    int i = 0;
    for (int u = u0; u < u1; ++u, ++i) {
      const int s = i % S, d = i % SD;
      if (!mbar_wait_bounded(L::full(sb, s), (i / S) & 1, a.wait_ns)) ok = false;
      if (ok && i >= SD && !mbar_wait_bounded(L::dempty(sb, d), ((i / SD) - 1) & 1, a.wait_ns)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      decode_token(sb + L::kStageOff + s * C::kStageBytes, sb + L::kScaleOff + s * 2 * C::kPageScale,
                   sb + L::kDecOff + d * 32768, n);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(L::dfull(sb, d));
        mbar_arrive(L::empty(sb, s));
      }
    }
    if (!ok && lane == 0) atomicOr(cta_flags, kErrTimeout);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) {
    a.err_bytes[blockIdx.x] = (uint8_t)*cta_flags;
    if (blockIdx.x == 0) *a.err_count = gridDim.x;
  }
}

}  // namespace

cudaError_t launch_q16(const ScoreArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.R * a.M;
  if (rows <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(q16_kernel, (int)((rows + 127) / 128), 128, 0, stream, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

namespace {

template <int KF, class RowScore>
cudaError_t launch_wide_kf(const ScoreArgs& a, const CUtensorMap& kmap, const CUtensorMap& qmap,
                           cudaStream_t stream) {
  using L = WLayout<KF>;
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int sms = cached_sm_count(dev);
  if (sms <= 0) return cudaErrorInvalidDevice;
  e = smem_limit_once(wide_kernel<KF, RowScore>, L::kSmemBytes, dev, attr_done);
  if (e != cudaSuccess) return e;
  const int lim = grid_limit();
  int grid = (lim > 0 && lim < sms) ? lim : sms;
  if (grid > kMaxScoreCtas) grid = kMaxScoreCtas;
  e = launch_pdl(wide_kernel<KF, RowScore>, grid, L::kThreads, L::kSmemBytes, stream, a, kmap,
                 qmap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <class RowScore>
cudaError_t launch_wide_bs(int key_format, const ScoreArgs& a, const CUtensorMap& kmap,
                           const CUtensorMap& qmap, cudaStream_t stream) {
  switch (key_format) {
    case kBf16:
      return launch_wide_kf<kBf16, RowScore>(a, kmap, qmap, stream);
    case kFp8:
      return launch_wide_kf<kFp8, RowScore>(a, kmap, qmap, stream);
    case kNvfp4:
      return launch_wide_kf<kNvfp4, RowScore>(a, kmap, qmap, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_wide(int key_format, int block_score, const ScoreArgs& args,
                        const CUtensorMap& payload_map, const CUtensorMap& q_map,
                        cudaStream_t stream) {
  if (block_score == kBlockLse)
    return launch_wide_bs<RowLse>(key_format, args, payload_map, q_map, stream);
  return launch_wide_bs<RowMax>(key_format, args, payload_map, q_map, stream);
}

}  // namespace idx

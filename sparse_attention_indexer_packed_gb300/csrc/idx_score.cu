// Packed index-score kernel: per-row masked q.k and a score per 128-token block
// (the block max, or its log-sum-exp).
//
// What it computes (sglang #45451, Modifications; sglang #42614 "[AMD]
// MiniMax-M3 indexer CP: packed scoring for EAGLE verify rows", Modifications 1):
// the P draft rows x G heads of a request (P*G <= 16) share one 16-row dot tile,
// so each key tile crosses HBM once per request; tile row i is (draft row i / G,
// head i % G); the keys are read up to the group's longest row while each row
// masks tokens at or past its own length; each row emits the score of every
// 128-token block it covers.
//
// How (sm_103a):
//  * persistent grid, one CTA per SM; the flattened (group, block) work list is
//    split into equal contiguous ranges, one per CTA, except a last part that
//    warps take one block at a time from a workspace counter;
//  * every warp of the CTA owns its own shared-memory stages: it resolves the
//    pages of its next blocks through the slot table, issues TMA tensor loads
//    of the 64-token pages (128-byte or 64-byte swizzle) plus 1-D bulk copies
//    of the per-key scales into its stage, each stage completing on an
//    mbarrier; after scoring a block it refills the same stage with its next
//    block, so copies are issued by many warps at once and no stage is ever
//    shared between warps;
//  * scoring a block: ldmatrix from the swizzled stage, mma.sync with the query
//    tile held in registers (bf16 m16n8k16, e4m3 m16n8k32; NVFP4 keys are
//    decoded to exact f16 in registers and use f16 m16n8k16), a mask by each
//    row's length and the block max by shuffles;
//  * every wait is bounded: on timeout the warp records IDX_DEVERR_TIMEOUT and
//    stops after its copies in flight have landed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "idx_internal.cuh"
#include "idx_ptx.cuh"
#if IDX_FUSED_TOPK
#include "idx_select.cuh"
#endif

namespace idx {

namespace {

constexpr uint32_t kErrBadPage = 1u;
constexpr uint32_t kErrTimeout = 2u;
constexpr uint32_t kErrLenClamped = 4u;
// Static blocks per warp whose pages are brought into L2 before the
// programmatic wait, for calls of at most kHintGroups groups.
constexpr int kPrefetchUnits = 2;
constexpr int kHintGroups = 256;

// Warps and stages per key format.  Every warp is a consumer that also issues
// the copies for its own stages (SPW stages per warp, S = NC * SPW in all).
template <int KF>
struct Cfg;

template <>
struct Cfg<kBf16> {
  static constexpr int kRowBytes = 256;
  static constexpr int kPagePayload = kPage * kRowBytes;  // 16 KB: two 8 KB swizzled boxes
  static constexpr int kScaleRow = 0;
  static constexpr int kWarps = 6;
  static constexpr int kStagesPerWarp = 1;
};
template <>
struct Cfg<kFp8> {
  static constexpr int kRowBytes = 128;
  static constexpr int kPagePayload = kPage * kRowBytes;  // 8 KB: one swizzled box
  static constexpr int kScaleRow = 4;
  static constexpr int kWarps = 12;
  static constexpr int kStagesPerWarp = 1;
};
template <>
struct Cfg<kNvfp4> {
  static constexpr int kRowBytes = 64;
  static constexpr int kPagePayload = kPage * kRowBytes;  // 4 KB: one 64B-swizzled box
  static constexpr int kScaleRow = 8;
  static constexpr int kWarps = 20;
  static constexpr int kStagesPerWarp = 1;
};

// Each warp owns D stages (one 128-token block each: two pages) and cycles
// through them strictly in order: its k-th block goes to stage k % D and is
// waited for with phase parity (k / D) & 1.  No other warp touches them, so a
// parity wait can never be satisfied by the phase before the one it means and
// no "stage empty" barrier is needed.  With D > 1 the warp's next blocks are in
// flight while it scores the current one.
template <int KF>
struct Layout {
  static constexpr int NC = Cfg<KF>::kWarps;
  static constexpr int D = Cfg<KF>::kStagesPerWarp;
  static_assert(D == 1 || D == 2, "one or two stages per warp");
  static constexpr int S = NC * D;
  static constexpr int kStagePayload = 2 * Cfg<KF>::kPagePayload;
  static constexpr int kPageScale = kPage * Cfg<KF>::kScaleRow;
  static constexpr int kStageScale = 2 * kPageScale;
  static constexpr int kPayloadOff = 0;
  static constexpr int kScaleOff = kPayloadOff + S * kStagePayload;
  static constexpr int kBarOff = kScaleOff + S * kStageScale;        // full[S]
  static constexpr int kCtlOff = kBarOff + S * 8;                    // control words
  static constexpr int kGroupOff = kCtlOff + 64;                     // group table
  static constexpr int kHintOff = kGroupOff + (2 * kMaxGroups + 1) * 4;  // hint table
  static constexpr int kBytes = kHintOff + (2 * kHintGroups + 4) * 4;
  static constexpr int kSmemBytes = kBytes + 1024;                   // + alignment slack
  static constexpr int kThreads = 32 * NC;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct Group {
  int r, slot, base_row, nrows, extent, nbk;
};

__device__ __forceinline__ int clamp_len(int L, int max_tokens) {
  return L > max_tokens ? max_tokens : L;
}

// Tokens the page table reaches, counted from the start of the context: a
// context shard's table begins at global block block_off.
__device__ __forceinline__ int token_cap(const ScoreArgs& a) {
  return (2 * a.block_off + a.max_pages) * kPage;
}

// A hint to bring the 128-byte line holding p into L2 (no result, nothing waits).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// A load of the call's inputs.  kHint: read before the programmatic wait, when
// the earlier work may still be writing them, so through L2 only (ld.global.cg):
// a line cached in L1 there could be returned stale by a read after the wait.
template <bool kHint = false>
__device__ __forceinline__ int ld_in(const int* p) {
  return kHint ? __ldcg(p) : __ldg(p);
}

// Geometry of scoring group v (a request when packed, a draft row when per-row).
template <bool kHint = false>
__device__ Group group_info(const ScoreArgs& a, int v) {
  Group g;
  int ext = 0;
  if (a.perrow) {
    g.r = v / a.P;
    const int j = v - g.r * a.P;
    g.base_row = g.r * a.M + j * a.G;
    g.nrows = a.G;
    ext = ld_in<kHint>(a.row_lens + v);
  } else {
    g.r = v;
    g.base_row = v * a.M;
    g.nrows = a.M;
    for (int j = 0; j < a.P; ++j) ext = max(ext, ld_in<kHint>(a.row_lens + v * a.P + j));
  }
  g.slot = ld_in<kHint>(a.slot_ids + g.r);
  const bool pad = g.slot < 0 || g.slot >= a.n_slots;
  ext = clamp_len(ext, token_cap(a));
  g.extent = pad ? 0 : max(ext, 0);
  // blocks held here: global blocks [block_off, ceil(extent / 128)), local from 0
  g.nbk = max(0, (g.extent + kBlock - 1) / kBlock - a.block_off);
  return g;
}

// Length of tile row i of group v (clamped; <= 0 means the row is empty).
__device__ __forceinline__ int tile_row_len(const ScoreArgs& a, int v, int r, int i) {
  const int L = a.perrow ? __ldg(a.row_lens + v) : __ldg(a.row_lens + r * a.P + i / a.G);
  return clamp_len(L, token_cap(a));
}

// Scores are finite, so the max needs no NaN rule of its own: fmaxf is a single
// FMNMX instruction (a compare-and-select pair would cost two).
__device__ __forceinline__ float fmax_finite(float a, float b) { return fmaxf(a, b); }

// Per-lane running block scores of the two tile rows a lane holds (row g and
// g + 8).  add() folds the four accumulator values of one 8-token slice: v0, v1
// belong to row g (tokens t0, t0 + 1), v2, v3 to row g + 8; kMask = false is
// for blocks that lie wholly inside every live row's length.  reduce() merges
// the four lanes of a row; out0/out1 give the block score of rows g / g + 8.
//
// Block max (sglang #45451, Modifications / Accuracy Tests: "max").
struct MaxScore {
  static constexpr bool kWholeBlockUnroll = true;
  float m0 = -INFINITY, m1 = -INFINITY;
  float post = 1.f;  // exact power-of-two rescale of the raw dot products
  __device__ __forceinline__ explicit MaxScore(float post_scale) : post(post_scale) {}
  template <bool kMask>
  __device__ __forceinline__ void add(float v0, float v1, float v2, float v3, int t0, int L0,
                                      int L1) {
    if (kMask) {
      if (t0 < L0) m0 = fmax_finite(m0, v0);
      if (t0 + 1 < L0) m0 = fmax_finite(m0, v1);
      if (t0 < L1) m1 = fmax_finite(m1, v2);
      if (t0 + 1 < L1) m1 = fmax_finite(m1, v3);
    } else {
      m0 = fmax3_finite(m0, v0, v1);
      m1 = fmax3_finite(m1, v2, v3);
    }
  }
  __device__ __forceinline__ void reduce() {
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      m0 = fmax_finite(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = fmax_finite(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
  }
  // a positive power of two commutes with the max: applied once, to the result
  __device__ __forceinline__ float out0() const { return m0 * post; }
  __device__ __forceinline__ float out1() const { return m1 * post; }
};

// Block log-sum-exp (sglang #45451, Accuracy Tests: "lse"): ln sum exp(s) over
// the block's valid tokens.  Kept per row as the running maximum m of the raw
// dot products and the sum of 2^((x - m) c), c = post * log2(e), so every term
// costs one fused multiply-add and one ex2; each call folds a lane's two values
// of a row in with one rescale and no branch (a masked value enters as -inf and
// adds 2^-inf = 0).  lse = (m c + log2 sum) ln 2.
struct LseScore {
  static constexpr bool kWholeBlockUnroll = false;
  float m0 = -INFINITY, s0 = 0.f, m1 = -INFINITY, s1 = 0.f;
  float c;
  __device__ __forceinline__ explicit LseScore(float post_scale)
      : c(post_scale * 1.4426950408889634f) {}
  __device__ __forceinline__ void push2(float& m, float& s, float x, float y) const {
    const float mn = fmax_finite(m, fmax_finite(x, y));
    const float r = mn == -INFINITY ? 0.f : mn * c;  // all -inf so far: keep s = 0
    s = fmaf(s, ex2_approx(fmaf(m, c, -r)), ex2_approx(fmaf(x, c, -r)) + ex2_approx(fmaf(y, c, -r)));
    m = mn;
  }
  __device__ __forceinline__ void merge(float& m, float& s, int o) const {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    const float mn = fmax_finite(m, om);
    const float r = mn == -INFINITY ? 0.f : mn * c;
    s = fmaf(s, ex2_approx(fmaf(m, c, -r)), os * ex2_approx(fmaf(om, c, -r)));
    m = mn;
  }
  template <bool kMask>
  __device__ __forceinline__ void add(float v0, float v1, float v2, float v3, int t0, int L0,
                                      int L1) {
    if (kMask) {
      v0 = t0 < L0 ? v0 : -INFINITY;
      v1 = t0 + 1 < L0 ? v1 : -INFINITY;
      v2 = t0 < L1 ? v2 : -INFINITY;
      v3 = t0 + 1 < L1 ? v3 : -INFINITY;
    }
    push2(m0, s0, v0, v1);
    push2(m1, s1, v2, v3);
  }
  __device__ __forceinline__ void reduce() {
    merge(m0, s0, 1);
    merge(m0, s0, 2);
    merge(m1, s1, 1);
    merge(m1, s1, 2);
  }
  __device__ __forceinline__ float lse(float m, float s) const {
    return m == -INFINITY ? m : (m * c + log2f(s)) * 0.6931471805599453f;
  }
  __device__ __forceinline__ float out0() const { return lse(m0, s0); }
  __device__ __forceinline__ float out1() const { return lse(m1, s1); }
};

// ---------------------------------------------------------------------------
// Query tiles in mma.sync A-fragment order.
// ---------------------------------------------------------------------------
template <int KF>
struct QTile;

// bf16: 8 k-steps of 16, a[ks] = {A[g][16ks+2t..], A[g+8][..], A[g][16ks+8+2t..], A[g+8][..]}
template <>
struct QTile<kBf16> {
  uint32_t a[8][4];
  __device__ float post_scale() const { return 1.f; }
  __device__ void load(const ScoreArgs& args, int q_row0, int nrows, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* r0 = args.q + (size_t)(q_row0 + g) * 256;
    const uint8_t* r1 = args.q + (size_t)(q_row0 + g + 8) * 256;
    const bool v0 = g < nrows, v1 = g + 8 < nrows;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int o0 = (16 * ks + 2 * t) * 2, o1 = (16 * ks + 8 + 2 * t) * 2;
      a[ks][0] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(r0 + o0)) : 0u;
      a[ks][1] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(r1 + o0)) : 0u;
      a[ks][2] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(r0 + o1)) : 0u;
      a[ks][3] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(r1 + o1)) : 0u;
    }
  }
};

// e4m3: 4 k-steps of 32, a[ks] = {A[g][32ks+4t..+3], A[g+8][..], A[g][32ks+16+4t..], A[g+8][..]}
template <>
struct QTile<kFp8> {
  uint32_t a[4][4];
  __device__ float post_scale() const { return 1.f; }
  __device__ void load(const ScoreArgs& args, int q_row0, int nrows, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* r0 = args.q + (size_t)(q_row0 + g) * 128;
    const uint8_t* r1 = args.q + (size_t)(q_row0 + g + 8) * 128;
    const bool v0 = g < nrows, v1 = g + 8 < nrows;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const int o0 = 32 * ks + 4 * t, o1 = 32 * ks + 16 + 4 * t;
      a[ks][0] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(r0 + o0)) : 0u;
      a[ks][1] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(r1 + o0)) : 0u;
      a[ks][2] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(r0 + o1)) : 0u;
      a[ks][3] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(r1 + o1)) : 0u;
    }
  }
};

// NVFP4 keys with bf16 q: the query is rescaled by 2^qexp (one power of two per
// group, chosen so its largest magnitude lands in [2^14, 2^15)) and stored as
// f16, exact for every element within 2^24 of the largest.  The decoded keys
// (e2m1 x E4M3) are exact in f16, so each product is exact and the fp32 sum is
// rescaled by 2^-qexp afterwards.
//
// k order: k-step ks = 2m + hh takes, for thread t, the elements
// d = 32m + 8t + 4hh + {0,1} (b0) and + {2,3} (b1) of its key, which is the order
// the packed bytes of the key arrive in; the query is gathered the same way.
template <>
struct QTile<kNvfp4> {
  uint32_t a[8][4];
  float inv_scale;  // 2^-qexp
  __device__ float post_scale() const { return inv_scale; }
  __device__ void load(const ScoreArgs& args, int q_row0, int nrows, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const bool v0 = g < nrows, v1 = g + 8 < nrows;
    const __nv_bfloat16* r0 = reinterpret_cast<const __nv_bfloat16*>(args.q) + (size_t)(q_row0 + g) * 128;
    const __nv_bfloat16* r1 = reinterpret_cast<const __nv_bfloat16*>(args.q) + (size_t)(q_row0 + g + 8) * 128;
    float x0[4][8], x1[4][8];
    float amax = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      uint4 u0 = v0 ? __ldg(reinterpret_cast<const uint4*>(r0 + 32 * m + 8 * t)) : make_uint4(0, 0, 0, 0);
      uint4 u1 = v1 ? __ldg(reinterpret_cast<const uint4*>(r1 + 32 * m + 8 * t)) : make_uint4(0, 0, 0, 0);
      const uint32_t w0[4] = {u0.x, u0.y, u0.z, u0.w};
      const uint32_t w1[4] = {u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x0[m][2 * e] = __uint_as_float(w0[e] << 16);
        x0[m][2 * e + 1] = __uint_as_float(w0[e] & 0xffff0000u);
        x1[m][2 * e] = __uint_as_float(w1[e] << 16);
        x1[m][2 * e + 1] = __uint_as_float(w1[e] & 0xffff0000u);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fmaxf(fabsf(x0[m][e]), fabsf(x1[m][e])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int qexp = 0;
    if (amax > 0.f) {
      const int e = ((__float_as_uint(amax) >> 23) & 0xff) - 127;  // amax in [2^e, 2^(e+1))
      qexp = 14 - e;
    }
    qexp = max(-100, min(100, qexp));
    const float up = ldexpf(1.f, qexp);
    inv_scale = ldexpf(1.f, -qexp);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int ks = 2 * m + hh;
        const float* p0 = &x0[m][4 * hh];
        const float* p1 = &x1[m][4 * hh];
        __half2 h;
        h = __floats2half2_rn(p0[0] * up, p0[1] * up);
        a[ks][0] = *reinterpret_cast<uint32_t*>(&h);
        h = __floats2half2_rn(p1[0] * up, p1[1] * up);
        a[ks][1] = *reinterpret_cast<uint32_t*>(&h);
        h = __floats2half2_rn(p0[2] * up, p0[3] * up);
        a[ks][2] = *reinterpret_cast<uint32_t*>(&h);
        h = __floats2half2_rn(p1[2] * up, p1[3] * up);
        a[ks][3] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
  }
};

// ---------------------------------------------------------------------------
// Block max of one 128-token block for the 16 tile rows (one warp).
// Returns the running maxima of rows g (mx0) and g + 8 (mx1) over the tokens
// this lane saw; the caller reduces across the 4 lanes of a row.
// ---------------------------------------------------------------------------
template <int KF>
struct BlockScorer;

template <>
struct BlockScorer<kBf16> {
  template <bool kMask, class Score>
  __device__ static void run(const QTile<kBf16>& qt, uint32_t stage, uint32_t /*scale_stage*/,
                             const float* /*scale_smem*/, int lane, int tbase, int L0, int L1,
                             float qs0, float qs1, Score& sc) {
    const int t = lane & 3;
    const int m = lane >> 3, rr = lane & 7;
#pragma unroll 2
    for (int nt = 0; nt < 16; ++nt) {
      const int j = nt * 8 + rr;
      const int p = j >> 6, n = j & 63;
      const uint32_t row_base = stage + (uint32_t)(p * 8192 + n * 128);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int qd = 4 * c + m;  // 16-byte chunk of d (0..15)
        const int h = qd >> 3, cq = qd & 7;
        const uint32_t addr = row_base + (uint32_t)(h * 16384) + (uint32_t)(((cq ^ rr) & 7) << 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(addr, b0, b1, b2, b3);
        mma_bf16_16816(acc, qt.a[2 * c], b0, b1);
        mma_bf16_16816(acc, qt.a[2 * c + 1], b2, b3);
      }
      const int t0 = tbase + nt * 8 + 2 * t;
      sc.template add<kMask>(acc[0], acc[1], acc[2], acc[3], t0, L0, L1);
    }
    (void)qs0;
    (void)qs1;
  }
};

template <>
struct BlockScorer<kFp8> {
  template <bool kMask, class Score>
  __device__ static void run(const QTile<kFp8>& qt, uint32_t stage, uint32_t /*scale_stage*/,
                             const float* scale_smem, int lane, int tbase, int L0, int L1,
                             float qs0, float qs1, Score& sc) {
    const int t = lane & 3;
    const int m = lane >> 3, rr = lane & 7;
#pragma unroll 2
    for (int nt = 0; nt < 16; ++nt) {
      const int j = nt * 8 + rr;
      const int p = j >> 6, n = j & 63;
      const uint32_t row_base = stage + (uint32_t)(p * 8192 + n * 128);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int qd = 4 * c + m;  // 16-byte chunk of the 128-byte row
        const uint32_t addr = row_base + (uint32_t)(((qd ^ rr) & 7) << 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(addr, b0, b1, b2, b3);
        mma_e4m3_16832(acc, qt.a[2 * c], b0, b1);
        mma_e4m3_16832(acc, qt.a[2 * c + 1], b2, b3);
      }
      const int jt = nt * 8 + 2 * t;  // token of acc[0] within the block
      const float2 ks = *reinterpret_cast<const float2*>(scale_smem + jt);
      const int t0 = tbase + jt;
      // (dot * q scale) * key scale, two scores per packed multiply
      const float2 y0 = fmul2_rn(fmul2_rn(make_float2(acc[0], acc[1]), make_float2(qs0, qs0)), ks);
      const float2 y1 = fmul2_rn(fmul2_rn(make_float2(acc[2], acc[3]), make_float2(qs1, qs1)), ks);
      sc.template add<kMask>(y0.x, y0.y, y1.x, y1.y, t0, L0, L1);
    }
  }
};

template <>
struct BlockScorer<kNvfp4> {
  template <bool kMask, class Score>
  __device__ static void run(const QTile<kNvfp4>& qt, uint32_t stage, uint32_t scale_stage,
                             const float* /*scale_smem*/, int lane, int tbase, int L0, int L1,
                             float /*qs0*/, float /*qs1*/, Score& score) {
    const int g = lane >> 2, t = lane & 3;
    const int m = lane >> 3, rr = lane & 7;
    const uint32_t th = (uint32_t)(t >> 1);
    // byte selectors {th, th, 2+th, 2+th}: duplicate the scale of group 2m + th
    const uint32_t sel = th | (th << 4) | ((2 + th) << 8) | ((2 + th) << 12);
    // the block max scores a whole block per loop (measured 3-4% faster than
    // two slices at a time); the lse accumulator needs the registers
    constexpr int kUnroll = Score::kWholeBlockUnroll ? 16 : 2;
#pragma unroll kUnroll
    for (int nt = 0; nt < 16; ++nt) {
      // B operand: this lane's ldmatrix row address (token nt*8 + rr, chunk m)
      const int j = nt * 8 + rr;
      const int p = j >> 6, n = j & 63;
      const uint32_t addr = stage + (uint32_t)(p * 4096 + n * 64) +
                            (uint32_t)(((m ^ ((n >> 1) & 3)) & 3) << 4);
      uint32_t w[4];
      ldmatrix_x4(addr, w[0], w[1], w[2], w[3]);
      // scales of the token this lane holds in the B fragment: token nt*8 + g
      const int jb = nt * 8 + g;
      const int pb = jb >> 6, nb = jb & 63;
      uint32_t s_lo, s_hi;
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                   : "=r"(s_lo), "=r"(s_hi)
                   : "r"(scale_stage + (uint32_t)(pb * 512 + nb * 8)));
      uint32_t sc[4];
      e4m3x4_to_f16x2x2(prmt(s_lo, 0u, sel), sc[0], sc[1]);
      e4m3x4_to_f16x2x2(prmt(s_hi, 0u, sel), sc[2], sc[3]);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {
        uint32_t f[4];
        e2m1x8_to_f16x2x4(w[mm], f);
        const uint32_t k0 = hmul2_f16(f[0], sc[mm]);
        const uint32_t k1 = hmul2_f16(f[1], sc[mm]);
        const uint32_t k2 = hmul2_f16(f[2], sc[mm]);
        const uint32_t k3 = hmul2_f16(f[3], sc[mm]);
        mma_f16_16816(acc, qt.a[2 * mm], k0, k1);
        mma_f16_16816(acc, qt.a[2 * mm + 1], k2, k3);
      }
      const int t0 = tbase + nt * 8 + 2 * t;
      // raw sums of the rescaled query: the score applies qt.post_scale()
      score.template add<kMask>(acc[0], acc[1], acc[2], acc[3], t0, L0, L1);
    }
  }
};

// ---------------------------------------------------------------------------
// Work units: unit u (one 128-token block) of the call's flattened list is
// block b of group v, found by binary search in the shared prefix table.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void locate(const int* gpre, int V, int u, int& v, int& b) {
  int lo = 0, hi = V - 1;  // largest v with gpre[v] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (gpre[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  v = lo;
  b = u - gpre[lo];
}

// Page ids of block b of group v (-1: no second page, -2: bad page id, not
// read).  Lanes 0 and 1 load one page-table entry each.  gslot[v] holds the
// group's slot, with bit 31 set when its last block needs only one page.
__device__ __forceinline__ int load_page(const ScoreArgs& a, const int* gpre, const int* gslot,
                                         int v, int b, int lane, uint32_t* flags) {
  int p = -1;
  if (lane < 2) {
    const int word = gslot[v];
    const int slot = word & 0x7fffffff;
    const bool last = b == gpre[v + 1] - gpre[v] - 1;
    const bool want = lane == 0 || !(last && word < 0);
    if (want) {
      p = __ldg(a.page_table + (size_t)slot * a.max_pages + 2 * b + lane);
      if (p < 0 || p >= a.num_pages) {
        atomicOr(flags, kErrBadPage);
        p = -2;
      }
    }
  }
  return p;
}

// Page ids of block b of group v as a prefetch hint (no flags; -1: none or
// out of range).  Lanes 0 and 1 load one page-table entry each.
__device__ __forceinline__ int hint_page(const ScoreArgs& a, const int* gpre, const int* gslot,
                                         int v, int b, int lane) {
  int p = -1;
  if (lane < 2) {
    const int word = gslot[v];
    const int slot = word & 0x7fffffff;
    const bool last = b == gpre[v + 1] - gpre[v] - 1;
    if ((lane == 0 || !(last && word < 0)) && slot < a.n_slots && 2 * b + lane < a.max_pages) {
      p = ld_in<true>(a.page_table + (size_t)slot * a.max_pages + 2 * b + lane);
      if (p < 0 || p >= a.num_pages) p = -1;
    }
  }
  return p;
}

// Bring one unit's pages (payload and scales) into L2 (lane 0 only).
template <int KF>
__device__ __forceinline__ void prefetch_unit(const ScoreArgs& a, const CUtensorMap* map, int p0,
                                              int p1) {
  using L = Layout<KF>;
  const int pg[2] = {p0, p1};
#pragma unroll
  for (int pp = 0; pp < 2; ++pp) {
    if (pg[pp] < 0) continue;
    const int y = pg[pp] * kPage;
    if (KF == kBf16) {
      tma_prefetch_2d(map, 0, y);
      tma_prefetch_2d(map, 64, y);
    } else {
      tma_prefetch_2d(map, 0, y);
      bulk_prefetch_l2(a.k_scale + (size_t)pg[pp] * L::kPageScale, L::kPageScale);
    }
  }
}

// Issue the copies of one unit into stage s (lane 0 only).
template <int KF>
__device__ __forceinline__ void issue_unit(const ScoreArgs& a, const CUtensorMap* map,
                                           uint32_t sbase, int s, int p0, int p1) {
  using L = Layout<KF>;
  using C = Cfg<KF>;
  uint32_t tx = 0;
  if (p0 >= 0) tx += C::kPagePayload + L::kPageScale;
  if (p1 >= 0) tx += C::kPagePayload + L::kPageScale;
  const uint32_t full = sbase + L::kBarOff + s * 8;
  mbar_arrive_expect_tx(full, tx);
  const uint32_t dst = sbase + L::kPayloadOff + s * L::kStagePayload;
  const uint32_t sdst = sbase + L::kScaleOff + s * L::kStageScale;
  const int pg[2] = {p0, p1};
#pragma unroll
  for (int pp = 0; pp < 2; ++pp) {
    if (pg[pp] < 0) continue;
    const int y = pg[pp] * kPage;
    if (KF == kBf16) {
      // two 64-column boxes per page: d 0..63 and d 64..127
      tma_load_2d(dst + pp * 8192, map, 0, y, full);
      tma_load_2d(dst + 16384 + pp * 8192, map, 64, y, full);
    } else {
      tma_load_2d(dst + pp * C::kPagePayload, map, 0, y, full);
      bulk_load(sdst + pp * L::kPageScale, a.k_scale + (size_t)pg[pp] * L::kPageScale,
                L::kPageScale, full);
    }
  }
}

// The shared group table, built by the calling warp: pre[v] = first unit of
// group v (prefix sum of the groups' block counts), pre[V] = units of the call,
// slot[v] = the group's slot with bit 31 set when its last block needs one
// page; ctl[0..2] = units, first dynamically scheduled unit, dynamic schedule
// on.  hint: built before the programmatic wait from inputs that may still
// change (read through L2 only); only pre, slot and ctl[0..1] are written.
template <int KF, bool hint>
__device__ __forceinline__ void build_groups(const ScoreArgs& a, int* pre, int* slot,
                                             volatile int* ctl, unsigned int* cta_flags, int V,
                                             int lane) {
  // read up front, so its round trip overlaps the row-length loads
  const bool tag_ok = lane == 0 && (hint ? __ldcg(a.sched_tag) : *a.sched_tag) == kSchedTag;
  int run = 0;
  bool clamped = false;
  for (int v0 = 0; v0 < V; v0 += 32) {
    const int v = v0 + lane;
    int nbk = 0, word = 0;
    if (v < V) {
      const Group gi = group_info<hint>(a, v);
      nbk = gi.nbk;
      const int rem = gi.extent - (a.block_off + nbk - 1) * kBlock;  // tokens in the last block
      word = (nbk > 0 ? gi.slot : 0) | ((nbk > 0 && rem <= kPage) ? (int)0x80000000 : 0);
      if (!hint && blockIdx.x == 0 && !a.shard && gi.slot >= 0 && gi.slot < a.n_slots) {
        const int j0 = a.perrow ? v - gi.r * a.P : 0, j1 = a.perrow ? j0 + 1 : a.P;
        for (int j = j0; j < j1; ++j)
          clamped |= __ldg(a.row_lens + gi.r * a.P + j) > a.max_pages * kPage;
      }
    }
    int incl = nbk;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (v < V) {
      pre[v] = run + incl - nbk;
      slot[v] = word;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  clamped = __any_sync(0xffffffffu, clamped);
  if (lane == 0) {
    pre[V] = run;
    // the last part of the blocks is handed out at run time, which evens out
    // the CTAs' finish times: an eighth from ~600 blocks per CTA, from 64 a
    // quarter for bf16 and an eighth for fp8 (measured best on 16 x 131K
    // calls: bf16 82.7 us a step against 84.3 with an eighth, fp8 52.9 against
    // 53.6 with a quarter; all static: 87.2 / 56.8); NVFP4 calls
    // below 600 stay static, since a block from another request costs a
    // query-tile conversion there.  Only when a previous call left the
    // counter at zero (its tag says so).
    const int grid = (int)gridDim.x;
    int share = 0;  // 1 / share of the blocks is dynamic
    if (tag_ok) {
      if (run >= 600 * grid) share = 8;
      else if (KF != kNvfp4 && run >= 64 * grid) share = KF == kFp8 ? 8 : 4;
    }
    ctl[0] = run;
    ctl[1] = share ? run - run / share : run;
    if (!hint) {
      ctl[2] = share ? 1 : 0;
      *cta_flags = clamped ? kErrLenClamped : 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int KF, class Score>
__global__ void __launch_bounds__(Layout<KF>::kThreads, 1)
    score_kernel(const ScoreArgs a, const __grid_constant__ CUtensorMap payload_map) {
  using L = Layout<KF>;
  constexpr int NC = L::NC;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + L::kCtlOff);
  // ctl[0] = units of the call, ctl[1] = first dynamically scheduled unit,
  // ctl[2] = dynamic schedule on, ctl[4] = this CTA's device error flags,
  // ctl[6] = the real group table is built (a hint to the warm-up work)
  unsigned int* cta_flags = reinterpret_cast<unsigned int*>(smem + L::kCtlOff) + 4;
  int* gpre = reinterpret_cast<int*>(smem + L::kGroupOff);  // [V + 1] block prefix
  int* gslot = gpre + kMaxGroups + 1;                      // [V] slot | one-page-last bit

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
#pragma unroll
    for (int d = 0; d < L::D; ++d) mbar_init(sbase + L::kBarOff + (warp * L::D + d) * 8, 1);
    if (warp == 0) mbar_init(sbase + L::kCtlOff + 32, 1);  // the stall test's barrier
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    prefetch_tensormap(&payload_map);
    ctl[6] = 0;
  }

  // ---- group table: block prefix sums and slots of every group -------------
  // The kernel is launched as a programmatic dependent of whatever ran before
  // on the stream, so it may start while that work still runs: inputs are
  // read and the workspace written only after griddepcontrol.wait.  Warp 1
  // waits and builds the real table.  Meanwhile the other warps read the
  // inputs as they stand, as a hint (through L2 only): warp 0 builds a hint
  // table of the groups, the others bring every request's page-table row into
  // L2 (one 128-byte line per thread), and then each warp brings the pages of
  // its first static blocks into L2.  A prefetch moves nothing into this CTA
  // and L2 is coherent, so a stale hint costs only bandwidth.  The warm-up
  // only pays while the wait holds: once warp 1 has built the real table
  // (nothing ran before, or it has finished) the other warps drop what is left
  // of it and start on their blocks.
  // NVFP4 calls are bound by the key decode, not by HBM, and measured slower
  // with the hint work: they wait first and warm only the page table.
  const int V = a.perrow ? a.R * a.P : a.R;
  if (KF == kNvfp4) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (warp == 1) {
      build_groups<KF, false>(a, gpre, gslot, ctl, cta_flags, V, lane);
    } else if (warp >= 2) {
      const int lines_per = (a.max_pages + 31) / 32;
      const int nthr = (int)gridDim.x * (NC - 2) * 32;
      const int gt = ((int)blockIdx.x * (NC - 2) + warp - 2) * 32 + lane;
      if (a.R * lines_per <= nthr && gt < a.R * lines_per) {
        const int r = gt / lines_per, line = gt - r * lines_per;
        const int slot = __ldg(a.slot_ids + r);
        if (slot >= 0 && slot < a.n_slots)
          prefetch_l2(a.page_table + (size_t)slot * a.max_pages + (size_t)line * 32);
      }
    }
  } else if (warp == 1) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    build_groups<KF, false>(a, gpre, gslot, ctl, cta_flags, V, lane);
    __syncwarp();
    if (lane == 0) ctl[6] = 1;
  } else {
    int* hpre = reinterpret_cast<int*>(smem + L::kHintOff);  // [V + 1]
    int* hslot = hpre + kHintGroups + 1;                     // [V]
    volatile int* hctl = hslot + kHintGroups;                // units, first dynamic unit
    const bool hinted = V <= kHintGroups;
    if (warp == 0) {
      if (hinted) {
        if (!__any_sync(0xffffffffu, ctl[6] != 0))
          build_groups<KF, true>(a, hpre, hslot, hctl, nullptr, V, lane);
        else if (lane == 0)
          hctl[0] = 0;  // no blocks to warm
      }
    } else if (ctl[6] == 0) {
      const int lines_per = (a.max_pages + 31) / 32;
      const int nthr = (int)gridDim.x * (NC - 2) * 32;
      const int gt = ((int)blockIdx.x * (NC - 2) + warp - 2) * 32 + lane;
      if (a.R * lines_per <= nthr && gt < a.R * lines_per) {
        const int r = gt / lines_per, line = gt - r * lines_per;
        const int slot = ld_in<true>(a.slot_ids + r);
        if (slot >= 0 && slot < a.n_slots)
          prefetch_l2(a.page_table + (size_t)slot * a.max_pages + (size_t)line * 32);
      }
    }
    // every warp but warp 1: the hint table is complete
    asm volatile("bar.sync 1, %0;" ::"r"((NC - 1) * 32) : "memory");
    if (hinted) {
      const int Uh = hctl[0], Ush = hctl[1];
      const int sh0 = (int)((long long)Ush * blockIdx.x / gridDim.x);
      const int sh1 = (int)((long long)Ush * (blockIdx.x + 1) / gridDim.x);
      // the CTA's first NC * kPrefetchUnits static units (warp w's j-th block is
      // unit sh0 + w + j NC), spread over the NC - 1 warps here
      const int rank = warp == 0 ? 0 : warp - 1;
      for (int k = rank; k < NC * kPrefetchUnits; k += NC - 1) {
        if (__any_sync(0xffffffffu, ctl[6] != 0)) break;
        const int u = sh0 + k;
        if (u < sh1 && u < Uh) {
          int v, b;
          locate(hpre, V, u, v, b);
          const int pg = hint_page(a, hpre, hslot, v, b, lane);
          const int p0 = __shfl_sync(0xffffffffu, pg, 0), p1 = __shfl_sync(0xffffffffu, pg, 1);
          if (lane == 0) prefetch_unit<KF>(a, &payload_map, p0, p1);
        }
      }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }
  __syncthreads();
  // the top-k kernel may be scheduled now; it waits for this grid's completion
  // (and memory) before reading the block maxima
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int U = ctl[0], Us = ctl[1];
  const bool dyn = ctl[2] != 0;
  const int s1 = (int)((long long)Us * (blockIdx.x + 1) / gridDim.x);
  int sk = (int)((long long)Us * blockIdx.x / gridDim.x) + warp;  // next static unit

  // this warp's units: its share of the CTA's static range, then blocks taken
  // one at a time from the dynamic pool (each take is issued one unit ahead:
  // the first when the last static unit is handed out, not at the start, where
  // its round trip would delay the first copies)
  int ahead = -1;
  if (dyn && sk >= s1 && lane == 0) ahead = Us + (int)atomicAdd(a.sched_counter, 1u);
  auto next_unit = [&]() -> int {
    if (sk < s1) {
      const int u = sk;
      sk += NC;
      if (dyn && sk >= s1 && lane == 0) ahead = Us + (int)atomicAdd(a.sched_counter, 1u);
      return u;
    }
    if (!dyn) return -1;
    const int u = __shfl_sync(0xffffffffu, ahead, 0);
    if (u >= U) return -1;
    if (lane == 0) ahead = Us + (int)atomicAdd(a.sched_counter, 1u);
    return u;
  };

  constexpr int D = L::D;
  const int g = lane >> 2, t = lane & 3;
  bool aborted = false;

  // blocks in flight for this warp, oldest first: fv/fb = group and block
  int fv[D], fb[D];
  int nin = 0;
#pragma unroll
  for (int d = 0; d < D; ++d) {
    if (nin == d) {
      const int u = next_unit();
      if (u >= 0) {
        locate(gpre, V, u, fv[d], fb[d]);
        const int pg = load_page(a, gpre, gslot, fv[d], fb[d], lane, cta_flags);
        const int p0 = __shfl_sync(0xffffffffu, pg, 0), p1 = __shfl_sync(0xffffffffu, pg, 1);
        if (lane == 0) issue_unit<KF>(a, &payload_map, sbase, warp * D + d, p0, p1);
        ++nin;
      }
    }
  }
  // the block that goes out when the oldest one is scored (pages looked up early)
  int nxt = nin == D ? next_unit() : -1, v_n = 0, b_n = 0, pg_n = -1;
  if (nxt >= 0) {
    locate(gpre, V, nxt, v_n, b_n);
    pg_n = load_page(a, gpre, gslot, v_n, b_n, lane, cta_flags);
  }

  int k = 0;  // blocks scored by this warp
  int cur_v = -1;
  QTile<KF> qt;
  int L0 = 0, L1 = 0, row0 = -1, row1 = -1;
  float qs0 = 1.f, qs1 = 1.f;
  while (nin > 0) {
    const int v_cur = fv[0], b_cur = fb[0];
    const int sidx = warp * D + (k % D);
    const uint32_t stage = sbase + L::kPayloadOff + sidx * L::kStagePayload;
    const uint32_t scale_stage = sbase + L::kScaleOff + sidx * L::kStageScale;
    const float* scale_smem = reinterpret_cast<const float*>(smem + L::kScaleOff + sidx * L::kStageScale);
    const uint32_t bar = sbase + L::kBarOff + sidx * 8;
    // a new group's query tile is loaded while the block's keys are in flight
    if (v_cur != cur_v) {
      const Group gi = group_info(a, v_cur);
      qt.load(a, gi.base_row, gi.nrows, lane);
      L0 = g < gi.nrows ? tile_row_len(a, v_cur, gi.r, g) : 0;
      L1 = g + 8 < gi.nrows ? tile_row_len(a, v_cur, gi.r, g + 8) : 0;
      row0 = g < gi.nrows ? gi.base_row + g : -1;
      row1 = g + 8 < gi.nrows ? gi.base_row + g + 8 : -1;
      if (KF == kFp8) {
        qs0 = row0 >= 0 ? __ldg(a.q_scale + row0) : 0.f;
        qs1 = row1 >= 0 ? __ldg(a.q_scale + row1) : 0.f;
      }
      cur_v = v_cur;
    }
    // stall test: warp 0's first wait goes to a barrier nothing completes
    const bool stall = a.stall_test && warp == 0 && k == 0;
    if (!mbar_wait_bounded(stall ? sbase + L::kCtlOff + 32 : bar, stall ? 0u : (k / D) & 1,
                           a.wait_ns)) {
      if (lane == 0) atomicOr(cta_flags, kErrTimeout);
      aborted = true;
      break;
    }
    __syncwarp();
    const int tbase = (a.block_off + b_cur) * kBlock;  // global token of the block
    Score score(qt.post_scale());
    // most blocks lie inside every live row: score them without the mask
    const bool whole = __all_sync(0xffffffffu, (row0 < 0 || tbase + kBlock <= L0) &&
                                                   (row1 < 0 || tbase + kBlock <= L1));
    if (whole)
      BlockScorer<KF>::template run<false>(qt, stage, scale_stage, scale_smem, lane, tbase, L0,
                                           L1, qs0, qs1, score);
    else
      BlockScorer<KF>::template run<true>(qt, stage, scale_stage, scale_smem, lane, tbase, L0,
                                          L1, qs0, qs1, score);
    // every lane's shared-memory reads of this stage are done; order them
    // before the asynchronous copies that overwrite it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    const int p0 = __shfl_sync(0xffffffffu, pg_n, 0), p1 = __shfl_sync(0xffffffffu, pg_n, 1);
    if (nxt >= 0 && lane == 0) issue_unit<KF>(a, &payload_map, sbase, sidx, p0, p1);
    score.reduce();
    if (t == 0) {
      if (row0 >= 0 && tbase < L0) a.blockmax[(size_t)row0 * a.nb_cap + b_cur] = score.out0();
      if (row1 >= 0 && tbase < L1) a.blockmax[(size_t)row1 * a.nb_cap + b_cur] = score.out1();
    }
#pragma unroll
    for (int d = 0; d + 1 < D; ++d) {
      fv[d] = fv[d + 1];
      fb[d] = fb[d + 1];
    }
    fv[D - 1] = v_n;
    fb[D - 1] = b_n;
    ++k;
    if (nxt < 0) {
      --nin;
      continue;
    }
    nxt = next_unit();
    pg_n = -1;
    if (nxt >= 0) {
      locate(gpre, V, nxt, v_n, b_n);
      pg_n = load_page(a, gpre, gslot, v_n, b_n, lane, cta_flags);
    }
  }
  // after a timeout, let this warp's copies still in flight land before exiting
  if (aborted && lane == 0) {
    for (int j = 0; j < nin; ++j) {
      const int kk = k + j;
      (void)mbar_wait_bounded(sbase + L::kBarOff + (warp * D + kk % D) * 8, (kk / D) & 1,
                              200000000ull);
    }
  }
  // publish this CTA's flags (one byte per CTA, overwritten by every call, so no
  // clearing is needed between calls)
  __syncthreads();
  if (threadIdx.x == 0) {
    a.err_bytes[blockIdx.x] = (uint8_t)*cta_flags;
    if (blockIdx.x == 0) *a.err_count = gridDim.x;
  }
#if IDX_FUSED_TOPK
  if (!a.fused) return;
  // ---- selection in this kernel: a grid barrier (every CTA of the persistent
  // grid is resident: one per SM), then row k is selected by CTA k % grid with
  // the block scores read from L2; the last CTA out resets the counters ------
  volatile int* go = ctl + 12;  // ctl[8..9] hold the stall test's barrier
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(a.arrive, 1u);
    const uint64_t t0 = global_timer_ns();
    int ok = 1;
    for (uint32_t it = 0;; ++it) {
      uint32_t n;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(n) : "l"(a.arrive) : "memory");
      if (n >= gridDim.x) break;
      if ((it & 15u) == 15u && global_timer_ns() - t0 > a.wait_ns) {
        ok = 0;
        break;
      }
    }
    if (!ok) a.err_bytes[blockIdx.x] = (uint8_t)(*cta_flags | kErrTimeout);
    *go = ok;
  }
  __syncthreads();
  if (*go) {
    const TopkArgs& ta = a.topk;
    for (int row = blockIdx.x; row < ta.R * ta.M; row += gridDim.x) {
      const int r = row / ta.M;
      const sel::RowPlan pl = sel::row_plan(ta, r, row - r * ta.M);
      sel::row_pads<L::kThreads>(ta, row, pl, threadIdx.x);
      sel::row_select<L::kThreads, true>(ta, row, pl, smem, threadIdx.x);
      __syncthreads();
    }
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.depart, 1u) == gridDim.x - 1) {
      *reinterpret_cast<volatile uint32_t*>(a.arrive) = 0u;
      *reinterpret_cast<volatile uint32_t*>(a.depart) = 0u;
      *reinterpret_cast<volatile uint32_t*>(a.sched_counter) = 0u;
      __threadfence();
      *reinterpret_cast<volatile unsigned long long*>(a.topk.sched_tag) = kSchedTag;
    }
  }
#endif
}

std::atomic<int> g_grid_limit{0};

template <int KF, class Score>
cudaError_t launch_kf(const ScoreArgs& a, const CUtensorMap& map, cudaStream_t stream) {
  using L = Layout<KF>;
  static std::atomic<unsigned long long> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int sms = cached_sm_count(dev);
  if (sms <= 0) return cudaErrorInvalidDevice;
  e = smem_limit_once(score_kernel<KF, Score>, L::kSmemBytes, dev, attr_done);
  if (e != cudaSuccess) return e;
  const int lim = g_grid_limit.load(std::memory_order_relaxed);
  int grid = (lim > 0 && lim < sms) ? lim : sms;
  if (grid > kMaxScoreCtas) grid = kMaxScoreCtas;
  e = launch_pdl(score_kernel<KF, Score>, grid, L::kThreads, L::kSmemBytes, stream, a, map);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <class Score>
cudaError_t launch_bs(int key_format, const ScoreArgs& args, const CUtensorMap& map,
                      cudaStream_t stream) {
  switch (key_format) {
    case kBf16:
      return launch_kf<kBf16, Score>(args, map, stream);
    case kFp8:
      return launch_kf<kFp8, Score>(args, map, stream);
    case kNvfp4:
      return launch_kf<kNvfp4, Score>(args, map, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

std::atomic<unsigned long long> g_wait_ns{2000000000ull};
void set_wait_limit_ns(unsigned long long ns) { g_wait_ns.store(ns ? ns : 2000000000ull); }
unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
std::atomic<int> g_stall_test{0};
void set_stall_test(int on) { g_stall_test.store(on ? 1 : 0); }
int stall_test() { return g_stall_test.load(std::memory_order_relaxed); }

void set_grid_limit(int max_ctas) { g_grid_limit.store(max_ctas < 0 ? 0 : max_ctas); }
int grid_limit() { return g_grid_limit.load(); }

cudaError_t launch_score(int key_format, int block_score, const ScoreArgs& args,
                         const CUtensorMap& payload_map, cudaStream_t stream) {
  if (block_score == kBlockLse) return launch_bs<LseScore>(key_format, args, payload_map, stream);
  return launch_bs<MaxScore>(key_format, args, payload_map, stream);
}

}  // namespace idx

// NVFP4 quantize-store of staged bf16 keys into the paged pool planes.
//
// What it computes (ROCm/ATOM #2745, Summary, "Store" and "Write"): each key of
// D = 128 is quantised per group of 16 elements with scale = E4M3(amax / 6) and
// e2m1 codes rounded half-to-even that saturate at 6, with a unit outer scale;
// two codes per byte, the even element in the low nibble; the payload (64 B) and
// the scale byte of each group (8 B) go to the key's real slot in two planes.
//
// Readings of the points the page leaves open: amax and amax/6 in fp32 with a
// correctly rounded division; the scale rounds half-to-even and saturates at
// 448; a zero scale writes all-zero codes; codes are those of the correctly
// rounded fp32 quotient x / scale; a negative value that rounds to zero keeps
// its sign.
//
// The codes come from the hardware e2m1 conversion (round to nearest, ties to
// the even code, saturating at 6, the sign kept) of a quotient q2 that equals
// x / s where that is on the e2m1 grid's midpoints and is within two ulps of it
// elsewhere: q1 = x * r with r = 1 / s, the residual e = x - q1 * s (exact in
// one fma), q2 = q1 + e * r (one correction step of a reciprocal-based
// quotient, after Markstein, "IA-64 and Elementary Functions", 2000).  This is
// enough: every midpoint t of the grid has at most three significant bits and
// s at most four, so t * s is a bf16 value, and a bf16 x either equals t * s
// (then the residual is exact and q2 = t) or lies a bf16 spacing away from it,
// far beyond the quotient's error, on the same side as fl(x / s).
//
// One thread per (key, group of 16): eight threads cover a key, a warp four.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>
#include <string.h>

#include "idx_internal.cuh"

namespace idx {

namespace {

// Value of an E4M3 byte with the sign bit clear (scales are never negative):
// exponent field 0 -> m * 2^-9; otherwise (8 + m) * 2^(e - 10).
__device__ __forceinline__ float e4m3_magnitude(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xfu, m = b & 7u;
  if (e == 0) return (float)m * 0.001953125f;
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

__device__ __forceinline__ __nv_bfloat162 as_bf16x2(uint32_t u) {
  __nv_bfloat162 v;
  memcpy(&v, &u, sizeof(v));
  return v;
}

// x / s on the e2m1 midpoints, within two ulps elsewhere (see above), with
// x's sign (the fma steps would turn -0 into +0).
__device__ __forceinline__ float grid_quotient(float x, float s, float r) {
  const float q1 = x * r;
  return copysignf(fmaf(fmaf(-q1, s, x), r, q1), x);
}

// Byte of two e2m1 codes: the code of lo in the low nibble, of hi in the high.
__device__ __forceinline__ uint32_t e2m1x2_byte(float lo, float hi) {
  uint32_t d;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(d)
      : "f"(hi), "f"(lo));
  return d;
}

// Quantise one group (its 16 bf16 values in w) and write it.
__device__ __forceinline__ void store_group(const uint32_t (&w)[8], int64_t row, int grp,
                                            uint8_t* payload, uint8_t* scale) {
  // amax of the 16 magnitudes (a max is exact in any order)
  __nv_bfloat162 m2 = as_bf16x2(w[0] & 0x7fff7fffu);
#pragma unroll
  for (int e = 1; e < 8; ++e) m2 = __hmax2(m2, as_bf16x2(w[e] & 0x7fff7fffu));
  const float amax = fmaxf(__low2float(m2), __high2float(m2));
  const float s_f = __fdiv_rn(amax, 6.0f);
  const uint32_t s_code =
      (uint32_t)__nv_cvt_float_to_fp8(s_f, __NV_SATFINITE, __NV_E4M3) & 0x7fu;
  const float s = e4m3_magnitude(s_code);
  uint32_t lo = 0, hi = 0;
  if (s > 0.f) {
    const float r = __frcp_rn(s);
    uint32_t byte[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x0 = __uint_as_float(w[e] << 16), x1 = __uint_as_float(w[e] & 0xffff0000u);
      byte[e] = e2m1x2_byte(grid_quotient(x0, s, r), grid_quotient(x1, s, r));
    }
    lo = byte[0] | (byte[1] << 8) | (byte[2] << 16) | (byte[3] << 24);
    hi = byte[4] | (byte[5] << 8) | (byte[6] << 16) | (byte[7] << 24);
  }
  *reinterpret_cast<uint2*>(payload + row * 64 + grp * 8) = make_uint2(lo, hi);
  scale[row * 8 + grp] = (uint8_t)s_code;
}

// Each thread quantises kGroups groups, blockDim apart (each load instruction
// of a warp covers 1 KB of consecutive keys); all their loads go out before
// any of them is used.
constexpr int kGroups = 2;

__global__ void __launch_bounds__(256) store_nvfp4_kernel(const uint16_t* __restrict__ src,
                                                          const int64_t* __restrict__ slot_mapping,
                                                          int64_t num_tokens, uint8_t* payload,
                                                          uint8_t* scale, int64_t num_rows) {
  const int64_t base = (int64_t)blockIdx.x * blockDim.x * kGroups + threadIdx.x;
  uint4 u[kGroups][2];
  int64_t row[kGroups];
#pragma unroll
  for (int j = 0; j < kGroups; ++j) {
    const int64_t gid = base + (int64_t)j * blockDim.x;
    const int64_t tok = gid >> 3;
    row[j] = -1;
    if (tok < num_tokens) {
      // the key's bytes do not depend on its slot: the loads go out together
      const uint4* p = reinterpret_cast<const uint4*>(src + tok * kDim + (gid & 7) * 16);
      row[j] = __ldg(slot_mapping + tok);
      u[j][0] = __ldcs(p);
      u[j][1] = __ldcs(p + 1);
    }
  }
#pragma unroll
  for (int j = 0; j < kGroups; ++j) {
    if (row[j] < 0 || row[j] >= num_rows) continue;
    const uint32_t w[8] = {u[j][0].x, u[j][0].y, u[j][0].z, u[j][0].w,
                           u[j][1].x, u[j][1].y, u[j][1].z, u[j][1].w};
    store_group(w, row[j], (int)((base + (int64_t)j * blockDim.x) & 7), payload, scale);
  }
}

}  // namespace

cudaError_t launch_store_nvfp4(const uint16_t* src, const int64_t* slot_mapping, int64_t num_tokens,
                               uint8_t* payload, uint8_t* scale, int64_t num_rows,
                               cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  const int64_t groups = num_tokens * 8;
  const int64_t blocks = (groups + 256 * kGroups - 1) / (256 * kGroups);
  store_nvfp4_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, slot_mapping, num_tokens, payload,
                                                         scale, num_rows);
  return cudaGetLastError();
}

}  // namespace idx

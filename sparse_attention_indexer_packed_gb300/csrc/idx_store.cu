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
// 448; a zero scale writes all-zero codes; codes use x / scale with a correctly
// rounded fp32 division; a negative value that rounds to zero keeps its sign.
//
// One thread per (key, group of 16): eight threads cover a key, a warp four.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

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

// e2m1 code of v: nearest of {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the code with
// a zero mantissa bit, saturating at 6; the sign bit follows v's sign.
__device__ __forceinline__ uint32_t e2m1_code(float v) {
  const float x = fabsf(v);
  uint32_t c = (x > 0.25f) + (x >= 0.75f) + (x > 1.25f) + (x >= 1.75f) + (x > 2.5f) +
               (x >= 3.5f) + (x > 5.0f);
  if (signbit(v)) c |= 8u;
  return c;
}

__global__ void __launch_bounds__(256) store_nvfp4_kernel(const uint16_t* __restrict__ src,
                                                          const int64_t* __restrict__ slot_mapping,
                                                          int64_t num_tokens, uint8_t* payload,
                                                          uint8_t* scale, int64_t num_rows) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t tok = gid >> 3;
  const int grp = (int)(gid & 7);
  if (tok >= num_tokens) return;
  const int64_t row = __ldg(slot_mapping + tok);
  if (row < 0 || row >= num_rows) return;

  const uint4* p = reinterpret_cast<const uint4*>(src + tok * kDim + grp * 16);
  const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  float x[16];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x[2 * e] = __uint_as_float(w[e] << 16);
    x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    amax = fmaxf(amax, fmaxf(fabsf(x[2 * e]), fabsf(x[2 * e + 1])));
  }
  const float s_f = __fdiv_rn(amax, 6.0f);
  const uint32_t s_code =
      (uint32_t)__nv_cvt_float_to_fp8(s_f, __NV_SATFINITE, __NV_E4M3) & 0x7fu;
  const float s = e4m3_magnitude(s_code);
  uint32_t lo = 0, hi = 0;
  if (s > 0.f) {
#pragma unroll
    for (int e = 0; e < 8; ++e) lo |= e2m1_code(__fdiv_rn(x[e], s)) << (4 * e);
#pragma unroll
    for (int e = 0; e < 8; ++e) hi |= e2m1_code(__fdiv_rn(x[8 + e], s)) << (4 * e);
  }
  *reinterpret_cast<uint2*>(payload + row * 64 + grp * 8) = make_uint2(lo, hi);
  scale[row * 8 + grp] = (uint8_t)s_code;
}

}  // namespace

cudaError_t launch_store_nvfp4(const uint16_t* src, const int64_t* slot_mapping, int64_t num_tokens,
                               uint8_t* payload, uint8_t* scale, int64_t num_rows,
                               cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  const int64_t threads = num_tokens * 8;
  const int64_t blocks = (threads + 255) / 256;
  store_nvfp4_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, slot_mapping, num_tokens, payload,
                                                         scale, num_rows);
  return cudaGetLastError();
}

}  // namespace idx

// Inline-PTX building blocks for the 5th-generation tensor cores of sm_103a:
// tensor-memory (TMEM) allocation, tcgen05.mma with shared-memory operand
// descriptors, completion through tcgen05.commit on an mbarrier, and
// tcgen05.ld of the fp32 accumulator back into registers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace idx {

// ---------------------------------------------------------------------------
// TMEM allocation (one full warp executes each of these)
// ---------------------------------------------------------------------------
// Allocate `ncols` columns (a power of two >= 32) of this SM's tensor memory;
// the TMEM address of the allocation is written to shared memory at dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Ordering of tcgen05 operations across a thread synchronisation (mbarrier or
// bar.sync): "before" on the signalling side, "after" on the waiting side.
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Operand descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor of a K-major operand stored with the 128-byte
// swizzle: rows of 128 bytes, the 16-byte chunks of row r XOR-permuted by r % 8,
// 8-row atoms (1024 B) stacked contiguously.  This is the layout a TMA tile load
// with CU_TENSOR_MAP_SWIZZLE_128B writes for a box 128 bytes wide.
//   bits  0-13  start address >> 4        bits 16-29  leading byte offset >> 4
//   bits 32-45  stride byte offset >> 4   bits 46-47  descriptor version (1)
//   bits 49-51  base offset (0: atoms are 1024-byte aligned)
//   bits 61-63  layout (2: 128-byte swizzle)
// Stepping K inside an atom moves the start address by the step's byte width.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;    // unused by swizzled K-major layouts
  d |= static_cast<uint64_t>(1024u >> 4) << 32;  // next 8-row atom
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor, fp32 accumulate, both operands K-major.
//   bits 4-5 D format (1: f32)      bits 7-9 A format     bits 10-12 B format
//   bit 15/16 A/B major (0: K)      bits 17-22 N >> 3     bits 24-28 M >> 4
// A/B format: kind::f16 -> 0 f16, 1 bf16; kind::f8f6f4 -> 0 e4m3.
constexpr uint32_t instr_desc(uint32_t ab_format, int M, int N) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// MMA (issued by one thread) and completion
// ---------------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T, 16-bit inputs (K = 16 per instruction).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with 8-bit float inputs (K = 32 per instruction).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Whole-warp forms: every lane of a converged warp executes them with the same
// (warp-uniform) operands and one lane, chosen by elect.sync (the same lane each
// time in a converged warp), issues.  Issued this way the operands stay in
// uniform registers; measured on sm_103a, an M = N = 128 bf16 MMA then issues
// every ~87 cycles against ~100-120 from a single thread inside a lane branch,
// and M = 128, N = 256 reaches the tensor cores' full rate.
__device__ __forceinline__ void tc_mma_f16_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_mma_f8_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Commit from the lane that issued the warp's MMAs (the same election).
__device__ __forceinline__ void tc_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

// Arrive (once) on the mbarrier when every tcgen05.mma this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// ---------------------------------------------------------------------------
// TMEM -> registers
// ---------------------------------------------------------------------------
// Lane (laneid) of the warp's 32-lane slice, 32 consecutive 32-bit columns.
__device__ __forceinline__ void tc_ld_32cols(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace idx

// tcgen05.cuh -- inline-PTX wrappers for the 5th-generation tensor cores of
// sm_100-class parts (tcgen05): tensor-memory allocation, MMA issue and
// completion, tensor-memory loads, and the shared-memory matrix descriptor.
#pragma once

#include <stdint.h>

namespace sgemm_gb300 {
namespace tc {

// ---- tensor memory (TMEM) allocation: one full warp executes these -------
// Allocates `ncols` columns (a power of two >= 32) of all 128 lanes; the
// TMEM address is written to shared memory at `dst_smem`. CG = 2 (the pair
// form of the MMA, whose accumulator spans the TMEM of two CTAs): one warp
// of each CTA of the pair executes it, and both get the same columns. Every
// tcgen05 instruction of a kernel uses the same CG.
template <int CG = 1>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}
template <int CG = 1>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (CG == 1)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int CG = 1>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// ---- ordering of tensor-core work around thread synchronisation ----------
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- MMA: D[tmem] (+)= A[smem] * B[smem], TF32 inputs, FP32 accumulate ---
// a_desc / b_desc: shared-memory matrix descriptors; idesc: instruction
// descriptor; accumulate == 0 overwrites D.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with A read from tensor memory (`a_tmem`: lane = row of A, one
// 32-bit column per TF32 value along K) and B from shared memory.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives (once) on the mbarrier when every MMA this thread issued before
// has completed.
__device__ __forceinline__ void commit(uint32_t mbar_smem) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          mbar_smem)
      : "memory");
}

// ---- the pair form (cta_group::2) ------------------------------------------
// D[tmem] (+)= A * B for an M = 256 tile spread over a CTA pair, issued by one
// thread of the even CTA: A rows 0-127 come from that CTA's shared memory and
// rows 128-255 from the odd CTA's, at the same offset (a_desc); B's N columns
// likewise in two halves (b_desc); D rows 0-127 land in the even CTA's TMEM,
// rows 128-255 in the odd CTA's, at the same TMEM address.
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Commit of the pair form: arrives on the mbarrier at offset `mbar_smem` of
// every CTA in `cta_mask` (or of this CTA only) when the MMAs issued so far
// have completed.
__device__ __forceinline__ void commit_pair_multicast(uint32_t mbar_smem, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(mbar_smem),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void commit_pair(uint32_t mbar_smem) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          mbar_smem)
      : "memory");
}

// ---- TMEM -> registers: 32 lanes x 32 bits, 16 consecutive columns -------
// Lane i of the warp receives row (lane base + i) of the addressed block.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- registers -> TMEM: 32 lanes x 32 bits, 32 consecutive columns --------
// Lane i of the warp writes row (lane base + i) of the addressed block.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Waits until this thread's tcgen05.st writes have completed.
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- shared-memory matrix descriptor ---------------------------------------
// For a K-major operand tile written by TMA with a ROW_BYTES-byte swizzle
// (128: 32 TF32 values along K per row; 64: 16 values; 32: 8): 8-row swizzle atoms
// of 8 * ROW_BYTES bytes laid out one after another along M (or N). Fields:
// start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29, unused for
// these layouts), stride byte offset >> 4 (32-45: one atom between 8-row
// groups), descriptor version 1 (46-47), base offset 0 (49-51, the tile
// starts on an atom boundary), layout type (61-63: 2 = 128-byte swizzle,
// 4 = 64-byte swizzle, 6 = 32-byte swizzle). Moving along K inside a row is done by advancing the
// start address (32 bytes per 8-wide k-step).
template <int ROW_BYTES>
__device__ __forceinline__ uint64_t smem_desc_k_swizzled(uint32_t smem_addr) {
  static_assert(ROW_BYTES == 128 || ROW_BYTES == 64 || ROW_BYTES == 32, "swizzle width");
  constexpr uint64_t kLayout = ROW_BYTES == 128 ? 2u : (ROW_BYTES == 64 ? 4u : 6u);
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)(1u) << 16;                  // leading byte offset (16 B), ignored here
  d |= (uint64_t)(((8u * ROW_BYTES) >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;                    // descriptor version
  d |= kLayout << 61;
  return d;
}

// Instruction descriptor of kind::tf32 with FP32 accumulation, both operands
// K-major: D format F32 (bits 4-5 = 1), A and B format TF32 (bits 7-9 and
// 10-12 = 2), no negation or transposition, N >> 3 (bits 17-22), M >> 4
// (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

}  // namespace tc
}  // namespace sgemm_gb300

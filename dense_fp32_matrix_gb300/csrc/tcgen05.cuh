// Inline-PTX wrappers for the sm_100-family tensor-core instructions
// (tcgen05): tensor-memory allocation, single-thread MMA issue with
// shared-memory operand descriptors, completion tracking on mbarriers, and
// tensor-memory loads. Bit layouts follow the public PTX ISA descriptions of
// the shared-memory matrix descriptor and the instruction descriptor.
#pragma once

#include <stdint.h>

namespace dfm {
namespace tc {

// ------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor (64 bits):
//   [0,14)  start address >> 4        [16,30) leading-dimension byte offset >> 4
//   [32,46) stride-dimension byte offset >> 4
//   [46,48) descriptor version (1)    [49,52) base offset   [52] LBO mode
//   [61,64) layout: 0 none, 2 128-byte swizzle, 4 64-byte, 6 32-byte
constexpr uint64_t kLayoutSwizzle128 = 2;

__device__ __forceinline__ uint64_t smem_desc(uint32_t smem_addr, uint32_t lbo,
                                              uint32_t sbo, uint64_t layout) {
  uint64_t d = 0;
  d |= uint64_t((smem_addr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= layout << 61;
  return d;
}

// Instruction descriptor of kind::tf32 (32 bits):
//   [4,6) D format (1 = f32)  [7,10) A format (2 = tf32)  [10,13) B format
//   [15] A major (0 = K-major, 1 = MN-major)  [16] B major
//   [17,23) N >> 3   [24,29) M >> 4
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool a_mn_major,
                                                  bool b_mn_major) {
  return (1u << 4) | (2u << 7) | (2u << 10) |
         (uint32_t(a_mn_major ? 1 : 0) << 15) |
         (uint32_t(b_mn_major ? 1 : 0) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// ------------------------------------------------------------ allocation

// Allocate `cols` tensor-memory columns (power of two, >= 32); the address is
// written to shared memory at dst. Whole warp, converged.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t cols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          dst_smem),
      "r"(cols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile(
      "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
      "r"(cols)
      : "memory");
}

// Pair (cta_group::2) variants: one warp in each CTA of the 2-CTA cluster
// allocates / frees the same columns in both tensor memories.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem,
                                                uint32_t cols) {
  asm volatile(
      "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          dst_smem),
      "r"(cols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr,
                                                  uint32_t cols) {
  asm volatile(
      "tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
      "r"(cols)
      : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------ MMA

// D (tensor memory) = A * B (+ D when accumulate != 0); A and B from shared
// memory descriptors. Issued by a single thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc,
                                        uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair MMA issued by the even CTA of a 2-CTA cluster: M = 256 rows, A rows
// 0..127 from this CTA's shared memory and 128..255 from the peer's at the
// same offsets, B columns split the same way; D lands in both tensor
// memories (each CTA holds its 128 rows x N).
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc,
                                             uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair form of commit: arrive once on the mbarrier at this shared::cluster
// address (this CTA's or the peer's) when the pair's tcgen05 operations
// issued so far by this thread have completed.
__device__ __forceinline__ void commit_pair(uint32_t cluster_mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(cluster_mbar)
      : "memory");
}

// Pair MMA with A from tensor memory: A rows 0..127 in this CTA's lanes
// 0..127 and rows 128..255 in the peer's, one 32-bit column per k (TF32),
// at column a_tmem; B from shared memory as for mma_tf32_pair.
__device__ __forceinline__ void mma_tf32_pair_tmem_a(uint32_t d_tmem,
                                                    uint32_t a_tmem,
                                                    uint64_t b_desc,
                                                    uint32_t idesc,
                                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on the mbarrier when all tcgen05 operations issued so far by
// this thread have completed.
__device__ __forceinline__ void commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(mbar)
      : "memory");
}

// ------------------------------------------------------------ loads

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (taddr.lane + t), columns taddr.col .. taddr.col + 31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr,
                                                   uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]),
        "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 16 consecutive 32-bit columns from registers: thread t writes
// lane (taddr.lane + t), columns taddr.col .. taddr.col + 15.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr,
                                                   const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
      "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
      "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Wait until this thread's tensor-memory stores have completed.
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace tc
}  // namespace dfm

// rsc_tc.cuh -- 5th-generation tensor core (tcgen05) building blocks for sm_103a:
// tensor-memory allocation, shared-memory operand descriptors, instruction descriptors,
// bf16 MMA with fp32 accumulation in tensor memory, commit to an mbarrier, and loads of
// accumulator columns back to registers.  All inline PTX; one CTA (cta_group::1).
//
// Operand layout used throughout (the "no swizzle, K-major" canonical layout): an operand
// of R rows (M or N) by KD contraction elements (bf16) is stored as 8x8 core matrices of
// 128 contiguous bytes (8 rows of 16 bytes).  Core matrix (row/8, k/8) sits at byte
//     ((row/8) * (KD/8) + k/8) * 128
// so core matrices adjacent along K are 128 bytes apart (leading byte offset) and 8-row
// groups are KD*16 bytes apart (stride byte offset).  One MMA consumes K = 16 (two core
// matrices along K); the next K slice starts 256 bytes further.
#pragma once

#include "rsc_common.cuh"

namespace rsc {
namespace tc {

// Byte offset of element (row, k) in a K-major no-swizzle operand with KD columns.
__device__ __forceinline__ uint32_t kmajor_offset(int row, int k, int KD) {
  return (uint32_t)((((row >> 3) * (KD >> 3) + (k >> 3)) << 7) + ((row & 7) << 4) + ((k & 7) << 1));
}

// Shared-memory matrix descriptor: start address, leading / stride byte offsets (all
// >> 4), descriptor version 1, base offset 0, layout SWIZZLE_NONE.
__device__ __forceinline__ uint64_t smem_desc(const void *smem, uint32_t lbo, uint32_t sbo) {
  const uint64_t a = (uint64_t)((smem_u32(smem) & 0x3FFFF) >> 4);
  return a | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) | ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) |
         (1ull << 46);
}
// Descriptor of the K slice [16*ks, 16*ks + 16) of a K-major operand with KD columns.
__device__ __forceinline__ uint64_t kmajor_desc(const void *base, int KD, int ks) {
  return smem_desc(static_cast<const char *>(base) + ks * 256, 128, (uint32_t)KD * 16);
}

// MN-major no-swizzle operand (used for B): element (n, kd) of an N x KD operand at
//     ((kd/8) * (N/8) + n/8) * 128 + (kd%8) * 16 + (n%8) * 2
// i.e. core matrices of 8 KD-rows of 16 bytes (8 consecutive n); core matrices adjacent
// along N are 128 bytes apart, along KD N*16 bytes apart.  A thread holding one kd and
// eight consecutive n writes one 16-byte vector.  Measured on GB300: for this form the
// leading byte offset is the stride along KD and the stride byte offset the stride
// along N (the assignment with the two swapped reads outside the operand).
__device__ __forceinline__ uint32_t mnmajor_offset(int n, int kd, int N) {
  return (uint32_t)((((kd >> 3) * (N >> 3) + (n >> 3)) << 7) + ((kd & 7) << 4) + ((n & 7) << 1));
}
__device__ __forceinline__ uint64_t mnmajor_desc(const void *base, int N, int ks) {
  return smem_desc(static_cast<const char *>(base) + ks * 2 * N * 16, (uint32_t)N * 16, 128);
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major, shape M x N.
template <int M, int N>
__host__ __device__ constexpr uint32_t idesc_bf16() {
  static_assert(M == 64 || M == 128, "M");
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "N");
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// The same with the B operand MN-major (transpose-B bit).
template <int M, int N>
__host__ __device__ constexpr uint32_t idesc_bf16_bmn() {
  return idesc_bf16<M, N>() | (1u << 16);
}

// ---------------------------------------------------------------- tensor memory
// Allocation and deallocation are warp-wide (.sync.aligned): call from one full warp.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
               ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n"
               ::"r"(taddr), "r"(ncols) : "memory");
}

// ---------------------------------------------------------------- MMA
// D[M x N] (+)= A[M x 16] * B[N x 16]^T on one K slice; issued by a single thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// Arrive once on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
               ::"r"(smem_u32(bar)) : "memory");
}

// Ordering of tensor-core work against thread barriers, and of generic shared-memory
// writes (st.shared) against the tensor core's (async-proxy) operand reads.
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_smem_to_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ---------------------------------------------------------------- accumulator loads
// 32 lanes x 16 consecutive 32-bit columns from tensor memory into 16 registers per
// thread (thread i of the warp gets lane base+i).  The warp must address its own lane
// quadrant (warp % 4).  The wait for the load is inside the same asm statement, so the
// compiler cannot move a use of the registers ahead of it.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// The same for 32 consecutive columns (one instruction, one wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// D[M x N] (+)= A[M x 16] * B[N x 16]^T with A in tensor memory: lane m holds row m, 32-bit
// column c the bf16 pair of k = 2c (low half) and 2c + 1 (high half); the K slice starting
// at k = 16 s is at column a_tmem + 8 s.  Measured on GB300 against torch (M=128, N = 32 and 64).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns from registers into tensor memory (thread i of the
// warp writes lane base+i; the warp must address its own lane quadrant).  Complete (for this
// thread) after tmem_wait_st.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}
// Descriptor `d` moved `bytes` further into shared memory (the start address field is
// the low 14 bits of address / 16; callers stay inside one operand, so it cannot carry).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }
// Tensor-memory address of (lane, column).
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, int lane, int col) {
  return base + ((uint32_t)lane << 16) + (uint32_t)col;
}

}  // namespace tc
}  // namespace rsc

// rsc_common.cuh -- device helpers shared by the sm_103a kernels of librsc.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rsc.h"

namespace rsc {

typedef __nv_bfloat16 bf16;

// L2 normalisation epsilon: x / sqrt(sum x^2 + eps).  The pages print an epsilon in the
// normalised-key formula of the ReplaySSM replay steps without a value; 1e-6 is used.
constexpr float kNormEps = 1e-6f;

// Everything a kernel needs to address one layer of the pool.
struct PoolView {
  void *ssm;        // [layers][P+1][H][V][K]
  void *conv;       // [layers][P+1][3][D]
  int32_t *err;     // device error word
  int P;            // usable slots; rows = P+1
  int H, K, V, D;
};

__device__ __forceinline__ void flag_error(int32_t *err, int bit) { atomicOr(err, bit); }

// ------------------------------------------------------------------ 16-byte vectors
// A 16-byte vector holds 4 fp32 or 8 bf16 values; loads widen to fp32.

template <typename T> struct VecTraits;
template <> struct VecTraits<float> { static constexpr int N = 4; };
template <> struct VecTraits<bf16> { static constexpr int N = 8; };

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void unpack16(const uint4 &v, float (&x)[4]) {
  x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
  x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack16(const uint4 &v, float (&x)[8]) {
  x[0] = bf16lo(v.x); x[1] = bf16hi(v.x); x[2] = bf16lo(v.y); x[3] = bf16hi(v.y);
  x[4] = bf16lo(v.z); x[5] = bf16hi(v.z); x[6] = bf16lo(v.w); x[7] = bf16hi(v.w);
}
__device__ __forceinline__ uint4 pack16(const float (&x)[4]) {
  return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                    __float_as_uint(x[3]));
}
__device__ __forceinline__ uint4 pack16(const float (&x)[8]) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                    pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
}

// Streaming (evict-first) 16-byte load / store.
__device__ __forceinline__ uint4 ld16_stream(const void *p) {
  return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st16_stream(void *p, const uint4 &v) {
  __stcs(reinterpret_cast<uint4 *>(p), v);
}
// Ask for the 128-byte line holding p in L2, without a register or a wait.
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}
__device__ __forceinline__ uint4 ld16(const void *p) {
  return *reinterpret_cast<const uint4 *>(p);
}
__device__ __forceinline__ void st16(void *p, const uint4 &v) {
  *reinterpret_cast<uint4 *>(p) = v;
}

// ------------------------------------------------------------------ scalars

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// ------------------------------------------------------------------ reductions

template <int WIDTH>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum three values over a block of NW warps; every thread gets the totals.
// `red` is shared scratch of at least 3*NW floats; ends with a __syncthreads.
template <int NW>
__device__ __forceinline__ void block3_sum(float &a, float &b, float &c, float *red) {
  a = group_sum<32>(a); b = group_sum<32>(b); c = group_sum<32>(c);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { red[warp] = a; red[NW + warp] = b; red[2 * NW + warp] = c; }
  __syncthreads();
  a = 0.f; b = 0.f; c = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) { a += red[w]; b += red[NW + w]; c += red[2 * NW + w]; }
}
__device__ __forceinline__ void block3_sum_128(float &a, float &b, float &c, float *red) {
  block3_sum<4>(a, b, c, red);
}

// ------------------------------------------------------------------ bulk rows
// Bytes of one streaming-copy chunk: 128 threads x 4 vectors x 16 bytes.
constexpr int kCopyChunk = 128 * 4 * 16;

// Copy bytes [off, min(off + kCopyChunk, bytes)) of a row; 16-byte vectors, all four
// loads of a thread in flight before its stores.  bytes must be a multiple of 16.
__device__ __forceinline__ void copy_chunk(char *dst, const char *src, size_t bytes, size_t off) {
  uint4 v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const size_t o = off + ((size_t)u * 128 + threadIdx.x) * 16;
    if (o < bytes) v[u] = ld16_stream(src + o);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const size_t o = off + ((size_t)u * 128 + threadIdx.x) * 16;
    if (o < bytes) st16_stream(dst + o, v[u]);
  }
}

// ------------------------------------------------------------------ async copies
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// ------------------------------------------------------------------ TMA bulk + mbarrier
// One-shot bulk copies global -> shared completed on an mbarrier (transaction count).
// Every wait is bounded: a wait that runs out sets RSC_DEVERR_TIMEOUT in the pool's
// error word and the caller skips its work instead of spinning forever.

#ifndef RSC_MBAR_SPIN_LIMIT
#define RSC_MBAR_SPIN_LIMIT (1u << 22)
#endif
constexpr uint32_t kMbarSpinLimit = RSC_MBAR_SPIN_LIMIT;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n"
               " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
               " selp.u32 %0, 1, 0, p;\n}\n"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(phase) : "memory");
  return ok != 0;
}
// Bounded wait for phase `phase` of `bar`; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t phase) {
  for (uint32_t i = 0; i < kMbarSpinLimit; ++i)
    if (mbar_try_wait(bar, phase)) return true;
  return false;
}
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) into this CTA's
// shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void *smem, const void *gmem, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(smem_u32(smem)), "l"(gmem), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------------ dependent launch
// Wait until the previous grid on the stream has completed and its writes are visible
// (no-op when the grid was not launched as a programmatic dependent), then allow the next
// grid to be scheduled early.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ------------------------------------------------------------------ clusters

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

}  // namespace rsc

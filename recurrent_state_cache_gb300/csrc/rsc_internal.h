// rsc_internal.h -- launchers behind the C ABI (host side).  Arguments have already
// been validated by rsc_api.cu when these are called.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "rsc_common.cuh"

namespace rsc {

struct LayerArgs {
  PoolView pv;
  int st, io, gate;   // state dtype, conv/io dtype, gate kind
  int layer;
};

// Per-call extras of the decode kernel (all null: the plain step).
struct DecodeExtras {
  const float *A_log = nullptr, *dt_bias = nullptr;  // fused gating: A_log [H], dt_bias [H][K] / [H]
  const uint8_t *track_mask = nullptr;               // tracking: [B]
  const int32_t *track_slots = nullptr;              // [B]
  bool overlap = false;  // programmatic dependent launch; the slot's rows read before the wait
};
int launch_decode(const LayerArgs &a, const int32_t *slots, int B, const void *qkv,
                  const float *conv_w, const float *g, const float *beta, void *out,
                  const DecodeExtras &ex, cudaStream_t s);

int launch_spec_verify(const LayerArgs &a, const int32_t *slots, int B, int T, int L,
                       void *spec_ssm, void *spec_conv, const void *qkv,
                       const float *conv_w, const float *g, const float *beta, void *out,
                       cudaStream_t s);

int launch_spec_commit(const LayerArgs &a, const int32_t *slots, int B, int T, int L,
                       const void *spec_ssm, const void *spec_conv, const int32_t *accept,
                       cudaStream_t s);

// ReplaySSM rings of the pool ([layer][P+1][H][depth][n]); see rsc_replay_rings.
struct RingView {
  void *d, *k, *rawv, *rawk;  // state dtype
  float *g, *beta;
  int depth;
};
int launch_replay_verify(const LayerArgs &a, const RingView &rv, const int32_t *slots,
                         const int32_t *pos, int B, int T, void *spec_conv, const void *qkv,
                         const float *conv_w, const float *g, const float *beta, void *out,
                         cudaStream_t s);
int launch_replay_commit(const LayerArgs &a, const RingView &rv, const int32_t *slots,
                         const int32_t *pos, int B, int T, const void *spec_conv,
                         const int32_t *accept, cudaStream_t s);

int launch_slot_copy(const PoolView &pv, int st, int io, int layer0, int nlayers,
                     const int32_t *src, const int32_t *dst, const uint8_t *mask, int n,
                     cudaStream_t s);

size_t prefill_workspace_bytes(const PoolView &pv, int st, int N, int T);

// The slot's window becomes the last three raw inputs of each sequence.
int launch_prefill_window(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N,
                          int T, const uint8_t *has_init, const void *qkv, cudaStream_t s);
// Recurrent form of every pool the tensor-core form does not take: the recurrence eight tokens
// at a time in closed form, fp32.
size_t prefill_blocked_bytes(const PoolView &pv, int N, int T);
int launch_prefill_blocked(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N,
                           int T, const uint8_t *has_init, const void *qkv,
                           const float *conv_w, const float *g, const float *beta, void *out,
                           void *ws, cudaStream_t s);
// Tensor-core chunkwise path (bf16 state, K = 128).
size_t prefill_tc_chunk_capacity(int N, int T);
size_t prefill_tc_block_bytes();
int launch_prefill_tc(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N, int T,
                      const uint8_t *has_init, const void *qkv, const float *conv_w,
                      const float *g, const float *beta, void *out, int32_t *chunk_base,
                      char *blocks, cudaStream_t s);

int launch_prefill(const LayerArgs &a, const int32_t *slots, const int32_t *cu_seqlens,
                   int N, int T, const uint8_t *has_init, const void *qkv,
                   const float *conv_w, const float *g, const float *beta, void *out,
                   void *ws, size_t ws_bytes, cudaStream_t s);

// One-time set-up per device (kernel attributes such as the dynamic shared-memory limit are
// per device): once_per_device(flag, setup) runs setup() with the current device until it
// has succeeded once on that device.  Thread-safe; the common path is one atomic load.
constexpr int kMaxDevices = 64;
struct PerDeviceFlag {
  std::atomic<uint64_t> done{0};
  std::mutex mu;
};
template <typename F>
int once_per_device(PerDeviceFlag &f, F setup) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return RSC_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return RSC_ERANGE;
  const uint64_t bit = 1ull << dev;
  if (f.done.load(std::memory_order_acquire) & bit) return RSC_OK;
  std::lock_guard<std::mutex> lock(f.mu);
  if (f.done.load(std::memory_order_relaxed) & bit) return RSC_OK;
  const int rc = setup();
  if (rc == RSC_OK) f.done.fetch_or(bit, std::memory_order_release);
  return rc;
}

inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? RSC_OK : RSC_ECUDA;
}

// Launch with programmatic stream serialization: the grid may be scheduled while the
// previous kernel on the stream drains.  Kernels launched this way call grid_dep_wait()
// before they touch anything that kernel may write, which waits for it to complete and its
// writes to be visible; what they read before the wait is the caller's contract.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
               Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) == cudaSuccess ? RSC_OK
                                                                                      : RSC_ECUDA;
}

// Compile-time dispatch over (state dtype, io dtype, K, V, gate) onto L<ST,IO,K,V,GATE>::run.
template <template <typename, typename, int, int, int> class L, typename ST, typename IO,
          int K, int V, typename... A>
int dispatch_gate(int gate, A... a) {
  return gate == RSC_GATE_KDA ? L<ST, IO, K, V, RSC_GATE_KDA>::run(a...)
                              : L<ST, IO, K, V, RSC_GATE_GDN>::run(a...);
}
template <template <typename, typename, int, int, int> class L, typename ST, typename IO,
          int K, typename... A>
int dispatch_v(int V, int gate, A... a) {
  if (V == 64) return dispatch_gate<L, ST, IO, K, 64>(gate, a...);
  if (V == 128) return dispatch_gate<L, ST, IO, K, 128>(gate, a...);
  return RSC_EDTYPE;
}
template <template <typename, typename, int, int, int> class L, typename ST, typename IO,
          typename... A>
int dispatch_k(int K, int V, int gate, A... a) {
  if (K == 64) return dispatch_v<L, ST, IO, 64>(V, gate, a...);
  if (K == 128) return dispatch_v<L, ST, IO, 128>(V, gate, a...);
  return RSC_EDTYPE;
}
template <template <typename, typename, int, int, int> class L, typename... A>
int dispatch_all(int st, int io, int K, int V, int gate, A... a) {
  if (st == RSC_F32) {
    return io == RSC_F32 ? dispatch_k<L, float, float>(K, V, gate, a...)
                         : dispatch_k<L, float, bf16>(K, V, gate, a...);
  }
  return io == RSC_F32 ? dispatch_k<L, bf16, float>(K, V, gate, a...)
                       : dispatch_k<L, bf16, bf16>(K, V, gate, a...);
}

}  // namespace rsc

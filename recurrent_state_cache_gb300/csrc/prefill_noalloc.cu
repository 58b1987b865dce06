// prefill_noalloc.cu -- kda_prefill_chunk for callers that cannot allocate device
// memory: the workspace is a file-scope device array instead of caller memory.
//
// Who needs this: a caller that gives every byte of HBM to its own pools at start-up
// (a serving engine's state and KV pools) has no memory left to hand over as a
// workspace, and a host path that cannot take cudaMalloc's implicit device
// synchronisation cannot allocate one per call.  This entry point runs the very same
// prefill launches as kda_prefill_chunk, pointed at the static array.
//
// The array is shared by every call on a device and keeps the last call's contents.
// Nothing needs clearing: the prefill writes every workspace byte it reads earlier in
// the same call.  Two calls that overlap on the GPU race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "rsc_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Device-side scratch; host code only ever sees its per-device address below.
__device__ __align__(256) unsigned char g_prefill_scratch[RSC_PREFILL_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Address of the scratch array on the current device, looked up once per device.
int scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return RSC_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return RSC_ERANGE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || p == nullptr)
      return RSC_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return RSC_OK;
}

}  // namespace

extern "C" int kda_prefill_chunk_noalloc(rsc_pool *pool, int layer, const int32_t *slot_ids,
                                         const int32_t *cu_seqlens, int num_seqs,
                                         int total_tokens, const uint8_t *has_initial_state,
                                         const void *qkv, const float *conv_w, const float *g,
                                         const float *beta, void *out, void *stream) {
  size_t need = 0;
  int rc = kda_prefill_workspace_size(pool, num_seqs, total_tokens, &need);
  if (rc != RSC_OK) return rc;
  if (need > RSC_PREFILL_STATIC_SCRATCH_BYTES) return RSC_ENOSPACE;
  void *scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != RSC_OK) return rc;
  return kda_prefill_chunk(pool, layer, slot_ids, cu_seqlens, num_seqs, total_tokens,
                           has_initial_state, qkv, conv_w, g, beta, out, scratch,
                           RSC_PREFILL_STATIC_SCRATCH_BYTES, stream);
}

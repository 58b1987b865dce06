// prefill.cu -- prefill of packed sequences over the slot pool: which form a pool takes, its
// workspace, and the window update of the recurrent form.
//
// Source: "SGLang之KV Cache内存池机制" §8.5 forward_extend: each sequence starts from the
// state its slot holds (or from zero), runs the recurrence over its tokens and leaves
// the final state (and conv window) in the slot.  Sequences are packed along tokens
// and delimited by cu_seqlens.
//
// bf16-state pools with head_k 128 take the chunkwise tensor-core form (prefill_tc.cu, which
// also writes the windows); every other pool takes the recurrence eight tokens at a time in
// closed form (prefill_blocked.cu), whose last launch is the window kernel below: grid
// (channel block, sequence), the slot's window becomes the last three raw inputs of the
// sequence (fewer than three tokens shift the old window).
#include "rsc_internal.h"

namespace rsc {

template <typename IO>
__global__ void __launch_bounds__(128)
prefill_window_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                      const int32_t *__restrict__ cu, int T,
                      const uint8_t *__restrict__ has_init, const IO *__restrict__ qkv) {
  const int n = blockIdx.y, c = blockIdx.x * 128 + threadIdx.x;
  const int D = pv.D;
  if (c >= D) return;
  const int start = cu[n], end = cu[n + 1];
  const int slot = slots[n];
  if (start < 0 || end < start || end > T || slot < 0 || slot > pv.P) return;  // flagged by the recurrence
  const bool init = has_init == nullptr || has_init[n] != 0;
  IO *W = reinterpret_cast<IO *>(pv.conv) + ((size_t)layer * (pv.P + 1) + slot) * 3 * (size_t)D;
  const int len = end - start;
  IO old[3], nw[3];
#pragma unroll
  for (int m = 0; m < 3; ++m) old[m] = init ? W[(size_t)m * D + c] : from_f32<IO>(0.f);
#pragma unroll
  for (int m = 0; m < 3; ++m) {
    const int pp = len - 3 + m;
    nw[m] = pp >= 0 ? qkv[(size_t)(start + pp) * D + c] : old[3 + pp];
  }
#pragma unroll
  for (int m = 0; m < 3; ++m) W[(size_t)m * D + c] = nw[m];
}

int launch_prefill_window(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N,
                          int T, const uint8_t *has_init, const void *qkv, cudaStream_t s) {
  const dim3 grid((a.pv.D + 127) / 128, N);
  if (a.io == RSC_BF16)
    prefill_window_kernel<bf16><<<grid, 128, 0, s>>>(a.pv, a.layer, slots, cu, T, has_init,
                                                     static_cast<const bf16 *>(qkv));
  else
    prefill_window_kernel<float><<<grid, 128, 0, s>>>(a.pv, a.layer, slots, cu, T, has_init,
                                                      static_cast<const float *>(qkv));
  return launch_status();
}

static bool use_tc(const PoolView &pv, int st) { return st == RSC_BF16 && pv.K == 128; }
static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t prefill_workspace_bytes(const PoolView &pv, int st, int N, int T) {
  if (use_tc(pv, st))
    return align256((size_t)(N + 1) * 4) +
           prefill_tc_chunk_capacity(N, T) * (size_t)pv.H * prefill_tc_block_bytes();
  return prefill_blocked_bytes(pv, N, T);
}

int launch_prefill(const LayerArgs &a, const int32_t *slots, const int32_t *cu_seqlens,
                   int N, int T, const uint8_t *has_init, const void *qkv,
                   const float *conv_w, const float *g, const float *beta, void *out,
                   void *ws, size_t ws_bytes, cudaStream_t s) {
  if (ws_bytes < prefill_workspace_bytes(a.pv, a.st, N, T)) return RSC_ENOSPACE;
  if (!use_tc(a.pv, a.st))
    return launch_prefill_blocked(a, slots, cu_seqlens, N, T, has_init, qkv, conv_w, g, beta,
                                  out, ws, s);
  int32_t *chunk_base = static_cast<int32_t *>(ws);
  char *blocks = static_cast<char *>(ws) + align256((size_t)(N + 1) * 4);
  // the tensor-core path writes the windows in its state pass
  return launch_prefill_tc(a, slots, cu_seqlens, N, T, has_init, qkv, conv_w, g, beta, out,
                           chunk_base, blocks, s);
}

}  // namespace rsc

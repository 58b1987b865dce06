// slot_copy.cu -- masked copy of whole slot rows (state and window) between slots.
//
// Source: "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理", mamba track section:
// when a request's track mask is set, its active slot's conv and ssm state are copied
// into a tracking slot; a prefix-cache fork copies a state the same way.
//
// A pure streaming kernel: grid (chunk, pair, layer), each CTA moves one 8 KB chunk of
// one row with 16-byte vectors (four loads in flight per thread before the stores).
// Rows are contiguous in the pool, so the copy is two contiguous byte ranges per
// (pair, layer): one launch for the state rows, one for the window rows.
#include "rsc_internal.h"

namespace rsc {

__global__ void __launch_bounds__(128)
ssm_slot_copy_kernel(char *__restrict__ base, size_t row_bytes, int rows_per_layer,
                     int layer0, int P, int32_t *err, int flag_errors,
                     const int32_t *__restrict__ src, const int32_t *__restrict__ dst,
                     const uint8_t *__restrict__ mask) {
  const int i = blockIdx.y;
  if (mask && !mask[i]) return;
  const int s = src[i], d = dst[i];
  if (s < 0 || s > P || d < 0 || d > P) {
    if (flag_errors && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0)
      flag_error(err, RSC_DEVERR_SLOT);
    return;
  }
  const size_t l = (size_t)layer0 + blockIdx.z;
  const char *from = base + (l * rows_per_layer + s) * row_bytes;
  char *to = base + (l * rows_per_layer + d) * row_bytes;
  copy_chunk(to, from, row_bytes, (size_t)blockIdx.x * kCopyChunk);
}

int launch_slot_copy(const PoolView &pv, int st, int io, int layer0, int nlayers,
                     const int32_t *src, const int32_t *dst, const uint8_t *mask, int n,
                     cudaStream_t s) {
  const size_t sb = (size_t)pv.H * pv.V * pv.K * (st == RSC_F32 ? 4 : 2);
  const size_t cb = (size_t)3 * pv.D * (io == RSC_F32 ? 4 : 2);
  dim3 gs((unsigned)((sb + kCopyChunk - 1) / kCopyChunk), n, nlayers);
  ssm_slot_copy_kernel<<<gs, 128, 0, s>>>(static_cast<char *>(pv.ssm), sb, pv.P + 1, layer0,
                                          pv.P, pv.err, 1, src, dst, mask);
  if (launch_status() != RSC_OK) return RSC_ECUDA;
  dim3 gc((unsigned)((cb + kCopyChunk - 1) / kCopyChunk), n, nlayers);
  ssm_slot_copy_kernel<<<gc, 128, 0, s>>>(static_cast<char *>(pv.conv), cb, pv.P + 1, layer0,
                                          pv.P, pv.err, 0, src, dst, mask);
  return launch_status();
}

}  // namespace rsc

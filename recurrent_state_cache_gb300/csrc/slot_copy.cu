// slot_copy.cu -- masked copy of whole slot rows (state and window) between slots.
//
// Source: "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理", mamba track section:
// when a request's track mask is set, its active slot's conv and ssm state are copied
// into a tracking slot; a prefix-cache fork copies a state the same way.
//
// A pure streaming kernel: grid (chunk, pair, layer), each CTA moves one 8 KB chunk of the
// pair's state row and, when the window row is that long, the same chunk of the window row,
// with 16-byte vectors (four loads in flight per thread before the stores).  Rows are
// contiguous in the pool, so the copy is two contiguous byte ranges per (pair, layer), in one
// launch.
#include "rsc_internal.h"

namespace rsc {

__global__ void __launch_bounds__(128)
ssm_slot_copy_kernel(char *__restrict__ ssm, size_t ssm_row_bytes, char *__restrict__ conv,
                     size_t conv_row_bytes, int rows_per_layer, int layer0, int P, int32_t *err,
                     const int32_t *__restrict__ src, const int32_t *__restrict__ dst,
                     const uint8_t *__restrict__ mask) {
  const int i = blockIdx.y;
  if (mask && !mask[i]) return;
  const int s = src[i], d = dst[i];
  if (s < 0 || s > P || d < 0 || d > P) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) flag_error(err, RSC_DEVERR_SLOT);
    return;
  }
  const size_t l = (size_t)layer0 + blockIdx.z;
  const size_t off = (size_t)blockIdx.x * kCopyChunk;
  if (off < ssm_row_bytes)
    copy_chunk(ssm + (l * rows_per_layer + d) * ssm_row_bytes,
               ssm + (l * rows_per_layer + s) * ssm_row_bytes, ssm_row_bytes, off);
  if (off < conv_row_bytes)
    copy_chunk(conv + (l * rows_per_layer + d) * conv_row_bytes,
               conv + (l * rows_per_layer + s) * conv_row_bytes, conv_row_bytes, off);
}

int launch_slot_copy(const PoolView &pv, int st, int io, int layer0, int nlayers,
                     const int32_t *src, const int32_t *dst, const uint8_t *mask, int n,
                     cudaStream_t s) {
  const size_t sb = (size_t)pv.H * pv.V * pv.K * (st == RSC_F32 ? 4 : 2);
  const size_t cb = (size_t)3 * pv.D * (io == RSC_F32 ? 4 : 2);
  const size_t longest = sb > cb ? sb : cb;
  dim3 grid((unsigned)((longest + kCopyChunk - 1) / kCopyChunk), n, nlayers);
  ssm_slot_copy_kernel<<<grid, 128, 0, s>>>(static_cast<char *>(pv.ssm), sb,
                                            static_cast<char *>(pv.conv), cb, pv.P + 1, layer0,
                                            pv.P, pv.err, src, dst, mask);
  return launch_status();
}

}  // namespace rsc

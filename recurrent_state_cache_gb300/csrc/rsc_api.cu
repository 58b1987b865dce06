// rsc_api.cu -- the C ABI of include/rsc.h: host-side validation and dispatch to the
// launchers.  Every value the host can see is checked here before anything is launched;
// values that live in device arrays (slot ids, accept counts, cu_seqlens) are checked
// by the kernels, which skip the bad row and set a bit of the pool's error word.
#include <cuda_runtime.h>

#include <atomic>
#include <new>

#include "rsc_internal.h"

struct rsc_pool {
  rsc_pool_desc d;
  rsc::PoolView pv;
  std::atomic<int> device{-1};  // device holding the pool's memory, looked up on first launch
};

namespace {

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool valid_dtype(int d) { return d == RSC_F32 || d == RSC_BF16; }
size_t dsize(int d) { return d == RSC_F32 ? 4 : 2; }
constexpr int kMaxGrid = 65535;  // gridDim.y / gridDim.z limit

int validate_desc(const rsc_pool_desc *d) {
  if (!d) return RSC_EINVAL;
  if (d->num_layers < 1 || d->num_slots < 0 || d->num_heads < 1 || d->num_heads > kMaxGrid)
    return RSC_ERANGE;
  if (d->conv_kernel != 4) return RSC_EDTYPE;
  if (d->head_k != 64 && d->head_k != 128) return RSC_EDTYPE;
  if (d->head_v != 64 && d->head_v != 128) return RSC_EDTYPE;
  if (!valid_dtype(d->state_dtype) || !valid_dtype(d->conv_dtype)) return RSC_EDTYPE;
  if (d->gate != RSC_GATE_KDA && d->gate != RSC_GATE_GDN) return RSC_EDTYPE;
  return RSC_OK;
}

rsc::LayerArgs layer_args(const rsc_pool *p, int layer) {
  rsc::LayerArgs a;
  a.pv = p->pv;
  a.st = p->d.state_dtype;
  a.io = p->d.conv_dtype;
  a.gate = p->d.gate;
  a.layer = layer;
  return a;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// The pool's memory must be device memory of the current device (the kernels run there and
// dereference it).  Looked up once per pool, after every host check of the call has passed.
int on_pool_device(rsc_pool *p) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return RSC_ECUDA;
  int d = p->device.load(std::memory_order_relaxed);
  if (d < 0) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p->d.ssm_base) != cudaSuccess) {
      cudaGetLastError();  // an unregistered host pointer: clear the sticky status
      return RSC_EDEVICE;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return RSC_EDEVICE;
    d = at.device;
    p->device.store(d, std::memory_order_relaxed);
  }
  return d == cur ? RSC_OK : RSC_EDEVICE;
}

// Shared checks and launch of every decode entry point; need_track / need_gate: the entry
// point's own option pointers are required.
int decode_impl(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch, const void *qkv,
                const float *conv_w, const float *g, const float *beta, void *out,
                const rsc::DecodeExtras &ex, bool need_track, bool need_gate, void *stream) {
  if (!pool) return RSC_EINVAL;
  if (layer < 0 || layer >= pool->d.num_layers || batch < 0 || batch > kMaxGrid)
    return RSC_ERANGE;
  if (batch == 0) return RSC_OK;
  if (!slot_ids || !qkv || !conv_w || !g || !beta || !out) return RSC_EINVAL;
  if (need_track && (!ex.track_mask || !ex.track_slots)) return RSC_EINVAL;
  if (need_gate && (!ex.A_log || !ex.dt_bias)) return RSC_EINVAL;
  if (!aligned(qkv, 16) || !aligned(out, 16) || !aligned(conv_w, 16) || !aligned(g, 16) ||
      !aligned(beta, 4) || !aligned(slot_ids, 4))
    return RSC_EALIGN;
  if (ex.A_log && (!aligned(ex.dt_bias, 16) || !aligned(ex.A_log, 4))) return RSC_EALIGN;
  if (ex.track_slots && !aligned(ex.track_slots, 4)) return RSC_EALIGN;
  if (const int rc = on_pool_device(pool)) return rc;
  return rsc::launch_decode(layer_args(pool, layer), slot_ids, batch, qkv, conv_w, g, beta, out,
                            ex, as_stream(stream));
}

}  // namespace

extern "C" {

int ssm_pool_bytes(const rsc_pool_desc *desc, uint64_t *ssm_bytes, uint64_t *conv_bytes) {
  int rc = validate_desc(desc);
  if (rc) return rc;
  if (!ssm_bytes || !conv_bytes) return RSC_EINVAL;
  const uint64_t rows = (uint64_t)desc->num_layers * (uint64_t)(desc->num_slots + 1);
  const uint64_t D = (uint64_t)desc->num_heads * (2 * desc->head_k + desc->head_v);
  *ssm_bytes = rows * desc->num_heads * desc->head_v * desc->head_k * dsize(desc->state_dtype);
  *conv_bytes = rows * 3 * D * dsize(desc->conv_dtype);
  return RSC_OK;
}

int ssm_pool_create(const rsc_pool_desc *desc, rsc_pool **out) {
  if (!out) return RSC_EINVAL;
  *out = nullptr;
  int rc = validate_desc(desc);
  if (rc) return rc;
  if (!desc->ssm_base || !desc->conv_base || !desc->dev_error) return RSC_EINVAL;
  if (!aligned(desc->ssm_base, 16) || !aligned(desc->conv_base, 16) || !aligned(desc->dev_error, 4))
    return RSC_EALIGN;
  rsc_pool *p = new (std::nothrow) rsc_pool;
  if (!p) return RSC_EINVAL;
  p->d = *desc;
  p->pv.ssm = desc->ssm_base;
  p->pv.conv = desc->conv_base;
  p->pv.err = desc->dev_error;
  p->pv.P = desc->num_slots;
  p->pv.H = desc->num_heads;
  p->pv.K = desc->head_k;
  p->pv.V = desc->head_v;
  p->pv.D = desc->num_heads * (2 * desc->head_k + desc->head_v);
  *out = p;
  return RSC_OK;
}

int ssm_pool_destroy(rsc_pool *pool) {
  delete pool;
  return RSC_OK;
}

int kda_decode_step_ex(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                       const void *qkv, const float *conv_w, const float *g, const float *beta,
                       void *out, const rsc_decode_opts *opts, void *stream) {
  rsc::DecodeExtras ex;
  if (opts) {
    if ((opts->flags & ~RSC_DECODE_OVERLAP) != 0) return RSC_EINVAL;
    if ((opts->A_log == nullptr) != (opts->dt_bias == nullptr)) return RSC_EINVAL;
    if ((opts->track_mask == nullptr) != (opts->track_slots == nullptr)) return RSC_EINVAL;
    ex.A_log = opts->A_log;
    ex.dt_bias = opts->dt_bias;
    ex.track_mask = opts->track_mask;
    ex.track_slots = opts->track_slots;
    ex.overlap = (opts->flags & RSC_DECODE_OVERLAP) != 0;
  }
  return decode_impl(pool, layer, slot_ids, batch, qkv, conv_w, g, beta, out, ex, false, false,
                     stream);
}

int kda_decode_step(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                    const void *qkv, const float *conv_w, const float *g, const float *beta,
                    void *out, void *stream) {
  return decode_impl(pool, layer, slot_ids, batch, qkv, conv_w, g, beta, out,
                     rsc::DecodeExtras{}, false, false, stream);
}

int kda_decode_step_overlap(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                            const void *qkv, const float *conv_w, const float *g,
                            const float *beta, void *out, void *stream) {
  rsc::DecodeExtras ex;
  ex.overlap = true;
  return decode_impl(pool, layer, slot_ids, batch, qkv, conv_w, g, beta, out, ex, false, false,
                     stream);
}

int kda_decode_step_track(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                          const void *qkv, const float *conv_w, const float *g, const float *beta,
                          void *out, const uint8_t *track_mask, const int32_t *track_slots,
                          void *stream) {
  rsc::DecodeExtras ex;
  ex.track_mask = track_mask;
  ex.track_slots = track_slots;
  return decode_impl(pool, layer, slot_ids, batch, qkv, conv_w, g, beta, out, ex, true, false,
                     stream);
}

int kda_decode_step_gated(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                          const void *qkv, const float *conv_w, const float *a, const float *b,
                          const float *A_log, const float *dt_bias, void *out, void *stream) {
  rsc::DecodeExtras ex;
  ex.A_log = A_log;
  ex.dt_bias = dt_bias;
  return decode_impl(pool, layer, slot_ids, batch, qkv, conv_w, a, b, out, ex, false, true,
                     stream);
}

int kda_prefill_workspace_size(const rsc_pool *pool, int num_seqs, int total_tokens,
                               size_t *bytes) {
  if (!pool || !bytes) return RSC_EINVAL;
  if (num_seqs < 1 || num_seqs > kMaxGrid || total_tokens < 0) return RSC_ERANGE;
  *bytes = rsc::prefill_workspace_bytes(pool->pv, pool->d.state_dtype, num_seqs, total_tokens);
  return RSC_OK;
}

int kda_prefill_chunk(rsc_pool *pool, int layer, const int32_t *slot_ids,
                      const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                      const uint8_t *has_initial_state, const void *qkv, const float *conv_w,
                      const float *g, const float *beta, void *out, void *workspace,
                      size_t workspace_bytes, void *stream) {
  if (!pool) return RSC_EINVAL;
  if (layer < 0 || layer >= pool->d.num_layers) return RSC_ERANGE;
  if (num_seqs < 1 || num_seqs > kMaxGrid || total_tokens < 0) return RSC_ERANGE;
  if (!slot_ids || !cu_seqlens || !conv_w) return RSC_EINVAL;
  if (total_tokens > 0 && (!qkv || !g || !beta || !out)) return RSC_EINVAL;
  const size_t need =
      rsc::prefill_workspace_bytes(pool->pv, pool->d.state_dtype, num_seqs, total_tokens);
  if (workspace_bytes < need) return RSC_ENOSPACE;
  if (need > 0 && !workspace) return RSC_EINVAL;
  if (!aligned(conv_w, 16) || !aligned(slot_ids, 4) || !aligned(cu_seqlens, 4) ||
      (workspace && !aligned(workspace, 16)))
    return RSC_EALIGN;
  if (total_tokens > 0 && (!aligned(qkv, 16) || !aligned(out, 16) || !aligned(g, 16) ||
                           !aligned(beta, 4)))
    return RSC_EALIGN;
  if (const int rc = on_pool_device(pool)) return rc;
  return rsc::launch_prefill(layer_args(pool, layer), slot_ids, cu_seqlens, num_seqs,
                             total_tokens, has_initial_state, qkv, conv_w, g, beta, out,
                             workspace, workspace_bytes, as_stream(stream));
}

int ssm_slot_copy(rsc_pool *pool, int layer, const int32_t *src, const int32_t *dst,
                  const uint8_t *mask, int n, void *stream) {
  if (!pool) return RSC_EINVAL;
  if (layer < -1 || layer >= pool->d.num_layers || n < 0 || n > kMaxGrid) return RSC_ERANGE;
  if (n == 0) return RSC_OK;
  if (!src || !dst) return RSC_EINVAL;
  if (!aligned(src, 4) || !aligned(dst, 4)) return RSC_EALIGN;
  const int l0 = layer < 0 ? 0 : layer;
  const int nl = layer < 0 ? pool->d.num_layers : 1;
  if (nl > kMaxGrid) return RSC_ERANGE;
  if (const int rc = on_pool_device(pool)) return rc;
  return rsc::launch_slot_copy(pool->pv, pool->d.state_dtype, pool->d.conv_dtype, l0, nl, src,
                               dst, mask, n, as_stream(stream));
}

int kda_spec_verify_commit(rsc_pool *pool, int layer, int mode, const int32_t *slot_ids,
                           int batch, int T, int L, void *spec_ssm, void *spec_conv,
                           const void *qkv, const float *conv_w, const float *g,
                           const float *beta, void *out, const int32_t *accept,
                           void *stream) {
  if (!pool) return RSC_EINVAL;
  if (mode != RSC_SPEC_VERIFY && mode != RSC_SPEC_COMMIT) return RSC_EINVAL;
  if (layer < 0 || layer >= pool->d.num_layers || batch < 0 || batch > kMaxGrid)
    return RSC_ERANGE;
  if (L < 1 || L > 4096 || (L & (L - 1)) != 0 || T < 1 || T > L) return RSC_ERANGE;
  if (batch == 0) return RSC_OK;
  if (!slot_ids || !spec_ssm || !spec_conv) return RSC_EINVAL;
  if (!aligned(spec_ssm, 16) || !aligned(spec_conv, 16) || !aligned(slot_ids, 4))
    return RSC_EALIGN;
  const rsc::LayerArgs a = layer_args(pool, layer);
  if (mode == RSC_SPEC_COMMIT) {
    if (!accept) return RSC_EINVAL;
    if (!aligned(accept, 4)) return RSC_EALIGN;
    if (const int rc = on_pool_device(pool)) return rc;
    return rsc::launch_spec_commit(a, slot_ids, batch, T, L, spec_ssm, spec_conv, accept,
                                   as_stream(stream));
  }
  if (!qkv || !conv_w || !g || !beta || !out) return RSC_EINVAL;
  if (!aligned(qkv, 16) || !aligned(out, 16) || !aligned(conv_w, 16) || !aligned(g, 16) ||
      !aligned(beta, 4))
    return RSC_EALIGN;
  if (const int rc = on_pool_device(pool)) return rc;
  return rsc::launch_spec_verify(a, slot_ids, batch, T, L, spec_ssm, spec_conv, qkv, conv_w, g,
                                 beta, out, as_stream(stream));
}

int kda_replay_verify_commit(rsc_pool *pool, const rsc_replay_rings *rings, int layer, int mode,
                             const int32_t *slot_ids, const int32_t *ring_pos, int batch, int T,
                             void *spec_conv, const void *qkv, const float *conv_w,
                             const float *g, const float *beta, void *out,
                             const int32_t *accept, void *stream) {
  if (!pool || !rings) return RSC_EINVAL;
  if (mode != RSC_SPEC_VERIFY && mode != RSC_SPEC_COMMIT) return RSC_EINVAL;
  if (layer < 0 || layer >= pool->d.num_layers || batch < 0 || batch > kMaxGrid)
    return RSC_ERANGE;
  const int L = rings->depth;
  if (L < 2 || L > 4096 || (L & (L - 1)) != 0 || T < 1 || 2 * T > L) return RSC_ERANGE;
  if (batch == 0) return RSC_OK;
  if (!slot_ids || !ring_pos || !spec_conv || !rings->d || !rings->k || !rings->rawv ||
      !rings->rawk || !rings->g || !rings->beta)
    return RSC_EINVAL;
  if (!aligned(spec_conv, 16) || !aligned(slot_ids, 4) || !aligned(ring_pos, 4) ||
      !aligned(rings->d, 16) || !aligned(rings->k, 16) || !aligned(rings->rawv, 16) ||
      !aligned(rings->rawk, 16) || !aligned(rings->g, 16) || !aligned(rings->beta, 4))
    return RSC_EALIGN;
  const rsc::LayerArgs a = layer_args(pool, layer);
  const rsc::RingView rv{rings->d, rings->k, rings->rawv, rings->rawk, rings->g, rings->beta, L};
  if (mode == RSC_SPEC_COMMIT) {
    if (!accept) return RSC_EINVAL;
    if (!aligned(accept, 4)) return RSC_EALIGN;
    if (const int rc = on_pool_device(pool)) return rc;
    return rsc::launch_replay_commit(a, rv, slot_ids, ring_pos, batch, T, spec_conv, accept,
                                     as_stream(stream));
  }
  if (!qkv || !conv_w || !g || !beta || !out) return RSC_EINVAL;
  if (!aligned(qkv, 16) || !aligned(out, 16) || !aligned(conv_w, 16) || !aligned(g, 16) ||
      !aligned(beta, 4))
    return RSC_EALIGN;
  if (const int rc = on_pool_device(pool)) return rc;
  return rsc::launch_replay_verify(a, rv, slot_ids, ring_pos, batch, T, spec_conv, qkv, conv_w,
                                   g, beta, out, as_stream(stream));
}

int rsc_get_device_error(rsc_pool *pool, int32_t *code, void *stream) {
  if (!pool || !code) return RSC_EINVAL;
  if (const int rc = on_pool_device(pool)) return rc;
  cudaStream_t s = as_stream(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, pool->pv.err, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RSC_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RSC_ECUDA;
  if (cudaMemsetAsync(pool->pv.err, 0, sizeof host, s) != cudaSuccess) return RSC_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RSC_ECUDA;
  *code = host;
  return RSC_OK;
}

const char *rsc_status_string(int status) {
  switch (status) {
    case RSC_OK: return "ok";
    case RSC_EINVAL: return "invalid argument (null pointer, count or mode)";
    case RSC_ERANGE: return "argument out of range (layer, batch, length or cache depth)";
    case RSC_EDTYPE: return "unsupported dtype, gate, head dims or conv kernel";
    case RSC_EALIGN: return "pointer not aligned as required";
    case RSC_ECUDA: return "CUDA runtime error";
    case RSC_ENOSPACE: return "workspace too small";
    case RSC_EDEVICE: return "the pool's memory is not device memory of the current device";
    default: return "unknown status";
  }
}

}  // extern "C"

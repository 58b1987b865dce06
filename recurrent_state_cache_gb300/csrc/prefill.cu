// prefill.cu -- prefill of packed sequences over the slot pool, token-serial form.
//
// Source: "SGLang之KV Cache内存池机制" §8.5 forward_extend: each sequence starts from the
// state its slot holds (or from zero), runs the recurrence over its tokens and leaves
// the final state (and conv window) in the slot.  Sequences are packed along tokens
// and delimited by cu_seqlens.
//
// Three launches:
//   prep       grid (token, head): conv of the head's q/k/v channels over the previous
//              three raw inputs (from the sequence, or the slot's window before the
//              sequence start, or zero for a fresh sequence), L2 norm of q and k;
//              writes q_hat, k_hat, v (fp32) and k_hat.q_hat to the workspace.
//   recurrent  grid (row tile, head, sequence): the delta-rule tile of decode.cu run
//              over the sequence's tokens with S in registers the whole time; per-token
//              operands are staged into shared memory 8 tokens at a time with cp.async,
//              double-buffered, so the serial loop never waits on HBM.  The final S is
//              rounded once to the state dtype and written back.
//   window     grid (channel block, sequence): the slot's window becomes the last three
//              raw inputs of the sequence (fewer than three tokens shift the old window).
// This is the exact fp32 recurrence; it is the path of pools with head_k 64 (fp32-state
// pools with head_k 128 take the same recurrence eight tokens at a time, prefill_blocked.cu).
#include "rsc_internal.h"
#include "rsc_step.cuh"

namespace rsc {

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

PrefillWs prefill_carve(void *ws, const PoolView &pv, int T) {
  char *p = static_cast<char *>(ws);
  PrefillWs w;
  const size_t nq = align256((size_t)T * pv.H * pv.K * 4);
  const size_t nv = align256((size_t)T * pv.H * pv.V * 4);
  w.q = reinterpret_cast<float *>(p);
  w.k = reinterpret_cast<float *>(p + nq);
  w.v = reinterpret_cast<float *>(p + 2 * nq);
  w.kq = reinterpret_cast<float *>(p + 2 * nq + nv);
  return w;
}

size_t prefill_prep_bytes(const PoolView &pv, int T) {
  return 2 * align256((size_t)T * pv.H * pv.K * 4) + align256((size_t)T * pv.H * pv.V * 4) +
         align256((size_t)T * pv.H * 4);
}

// Index of the sequence holding token t: the last n with cu[n] <= t.
__device__ __forceinline__ int seq_of(const int32_t *cu, int N, int t) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename IO, int K, int V>
__global__ void __launch_bounds__(128)
prefill_prep_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                    const int32_t *__restrict__ cu, int N, const uint8_t *__restrict__ has_init,
                    const IO *__restrict__ qkv, const float *__restrict__ conv_w, PrefillWs ws) {
  constexpr int CH = 2 * K + V;
  __shared__ float y[CH];
  __shared__ float red[12];
  const int t = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int H = pv.H, D = pv.D;
  const int T = gridDim.x;
  const int n = seq_of(cu, N, t);
  const int start = cu[n], end = cu[n + 1];
  if (start < 0 || end > T || !(start <= t && t < end)) {
    if (tid == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_SEQ);
    return;
  }
  const int slot = slots[n];
  if (slot < 0 || slot > pv.P) {
    if (tid == 0 && h == 0 && t == start) flag_error(pv.err, RSC_DEVERR_SLOT);
    return;
  }
  const bool init = has_init == nullptr || has_init[n] != 0;
  const int pos = t - start;
  const IO *W = reinterpret_cast<const IO *>(pv.conv) + ((size_t)layer * (pv.P + 1) + slot) * 3 * (size_t)D;
  for (int ci = tid; ci < CH; ci += 128) {
    const int c = ci < K ? h * K + ci
                : ci < 2 * K ? H * K + h * K + (ci - K)
                             : 2 * H * K + h * V + (ci - 2 * K);
    float xm[4];  // inputs at positions pos-3 .. pos (oldest first)
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      const int pp = pos - 3 + m;
      xm[m] = pp >= 0 ? to_f32(qkv[(size_t)(start + pp) * D + c])
                      : (init ? to_f32(W[(size_t)(3 + pp) * D + c]) : 0.f);
    }
    xm[3] = to_f32(qkv[(size_t)t * D + c]);
    const float4 w = *reinterpret_cast<const float4 *>(conv_w + 4 * (size_t)c);
    y[ci] = conv4(w, xm[0], xm[1], xm[2], xm[3]);
  }
  __syncthreads();
  float qq = 0.f, kk = 0.f, qk = 0.f;
  if (tid < K) {
    const float a = y[tid], c = y[K + tid];
    qq = a * a; kk = c * c; qk = a * c;
  }
  block3_sum_128(qq, kk, qk, red);
  const float rq = 1.0f / sqrtf(qq + kNormEps), rk = 1.0f / sqrtf(kk + kNormEps);
  const size_t th = (size_t)t * H + h;
  for (int i = tid; i < K; i += 128) {
    ws.q[th * K + i] = y[i] * rq;
    ws.k[th * K + i] = y[K + i] * rk;
  }
  for (int i = tid; i < V; i += 128) ws.v[th * V + i] = y[2 * K + i];
  if (tid == 0) ws.kq[th] = qk * rq * rk;
}

template <typename ST, typename IO, int K, int V, int NVT, int GATE>
__global__ void __launch_bounds__(128)
prefill_recurrent_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                         const int32_t *__restrict__ cu, int T,
                         const uint8_t *__restrict__ has_init, PrefillWs ws,
                         const float *__restrict__ g, const float *__restrict__ beta,
                         IO *__restrict__ out) {
  constexpr int VT = V / NVT;
  constexpr int TS = 8;                         // tokens per staged block
  constexpr int GW = GATE == RSC_GATE_KDA ? K : 1;
  using G = TileGeom<ST, K, VT>;
  __shared__ __align__(16) float s_q[2][TS][K];
  __shared__ __align__(16) float s_k[2][TS][K];
  __shared__ __align__(16) float s_g[2][TS][GW];
  __shared__ __align__(16) float s_v[2][TS][VT];
  __shared__ float s_b[2][TS], s_kq[2][TS];

  const int j = blockIdx.x, h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x;
  const int H = pv.H;
  const int start = cu[n], end = cu[n + 1];
  if (start < 0 || end < start || end > T) {
    if (tid == 0 && j == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_SEQ);
    return;
  }
  const int slot = slots[n];
  if (slot < 0 || slot > pv.P) {
    if (tid == 0 && j == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_SLOT);
    return;
  }
  const bool init = has_init == nullptr || has_init[n] != 0;
  const size_t prow = (size_t)layer * (pv.P + 1) + slot;
  ST *S = reinterpret_cast<ST *>(pv.ssm) + ((prow * H + h) * V + (size_t)j * VT) * K;
  float s[G::NP][G::EPL];
  if (init) {
    tile_load<ST, K, VT>(S, s);
  } else {
#pragma unroll
    for (int p = 0; p < G::NP; ++p)
#pragma unroll
      for (int e = 0; e < G::EPL; ++e) s[p][e] = 0.f;
  }

  auto stage = [&](int buf, int t0) {
    const int cnt = min(TS, end - t0);
    for (int i = tid; i < cnt * (K / 4); i += 128) {
      const int tau = i / (K / 4), c4 = (i % (K / 4)) * 4;
      const size_t th = (size_t)(t0 + tau) * H + h;
      cp_async16(&s_q[buf][tau][c4], ws.q + th * K + c4);
      cp_async16(&s_k[buf][tau][c4], ws.k + th * K + c4);
      if (GATE == RSC_GATE_KDA) cp_async16(&s_g[buf][tau][c4], g + th * K + c4);
    }
    for (int i = tid; i < cnt * (VT / 4); i += 128) {
      const int tau = i / (VT / 4), c4 = (i % (VT / 4)) * 4;
      const size_t th = (size_t)(t0 + tau) * H + h;
      cp_async16(&s_v[buf][tau][c4], ws.v + th * V + (size_t)j * VT + c4);
    }
    if (tid < cnt) {
      const size_t th = (size_t)(t0 + tid) * H + h;
      cp_async4(&s_b[buf][tid], beta + th);
      cp_async4(&s_kq[buf][tid], ws.kq + th);
      if (GATE != RSC_GATE_KDA) cp_async4(&s_g[buf][tid][0], g + th);
    }
    cp_async_commit();
  };

  const int k0 = G::kofs();
  int cur = 0;
  if (start < end) stage(0, start);
  for (int t0 = start; t0 < end; t0 += TS) {
    cp_async_wait_all();
    __syncthreads();  // block `cur` landed; everyone is done with block cur^1
    if (t0 + TS < end) stage(cur ^ 1, t0 + TS);
    const int cnt = min(TS, end - t0);
    for (int tau = 0; tau < cnt; ++tau) {
      float qh[G::EPL], kh[G::EPL], al[G::EPL];
#pragma unroll
      for (int e = 0; e < G::EPL; ++e) {
        qh[e] = s_q[cur][tau][k0 + e];
        kh[e] = s_k[cur][tau][k0 + e];
        al[e] = expf(GATE == RSC_GATE_KDA ? s_g[cur][tau][k0 + e] : s_g[cur][tau][0]);
      }
      float o[G::NP];
      delta_rule_tile<ST, K, VT>(s, qh, kh, al, s_b[cur][tau], s_kq[cur][tau], s_v[cur][tau], o);
      if (k0 == 0) {
        IO *ob = out + ((size_t)(t0 + tau) * H + h) * V + (size_t)j * VT;
#pragma unroll
        for (int p = 0; p < G::NP; ++p) ob[G::row(p)] = from_f32<IO>(o[p]);
      }
    }
    cur ^= 1;
  }
  tile_store<ST, K, VT>(S, s);
}

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

template <typename ST, typename IO, int K, int V, int GATE>
struct PrefillSerialLaunch {
  static int run(const LayerArgs *a, const int32_t *slots, const int32_t *cu, int N, int T,
                 const uint8_t *has_init, const void *qkv, const float *conv_w,
                 const float *g, const float *beta, void *out, void *ws, cudaStream_t s) {
    constexpr int NVT = V / 32;
    const PrefillWs w = prefill_carve(ws, a->pv, T);
    if (T > 0) {
      prefill_prep_kernel<IO, K, V><<<dim3(T, a->pv.H), 128, 0, s>>>(
          a->pv, a->layer, slots, cu, N, has_init, static_cast<const IO *>(qkv), conv_w, w);
      if (launch_status() != RSC_OK) return RSC_ECUDA;
    }
    prefill_recurrent_kernel<ST, IO, K, V, NVT, GATE><<<dim3(NVT, a->pv.H, N), 128, 0, s>>>(
        a->pv, a->layer, slots, cu, T, has_init, w, g, beta, static_cast<IO *>(out));
    if (launch_status() != RSC_OK) return RSC_ECUDA;
    prefill_window_kernel<IO><<<dim3((a->pv.D + 127) / 128, N), 128, 0, s>>>(
        a->pv, a->layer, slots, cu, T, has_init, static_cast<const IO *>(qkv));
    return launch_status();
  }
};

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

int launch_prefill_serial(const LayerArgs &a, const int32_t *slots, const int32_t *cu,
                          int N, int T, const uint8_t *has_init, const void *qkv,
                          const float *conv_w, const float *g, const float *beta,
                          void *out, void *ws, cudaStream_t s) {
  // head_k 64 only: head_k 128 pools take the tensor-core or the blocked form
  if (a.pv.K != 64) return RSC_EDTYPE;
  if (a.st == RSC_F32)
    return a.io == RSC_F32
               ? dispatch_v<PrefillSerialLaunch, float, float, 64>(a.pv.V, a.gate, &a, slots, cu,
                                                                   N, T, has_init, qkv, conv_w,
                                                                   g, beta, out, ws, s)
               : dispatch_v<PrefillSerialLaunch, float, bf16, 64>(a.pv.V, a.gate, &a, slots, cu,
                                                                  N, T, has_init, qkv, conv_w, g,
                                                                  beta, out, ws, s);
  return a.io == RSC_F32
             ? dispatch_v<PrefillSerialLaunch, bf16, float, 64>(a.pv.V, a.gate, &a, slots, cu, N,
                                                                T, has_init, qkv, conv_w, g, beta,
                                                                out, ws, s)
             : dispatch_v<PrefillSerialLaunch, bf16, bf16, 64>(a.pv.V, a.gate, &a, slots, cu, N,
                                                               T, has_init, qkv, conv_w, g, beta,
                                                               out, ws, s);
}

int launch_prefill_prep(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N,
                        int T, const uint8_t *has_init, const void *qkv, const float *conv_w,
                        const PrefillWs &w, cudaStream_t s) {
  if (T == 0) return RSC_OK;
  const int K = a.pv.K, V = a.pv.V;
  const dim3 grid(T, a.pv.H);
#define RSC_PREP(IO_, K_, V_)                                                               \
  prefill_prep_kernel<IO_, K_, V_><<<grid, 128, 0, s>>>(a.pv, a.layer, slots, cu, N, has_init, \
                                                        static_cast<const IO_ *>(qkv), conv_w, w)
  if (a.io == RSC_BF16) {
    if (K == 128 && V == 128) RSC_PREP(bf16, 128, 128);
    else if (K == 128) RSC_PREP(bf16, 128, 64);
    else if (V == 128) RSC_PREP(bf16, 64, 128);
    else RSC_PREP(bf16, 64, 64);
  } else {
    if (K == 128 && V == 128) RSC_PREP(float, 128, 128);
    else if (K == 128) RSC_PREP(float, 128, 64);
    else if (V == 128) RSC_PREP(float, 64, 128);
    else RSC_PREP(float, 64, 64);
  }
#undef RSC_PREP
  return launch_status();
}

static bool use_tc(const PoolView &pv, int st) { return st == RSC_BF16 && pv.K == 128; }
static bool use_blocked(const PoolView &pv, int st) { return st == RSC_F32 && pv.K == 128; }

size_t prefill_workspace_bytes(const PoolView &pv, int st, int N, int T) {
  if (use_tc(pv, st))
    return align256((size_t)(N + 1) * 4) +
           prefill_tc_chunk_capacity(N, T) * (size_t)pv.H * prefill_tc_block_bytes();
  if (use_blocked(pv, st)) return prefill_blocked_bytes(pv, N, T);
  return prefill_prep_bytes(pv, T);
}

int launch_prefill(const LayerArgs &a, const int32_t *slots, const int32_t *cu_seqlens,
                   int N, int T, const uint8_t *has_init, const void *qkv,
                   const float *conv_w, const float *g, const float *beta, void *out,
                   void *ws, size_t ws_bytes, cudaStream_t s) {
  if (ws_bytes < prefill_workspace_bytes(a.pv, a.st, N, T)) return RSC_ENOSPACE;
  if (use_blocked(a.pv, a.st))
    return launch_prefill_blocked(a, slots, cu_seqlens, N, T, has_init, qkv, conv_w, g, beta,
                                  out, ws, s);
  if (!use_tc(a.pv, a.st))
    return launch_prefill_serial(a, slots, cu_seqlens, N, T, has_init, qkv, conv_w, g, beta,
                                 out, ws, s);
  int32_t *chunk_base = static_cast<int32_t *>(ws);
  char *blocks = static_cast<char *>(ws) + align256((size_t)(N + 1) * 4);
  // the tensor-core path writes the windows in its state pass
  return launch_prefill_tc(a, slots, cu_seqlens, N, T, has_init, qkv, conv_w, g, beta, out,
                           chunk_base, blocks, s);
}

}  // namespace rsc

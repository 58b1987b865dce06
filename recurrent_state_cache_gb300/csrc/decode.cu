// decode.cu -- fused decode step: slot lookup, short conv with in-place window roll,
// L2 norm of q and k, gated delta rule on the slot's state, output.
//
// Sources: decode pseudo-code of "SGLang之KV Cache内存池机制" §8.5 (decay, delta, beta,
// rank-1 write, output; the state read and written in place through cache_indices) and
// the conv window of "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理", section
// "Conv state".
//
// One thread-block cluster per (request, head): NVT CTAs of NW warps, CTA j owning
// rows [j*VT, (j+1)*VT) of the head's state S[V][K] (VT = V/NVT).  Data flow of a CTA:
//   1. the slot id is bounds-checked and one elected thread starts a TMA bulk copy of
//      the CTA's whole S tile (VT*K contiguous elements) into shared memory, completing
//      on an mbarrier: the tile's HBM traffic is in flight while the rest of the
//      prologue runs, and no registers are tied up holding it;
//   2. every CTA of the cluster computes the conv of all 2K q/k channels of its head
//      (redundantly, a few KB from L2) and of its own VT value channels;
//   3. block reductions give |q|^2, |k|^2, q.k, hence q_hat, k_hat and k_hat.q_hat;
//   4. a cluster barrier orders every CTA's window reads before any window write; each
//      window channel is then rolled by exactly one thread of the cluster (q/k channels
//      partitioned over the NVT CTAs, value channels by row tile), so the window update
//      is a bit-exact shift with a single writer per byte;
//   5. after a bounded wait on the mbarrier, each warp streams its rows out of shared
//      memory pass by pass: delta rule on 16-byte row segments (rsc_step.cuh), the new
//      state stored straight back to the slot with coalesced 16-byte stores.
#include "rsc_internal.h"
#include "rsc_step.cuh"

namespace rsc {

template <typename ST, typename IO, int K, int V, int NVT, int NW, int GATE>
__global__ void __cluster_dims__(NVT, 1, 1) __launch_bounds__(NW * 32)
kda_decode_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                  const IO *__restrict__ qkv, const float *__restrict__ conv_w,
                  const float *__restrict__ g, const float *__restrict__ beta,
                  IO *__restrict__ out) {
  constexpr int NT = NW * 32;
  constexpr int VT = V / NVT;
  using G = TileGeom<ST, K, VT, NW>;
  constexpr int QK_T = (2 * K + NT - 1) / NT;  // q/k channels per thread
  constexpr int OWN = 2 * K / NVT;             // q/k channels rolled by each CTA
  constexpr uint32_t TILE_BYTES = VT * K * sizeof(ST);
  static_assert(VT <= NT && K <= NT, "one value row and one key channel per thread");
  static_assert(TILE_BYTES % 16 == 0, "bulk copy granularity");

  extern __shared__ __align__(128) unsigned char smem_raw[];
  ST *s_S = reinterpret_cast<ST *>(smem_raw);  // the VT x K tile
  __shared__ float s_qk[2 * K];                // conv outputs: q then k of this head
  __shared__ float s_v[VT];                    // conv outputs of this tile's value rows
  __shared__ float s_red[3 * NW];
  __shared__ __align__(8) uint64_t s_bar;

  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int H = pv.H, D = pv.D;

  const int slot = slots[b];
  if (slot < 0 || slot > pv.P) {
    if (tid == 0 && j == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_SLOT);
    return;  // uniform over the cluster: every CTA of it sees the same slot
  }
  const size_t prow = (size_t)layer * (pv.P + 1) + slot;
  ST *S = reinterpret_cast<ST *>(pv.ssm) + ((prow * H + h) * V + (size_t)j * VT) * K;

  // 1. S tile -> shared memory, asynchronously.
  if (tid == 0) mbar_init(&s_bar, 1);
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&s_bar, TILE_BYTES);
    bulk_g2s(s_S, S, TILE_BYTES, &s_bar);
  }

  // 2. conv of the head's q/k channels and of this tile's value channels.
  IO *W = reinterpret_cast<IO *>(pv.conv) + prow * 3 * (size_t)D;
  const IO *x = qkv + (size_t)b * D;
  IO keep[QK_T][3];
#pragma unroll
  for (int u = 0; u < QK_T; ++u) {
    const int i2 = tid + u * NT;
    if (i2 < 2 * K) {
      const int c = i2 < K ? h * K + i2 : H * K + h * K + (i2 - K);
      const float4 w = *reinterpret_cast<const float4 *>(conv_w + 4 * (size_t)c);
      const IO w0 = W[c], w1 = W[D + c], w2 = W[2 * D + c], xc = x[c];
      s_qk[i2] = conv4(w, to_f32(w0), to_f32(w1), to_f32(w2), to_f32(xc));
      keep[u][0] = w1; keep[u][1] = w2; keep[u][2] = xc;
    }
  }
  IO keepv[3];
  const int cv = 2 * H * K + h * V + j * VT + tid;
  if (tid < VT) {
    const float4 w = *reinterpret_cast<const float4 *>(conv_w + 4 * (size_t)cv);
    const IO w0 = W[cv], w1 = W[D + cv], w2 = W[2 * D + cv], xc = x[cv];
    s_v[tid] = conv4(w, to_f32(w0), to_f32(w1), to_f32(w2), to_f32(xc));
    keepv[0] = w1; keepv[1] = w2; keepv[2] = xc;
  }
  __syncthreads();

  // 3. norms and k.q.
  float qq = 0.f, kk = 0.f, qk = 0.f;
  if (tid < K) {
    const float a = s_qk[tid], c = s_qk[K + tid];
    qq = a * a; kk = c * c; qk = a * c;
  }
  block3_sum<NW>(qq, kk, qk, s_red);
  const float rq = 1.0f / sqrtf(qq + kNormEps);
  const float rk = 1.0f / sqrtf(kk + kNormEps);
  const float kq = qk * rq * rk;

  float qh[G::EPL], kh[G::EPL], al[G::EPL];
  const int k0 = G::kofs();
#pragma unroll
  for (int e = 0; e < G::EPL; ++e) {
    qh[e] = s_qk[k0 + e] * rq;
    kh[e] = s_qk[K + k0 + e] * rk;
  }
  if (GATE == RSC_GATE_KDA) {
    const float *gg = g + ((size_t)b * H + h) * K + k0;
#pragma unroll
    for (int e = 0; e < G::EPL; ++e) al[e] = expf(gg[e]);
  } else {
    const float a = expf(g[(size_t)b * H + h]);
#pragma unroll
    for (int e = 0; e < G::EPL; ++e) al[e] = a;
  }
  const float bt = beta[(size_t)b * H + h];

  // 4. window roll: all reads of the cluster happen before any write.
  if (NVT > 1) cluster_sync_all();
#pragma unroll
  for (int u = 0; u < QK_T; ++u) {
    const int i2 = tid + u * NT;
    if (i2 < 2 * K && i2 >= j * OWN && i2 < (j + 1) * OWN) {
      const int c = i2 < K ? h * K + i2 : H * K + h * K + (i2 - K);
      W[c] = keep[u][0]; W[D + c] = keep[u][1]; W[2 * D + c] = keep[u][2];
    }
  }
  if (tid < VT) { W[cv] = keepv[0]; W[D + cv] = keepv[1]; W[2 * D + cv] = keepv[2]; }

  // 5. delta rule pass by pass out of shared memory; state back in place.
  if (!mbar_wait(&s_bar, 0)) {
    flag_error(pv.err, RSC_DEVERR_TIMEOUT);
    mbar_wait(&s_bar, 0);  // give the copy one more bounded chance to land
    return;
  }
  IO *ob = out + ((size_t)b * H + h) * V + (size_t)j * VT;
#pragma unroll 2
  for (int p = 0; p < G::NP; ++p) {
    const int r = G::row(p);
    float s[G::EPL];
    unpack16(*reinterpret_cast<const uint4 *>(s_S + (size_t)r * K + k0), s);
    const float o = delta_rule_row<G::EPL, G::LPR>(s, qh, kh, al, bt, kq, s_v[r]);
    st16(S + (size_t)r * K + k0, pack16(s));
    if (k0 == 0) ob[r] = from_f32<IO>(o);
  }
}

// Tile shape per state dtype: rows per CTA (VT) and warps per CTA.
#ifndef RSC_DECODE_ROWS_BF16
#define RSC_DECODE_ROWS_BF16 32
#endif
#ifndef RSC_DECODE_WARPS_BF16
#define RSC_DECODE_WARPS_BF16 4
#endif
#ifndef RSC_DECODE_ROWS_F32
#define RSC_DECODE_ROWS_F32 32
#endif
#ifndef RSC_DECODE_WARPS_F32
#define RSC_DECODE_WARPS_F32 4
#endif

template <typename ST> struct DecodeTile;
template <> struct DecodeTile<bf16> {
  static constexpr int ROWS = RSC_DECODE_ROWS_BF16, WARPS = RSC_DECODE_WARPS_BF16;
};
template <> struct DecodeTile<float> {
  static constexpr int ROWS = RSC_DECODE_ROWS_F32, WARPS = RSC_DECODE_WARPS_F32;
};

template <typename ST, typename IO, int K, int V, int GATE>
struct DecodeLaunch {
  static int run(const LayerArgs *a, const int32_t *slots, int B, const void *qkv,
                 const float *conv_w, const float *g, const float *beta, void *out,
                 cudaStream_t s) {
    constexpr int ROWS = DecodeTile<ST>::ROWS < V ? DecodeTile<ST>::ROWS : V;
    constexpr int NVT = V / ROWS;
    constexpr int NW = DecodeTile<ST>::WARPS;
    constexpr size_t SMEM = (size_t)ROWS * K * sizeof(ST);
    auto kern = kda_decode_kernel<ST, IO, K, V, NVT, NW, GATE>;
    static bool attr_set = false;  // per instantiation; set on the first (uncaptured) call
    if (!attr_set) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) !=
          cudaSuccess)
        return RSC_ECUDA;
      attr_set = true;
    }
    dim3 grid(NVT, a->pv.H, B);
    kern<<<grid, NW * 32, SMEM, s>>>(a->pv, a->layer, slots, static_cast<const IO *>(qkv),
                                     conv_w, g, beta, static_cast<IO *>(out));
    return launch_status();
  }
};

int launch_decode(const LayerArgs &a, const int32_t *slots, int B, const void *qkv,
                  const float *conv_w, const float *g, const float *beta, void *out,
                  cudaStream_t s) {
  return dispatch_all<DecodeLaunch>(a.st, a.io, a.pv.K, a.pv.V, a.gate, &a, slots, B, qkv,
                                    conv_w, g, beta, out, s);
}

}  // namespace rsc

// decode.cu -- fused decode step: slot lookup, short conv with in-place window roll,
// L2 norm of q and k, gated delta rule on the slot's state, output.
//
// Sources: decode pseudo-code of "SGLang之KV Cache内存池机制" §8.5 (decay, delta, beta,
// rank-1 write, output; the state read and written in place through cache_indices) and
// the conv window of "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理", section
// "Conv state".
//
// One thread-block cluster per (request, head): NVT CTAs of NW warps, CTA j owning
// rows [j*VT, (j+1)*VT) of the head's state S[V][K] (VT = V/NVT; NVT = 1 by default, a
// whole head per CTA).  Data flow of a CTA:
//   1. plain launch: the small inputs are requested first -- qkv, conv taps, gate and beta
//      before the slot id returns, the slot's window right after -- because the conv
//      depends on them and, requested later, they would queue in DRAM behind the tile
//      copies of every CTA on the GPU (measured: the conv then finished ~5 us into a 13 us
//      launch).  Overlapped launch (kda_decode_step_overlap, a programmatic dependent of
//      the previous kernel on the stream): the slot id, the window and the first tile
//      chunks are requested while that kernel still runs, and only the call's own inputs
//      wait for it; the grid releases its own dependents after that wait;
//   2. one elected thread starts TMA bulk copies of the CTA's S tile (VT*K contiguous
//      elements) into shared memory in NCH row chunks, each completing on its own
//      mbarrier: EARLY chunks at once, the rest as soon as the conv is computed;
//   3. block reductions give |q|^2, |k|^2, q.k, hence q_hat, k_hat and k_hat.q_hat;
//   4. (clusters only) a cluster barrier orders every CTA's window reads before any
//      window write; each window channel is rolled by exactly one thread of the cluster
//      (q/k channels partitioned over the NVT CTAs, value channels by row tile), so the
//      window update is a bit-exact shift with a single writer per byte;
//   5. each warp streams its rows out of shared memory pass by pass, waiting (bounded)
//      for a chunk only when it reaches it: delta rule on 16-byte row segments
//      (rsc_step.cuh), the new state stored straight back to the slot with coalesced
//      16-byte stores, so a CTA's writes overlap its own later reads.
//
// Extras, chosen per call (uniform branches, one kernel):
//   fused gating (kda_decode_step_gated, ex.A_log set): `g` and `beta` carry the layer's raw
//     gate projections a, b and the gates are formed in the kernel (reading of the fused
//     sigmoid-gating decode named by "SGLang之KV Cache内存池机制" §10; the pages give no
//     formula): beta = sigmoid(b), g = -exp(A_log[h]) * softplus(a + dt_bias), per key
//     channel (KDA) or per head (GDN);
//   tracking (kda_decode_step_track, ex.track_mask set): "SGLang Qwen3/kimi-k3 Hybrid Linear
//     Mamba KV cache管理", mamba_track_interval: when track_mask[b] is set, the updated state
//     and window of the request also go to slot track_slots[b] (the masked track copy of the
//     pages, written from registers instead of re-read from the active slot).
#include "rsc_internal.h"
#include "rsc_step.cuh"

namespace rsc {

__device__ __forceinline__ float softplus_f(float x) {
  return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_f(float x) {
  if (x >= 0.f) return 1.f / (1.f + expf(-x));
  const float e = expf(x);
  return e / (1.f + e);
}

template <typename ST, typename IO, int K, int V, int NVT, int NW, int NCH, int EARLY, int GATE,
          bool OVL>
__global__ void __cluster_dims__(NVT, 1, 1) __launch_bounds__(NW * 32)
kda_decode_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                  const IO *__restrict__ qkv, const float *__restrict__ conv_w,
                  const float *__restrict__ g, const float *__restrict__ beta,
                  IO *__restrict__ out, DecodeExtras ex) {
  constexpr int NT = NW * 32;
  constexpr int VT = V / NVT;
  using G = TileGeom<ST, K, VT, NW>;
  constexpr int QK_T = (2 * K + NT - 1) / NT;  // q/k channels per thread
  constexpr int OWN = 2 * K / NVT;             // q/k channels rolled by each CTA
  constexpr uint32_t TILE_BYTES = VT * K * sizeof(ST);
  constexpr uint32_t CHUNK_BYTES = TILE_BYTES / NCH;  // one bulk copy + mbarrier each
  constexpr int PPC = G::NP / NCH;                    // passes per chunk
  static_assert(VT <= NT && K <= NT, "one value row and one key channel per thread");
  static_assert(PPC * NCH == G::NP && CHUNK_BYTES % 16 == 0, "chunks of whole passes");

  extern __shared__ __align__(128) unsigned char smem_raw[];
  ST *s_S = reinterpret_cast<ST *>(smem_raw);  // the VT x K tile
  __shared__ float s_qk[2 * K];                // conv outputs: q then k of this head
  __shared__ float s_v[VT];                    // conv outputs of this tile's value rows
  __shared__ float s_red[3 * NW];
  __shared__ __align__(8) uint64_t s_bar[NCH];
  // fused gating, KDA: each key channel's gate once per CTA (thread t, channel t)
  __shared__ float s_gate[GATE == RSC_GATE_KDA ? K : 1];

  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int H = pv.H, D = pv.D;
  const int cv = 2 * H * K + h * V + j * VT + tid;  // value channel of thread tid < VT
  const int k0 = G::kofs();
  const bool raw = ex.A_log != nullptr;

  // The call's own inputs: qkv, conv taps, gate and beta, into registers.
  const IO *x = qkv + (size_t)b * D;
  float4 wqk[QK_T];
  IO xqk[QK_T];
  float4 wv = make_float4(0.f, 0.f, 0.f, 0.f);
  IO xv = from_f32<IO>(0.f);
  float gl[G::EPL];  // the gate
  float a_raw = 0.f, d_raw = 0.f, s_raw = 0.f;  // raw gate inputs, used once the tile is requested
  float bt = 0.f;
  auto load_inputs = [&]() {
#pragma unroll
    for (int u = 0; u < QK_T; ++u) {
      const int i2 = tid + u * NT;
      if (i2 < 2 * K) {
        const int c = i2 < K ? h * K + i2 : H * K + h * K + (i2 - K);
        wqk[u] = *reinterpret_cast<const float4 *>(conv_w + 4 * (size_t)c);
        xqk[u] = x[c];
      }
    }
    if (tid < VT) {
      wv = *reinterpret_cast<const float4 *>(conv_w + 4 * (size_t)cv);
      xv = x[cv];
    }
    if (GATE == RSC_GATE_KDA && raw) {
      if (tid < K) {
        a_raw = g[((size_t)b * H + h) * K + tid];
        d_raw = ex.dt_bias[(size_t)h * K + tid];
        s_raw = ex.A_log[h];
      }
    } else if (GATE == RSC_GATE_KDA) {
      float4 g4[G::EPL / 4];
      const float4 *gg = reinterpret_cast<const float4 *>(g + ((size_t)b * H + h) * K + k0);
#pragma unroll
      for (int e = 0; e < G::EPL / 4; ++e) g4[e] = gg[e];
#pragma unroll
      for (int e = 0; e < G::EPL / 4; ++e) {
        gl[4 * e] = g4[e].x; gl[4 * e + 1] = g4[e].y; gl[4 * e + 2] = g4[e].z; gl[4 * e + 3] = g4[e].w;
      }
    } else {
      const float gh = g[(size_t)b * H + h];
#pragma unroll
      for (int e = 0; e < G::EPL; ++e) gl[e] = gh;
    }
    bt = beta[(size_t)b * H + h];
    if (raw && GATE != RSC_GATE_KDA) {
      d_raw = ex.dt_bias[h];
      s_raw = ex.A_log[h];
    }
  };

  // The slot's rows: its state tile S and conv window W; the window channels this thread
  // rolls go to registers, the tile to shared memory in NCH row chunks on their own
  // mbarriers (chunk c holds the rows of passes [c*PPC, (c+1)*PPC)), EARLY of them now.
  ST *S = nullptr;
  IO *W = nullptr;
  IO keep[QK_T][3];
  IO keepv[3];
  auto issue_chunk = [&](int c) {
    mbar_arrive_expect_tx(&s_bar[c], CHUNK_BYTES);
#ifdef RSC_TEST_STARVE_FIRST_CHUNK
    // Test build only (never in the library): request 0's first chunk is armed but not
    // copied, so its bounded wait runs out and the give-up path runs with no copy in flight.
    if (b == 0 && c == 0) return;
#endif
    bulk_g2s(reinterpret_cast<char *>(s_S) + c * CHUNK_BYTES,
             reinterpret_cast<const char *>(S) + c * CHUNK_BYTES, CHUNK_BYTES, &s_bar[c]);
  };
  auto load_slot = [&]() -> bool {
    const int slot = slots[b];
    if (slot < 0 || slot > pv.P) {
      if (tid == 0 && j == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_SLOT);
      return false;  // uniform over the cluster: every CTA of it sees the same slot
    }
    const size_t prow = (size_t)layer * (pv.P + 1) + slot;
    S = reinterpret_cast<ST *>(pv.ssm) + ((prow * H + h) * V + (size_t)j * VT) * K;
    W = reinterpret_cast<IO *>(pv.conv) + prow * 3 * (size_t)D;
#pragma unroll
    for (int u = 0; u < QK_T; ++u) {
      const int i2 = tid + u * NT;
      if (i2 < 2 * K) {
        const int c = i2 < K ? h * K + i2 : H * K + h * K + (i2 - K);
        keep[u][0] = W[c]; keep[u][1] = W[D + c]; keep[u][2] = W[2 * D + c];
      }
    }
    if (tid < VT) { keepv[0] = W[cv]; keepv[1] = W[D + cv]; keepv[2] = W[2 * D + cv]; }
    if (tid == 0) {
#pragma unroll
      for (int c = 0; c < NCH; ++c) mbar_init(&s_bar[c], 1);
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int c = 0; c < EARLY; ++c) issue_chunk(c);
    }
    return true;
  };

  // 1. Request order.  Plain launch: the call's inputs first, then the slot id, the window
  //    and the first tile chunks -- the conv (and with it every row update) waits on the
  //    small inputs, and requested after the tiles of every CTA on the GPU they would queue
  //    behind them in DRAM (measured: the conv then finished ~5 us into a 13 us launch).
  //    Overlapped launch (programmatic dependent of the previous kernel on the stream): the
  //    slot's rows are requested while that kernel still runs, and only the call's inputs,
  //    which it may produce, wait for its completion.  This grid releases its own dependents
  //    only after that wait, when every kernel before it has completed: the early reads of a
  //    dependent can then overlap this grid alone, never one further back in the stream.
  if constexpr (OVL) {
    const bool have_slot = load_slot();
    grid_dep_wait();
    grid_dep_launch_dependents();
    if (!have_slot) return;
    load_inputs();
  } else {
    load_inputs();
    if (!load_slot()) return;
  }
  // tracking: the same tile and window channels of the track slot (null when not tracked)
  ST *St = nullptr;
  IO *Wt = nullptr;
  if (ex.track_mask != nullptr && ex.track_mask[b]) {
    const int ts = ex.track_slots[b];
    if (ts < 0 || ts > pv.P) {
      if (tid == 0 && j == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_SLOT);
    } else {
      const size_t trow = (size_t)layer * (pv.P + 1) + ts;
      St = reinterpret_cast<ST *>(pv.ssm) + ((trow * H + h) * V + (size_t)j * VT) * K;
      Wt = reinterpret_cast<IO *>(pv.conv) + trow * 3 * (size_t)D;
    }
  }
  // fused gating, formed only now so that waiting for its inputs holds back no request
  // (b in bt; GDN: a in gl)
  if (raw) {
    if (GATE == RSC_GATE_KDA) {
      if (tid < K) s_gate[tid] = -expf(s_raw) * softplus_f(a_raw + d_raw);
    } else {
      const float gh = -expf(s_raw) * softplus_f(gl[0] + d_raw);
#pragma unroll
      for (int e = 0; e < G::EPL; ++e) gl[e] = gh;
    }
    bt = sigmoid_f(bt);
    __syncthreads();  // uniform: raw is a kernel argument
    if (GATE == RSC_GATE_KDA) {
#pragma unroll
      for (int e = 0; e < G::EPL; ++e) gl[e] = s_gate[k0 + e];
    }
  }

  // 2. conv of the head's q/k channels and of this tile's value channels; the window values
  // each thread will roll are kept (keep[u] becomes rows 1, 2 and the input).
#pragma unroll
  for (int u = 0; u < QK_T; ++u) {
    const int i2 = tid + u * NT;
    if (i2 < 2 * K) {
      s_qk[i2] = conv4(wqk[u], to_f32(keep[u][0]), to_f32(keep[u][1]), to_f32(keep[u][2]),
                       to_f32(xqk[u]));
      keep[u][0] = keep[u][1]; keep[u][1] = keep[u][2]; keep[u][2] = xqk[u];
    }
  }
  if (tid < VT) {
    s_v[tid] = conv4(wv, to_f32(keepv[0]), to_f32(keepv[1]), to_f32(keepv[2]), to_f32(xv));
    keepv[0] = keepv[1]; keepv[1] = keepv[2]; keepv[2] = xv;
  }
  __syncthreads();
  if (tid == 0) {
#pragma unroll
    for (int c = EARLY; c < NCH; ++c) issue_chunk(c);
  }

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

  constexpr int E2 = G::EPL / 2;
  float2 qh[E2], kh[E2], al[E2];
#pragma unroll
  for (int e = 0; e < E2; ++e) {
    qh[e] = make_float2(s_qk[k0 + 2 * e] * rq, s_qk[k0 + 2 * e + 1] * rq);
    kh[e] = make_float2(s_qk[K + k0 + 2 * e] * rk, s_qk[K + k0 + 2 * e + 1] * rk);
    al[e] = make_float2(expf(gl[2 * e]), expf(gl[2 * e + 1]));
  }

  // 4. window roll: all reads of the cluster happen before any write.
  if (NVT > 1) cluster_sync_all();
#pragma unroll
  for (int u = 0; u < QK_T; ++u) {
    const int i2 = tid + u * NT;
    if (i2 < 2 * K && i2 >= j * OWN && i2 < (j + 1) * OWN) {
      const int c = i2 < K ? h * K + i2 : H * K + h * K + (i2 - K);
      W[c] = keep[u][0]; W[D + c] = keep[u][1]; W[2 * D + c] = keep[u][2];
      if (Wt) { Wt[c] = keep[u][0]; Wt[D + c] = keep[u][1]; Wt[2 * D + c] = keep[u][2]; }
    }
  }
  if (tid < VT) {
    W[cv] = keepv[0]; W[D + cv] = keepv[1]; W[2 * D + cv] = keepv[2];
    if (Wt) { Wt[cv] = keepv[0]; Wt[D + cv] = keepv[1]; Wt[2 * D + cv] = keepv[2]; }
  }

  // 5. delta rule pass by pass out of shared memory; state back in place.
  IO *ob = out + ((size_t)b * H + h) * V + (size_t)j * VT;
#pragma unroll 2
  for (int p = 0; p < G::NP; ++p) {
    if (p % PPC == 0 && !mbar_wait(&s_bar[p / PPC], 0)) {
      flag_error(pv.err, RSC_DEVERR_TIMEOUT);
      for (int c = p / PPC; c < NCH; ++c) mbar_wait(&s_bar[c], 0);  // let copies land
      return;
    }
    const int r = G::row(p);
    float sf[G::EPL];
    unpack16(*reinterpret_cast<const uint4 *>(s_S + (size_t)r * K + k0), sf);
    float2 s[E2];
#pragma unroll
    for (int e = 0; e < E2; ++e) s[e] = make_float2(sf[2 * e], sf[2 * e + 1]);
    const float o = delta_rule_row2<E2, G::LPR>(s, qh, kh, al, bt, kq, s_v[r]);
#pragma unroll
    for (int e = 0; e < E2; ++e) { sf[2 * e] = s[e].x; sf[2 * e + 1] = s[e].y; }
    const uint4 packed = pack16(sf);
    st16(S + (size_t)r * K + k0, packed);
    if (St) st16(St + (size_t)r * K + k0, packed);
    if (k0 == 0) ob[r] = from_f32<IO>(o);
  }
}

// Tile shape per state dtype: rows per CTA (VT) and warps per CTA.
#ifndef RSC_DECODE_ROWS_BF16
#define RSC_DECODE_ROWS_BF16 128
#endif
#ifndef RSC_DECODE_WARPS_BF16
#define RSC_DECODE_WARPS_BF16 4
#endif
#ifndef RSC_DECODE_ROWS_F32
#define RSC_DECODE_ROWS_F32 128
#endif
#ifndef RSC_DECODE_WARPS_F32
#define RSC_DECODE_WARPS_F32 8
#endif

// Bulk copies (and mbarriers) per CTA tile, and how many of them start before the conv.
#ifndef RSC_DECODE_CHUNKS
#define RSC_DECODE_CHUNKS 4
#endif
#ifndef RSC_DECODE_EARLY_CHUNKS
#define RSC_DECODE_EARLY_CHUNKS 2
#endif
// The same for the overlapped launch, where the early chunks are requested before the wait
// for the previous kernel, per state dtype.  bf16, 69-layer KDA graph at batch 64, us per
// layer: 4 chunks with 1/2/3/4 early 10.1/9.05/10.0/11.0; 8 with 2/4/6 early 10.1/9.2/10.0;
// 2 with 1 early 8.98.  fp32 (64 KB tiles), 48-layer GDN graph at batch 1/16/64: 2 with 1
// early 4.74/13.7/42.6; 4 with 2 early 4.23/13.1/42.3; 4 with 1 or 3 and 8 with 4 no better.
#ifndef RSC_DECODE_OVL_CHUNKS_BF16
#define RSC_DECODE_OVL_CHUNKS_BF16 2
#endif
#ifndef RSC_DECODE_OVL_EARLY_BF16
#define RSC_DECODE_OVL_EARLY_BF16 1
#endif
#ifndef RSC_DECODE_OVL_CHUNKS_F32
#define RSC_DECODE_OVL_CHUNKS_F32 4
#endif
#ifndef RSC_DECODE_OVL_EARLY_F32
#define RSC_DECODE_OVL_EARLY_F32 2
#endif

template <typename ST> struct DecodeTile;
template <> struct DecodeTile<bf16> {
  static constexpr int ROWS = RSC_DECODE_ROWS_BF16, WARPS = RSC_DECODE_WARPS_BF16;
  static constexpr int OVL_CHUNKS = RSC_DECODE_OVL_CHUNKS_BF16, OVL_EARLY = RSC_DECODE_OVL_EARLY_BF16;
};
template <> struct DecodeTile<float> {
  static constexpr int ROWS = RSC_DECODE_ROWS_F32, WARPS = RSC_DECODE_WARPS_F32;
  static constexpr int OVL_CHUNKS = RSC_DECODE_OVL_CHUNKS_F32, OVL_EARLY = RSC_DECODE_OVL_EARLY_F32;
};

template <typename ST, typename IO, int K, int V, int GATE>
struct DecodeLaunch {
  static int run(const LayerArgs *a, const int32_t *slots, int B, const void *qkv,
                 const float *conv_w, const float *g, const float *beta, void *out,
                 DecodeExtras ex, cudaStream_t s) {
    constexpr int ROWS = DecodeTile<ST>::ROWS < V ? DecodeTile<ST>::ROWS : V;
    constexpr int NVT = V / ROWS;
    constexpr int NW = DecodeTile<ST>::WARPS;
    constexpr size_t SMEM = (size_t)ROWS * K * sizeof(ST);
    constexpr int NP = TileGeom<ST, K, ROWS, NW>::NP;
    constexpr int NCH = NP % RSC_DECODE_CHUNKS == 0 ? RSC_DECODE_CHUNKS : 1;
    constexpr int EARLY = RSC_DECODE_EARLY_CHUNKS < NCH ? RSC_DECODE_EARLY_CHUNKS : NCH;
    constexpr int ONCH = NP % DecodeTile<ST>::OVL_CHUNKS == 0 ? DecodeTile<ST>::OVL_CHUNKS : 1;
    constexpr int OEARLY = DecodeTile<ST>::OVL_EARLY < ONCH ? DecodeTile<ST>::OVL_EARLY : ONCH;
    auto kern = kda_decode_kernel<ST, IO, K, V, NVT, NW, NCH, EARLY, GATE, false>;
    auto kern_ovl = kda_decode_kernel<ST, IO, K, V, NVT, NW, ONCH, OEARLY, GATE, true>;
    static PerDeviceFlag attr;  // per instantiation and device; set on the first call there
    const int rc = once_per_device(attr, [&] {
      return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) ==
                         cudaSuccess &&
                     cudaFuncSetAttribute(kern_ovl, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)SMEM) == cudaSuccess
                 ? RSC_OK
                 : RSC_ECUDA;
    });
    if (rc != RSC_OK) return rc;
    dim3 grid(NVT, a->pv.H, B);
    if (ex.overlap)
      return launch_pdl(kern_ovl, grid, dim3(NW * 32), SMEM, s, a->pv, a->layer, slots,
                        static_cast<const IO *>(qkv), conv_w, g, beta, static_cast<IO *>(out), ex);
    kern<<<grid, NW * 32, SMEM, s>>>(a->pv, a->layer, slots, static_cast<const IO *>(qkv),
                                     conv_w, g, beta, static_cast<IO *>(out), ex);
    return launch_status();
  }
};
int launch_decode(const LayerArgs &a, const int32_t *slots, int B, const void *qkv,
                  const float *conv_w, const float *g, const float *beta, void *out,
                  const DecodeExtras &ex, cudaStream_t s) {
  return dispatch_all<DecodeLaunch>(a.st, a.io, a.pv.K, a.pv.V, a.gate, &a, slots, B, qkv,
                                    conv_w, g, beta, out, ex, s);
}

}  // namespace rsc

// prefill_tc.cu -- chunked prefill in the chunkwise (WY / UT) form on the tcgen05 tensor
// cores, for bf16-state pools with K = 128.
//
// Source: "SGLang之KV Cache内存池机制" §8.5 (chunk-based extend with chunk 64: an
// inter-chunk recurrence plus intra-chunk parallel work) and the unrolled closed form of
// the recurrence printed in "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理"
// (ReplaySSM section).  The pages give no more than that; the algebra below is derived
// from the recurrence and is checked against it by the oracle's own chunkwise form.
//
// For a chunk of c <= 64 tokens starting from state S0, with per-channel cumulative log
// gates G_r = sum_{i<=r} g_i, Gamma_r = exp(G_r):
//   A[r][j]  = beta_r sum_k k_r[k] k_j[k] exp(G_r[k] - G_j[k])   (j < r)
//   P[r][j]  =        sum_k q_r[k] k_j[k] exp(G_r[k] - G_j[k])   (j <= r)
//   W  = (I + A)^-1 Diag(beta) (K . Gamma),   U' = (I + A)^-1 Diag(beta) V
//   U  = U' - W S0^T              (row r of U is the delta d_r of token r)
//   O  = (Q . Gamma) S0^T + P U
//   S_c = S0 Diag(Gamma_c) + U^T (K . Gamma_c / Gamma)
//
// Launches (after the conv/norm prep kernel of prefill.cu):
//   chunk table  one warp: chunk_base[n] = chunks before sequence n (64-token chunks).
//   intra        grid (chunk, head): the parts that do not depend on the state.  The
//                products A and P are one 128x64x128 MMA ([K.e^(G-R); Q.e^(G-R)] times
//                (K.e^(R-G))^T, R the per-channel midpoint of G over the chunk, so no
//                factor exceeds e^(range/2)); W and U' by forward substitution in fp32.
//                Writes per (chunk, head) a block of bf16 tensor-core operands already
//                in the canonical shared-memory layout: [W; Q.Gamma] (128xK),
//                (K.Gamma_c/Gamma)^T (Kx64), P (64x64), U' by 32-column tiles, Gamma_c.
//   state        grid (32-row tile of S, head, sequence): walks the sequence's chunks in
//                order with the tile's state in fp32 registers (thread k holds column k)
//                and per chunk runs MMA1 = [W; Q.Gamma] S0^T (U correction and the
//                inter-chunk output in one 128x32x128 MMA), then MMA2 = (K.Gamma_c/
//                Gamma)^T U (state update) and MMA3 = [0; P] U (intra-chunk output).
//                The next chunk's operand block is fetched by TMA bulk copies into the
//                other half of a double buffer while the current chunk runs.
//   window       prefill.cu's window kernel.
#include "rsc_internal.h"
#include "rsc_step.cuh"
#include "rsc_tc.cuh"

namespace rsc {

namespace {

constexpr int kC = 64;     // chunk length
constexpr int kK = 128;    // key dim of the tensor-core path
constexpr int kVT = 32;    // state rows per state-pass CTA
// Largest per-channel spread of the cumulative log gate inside one chunk for which the
// split exponentials e^(+-(G - R)) stay far from the fp32 / bf16 range (e^80 ~ 5.5e34).
constexpr float kGateSpreadLimit = 160.f;

// Per (chunk, head) operand block in the workspace (bytes).
constexpr size_t kOffXW = 0;                         // [W; Q.Gamma]   128 x K   canonical, KD = K
constexpr size_t kOffBT = kOffXW + 128 * kK * 2;     // (K.Gamma_c/Gamma)^T  K x 64  canonical, KD = 64
constexpr size_t kOffP = kOffBT + kK * kC * 2;       // P  64 x 64  canonical, KD = 64
constexpr size_t kOffUP = kOffP + kC * kC * 2;       // U' as [V/32][64][32] bf16 (room for V = 128)
constexpr size_t kOffGC = kOffUP + 128 * kC * 2;     // Gamma_c [K] fp32
constexpr size_t kBlockBytes = ((kOffGC + kK * 4) + 1023) / 1024 * 1024;

// Shared-memory buffer of the state pass (one per double-buffer half).
constexpr uint32_t kBufXW = 0;
constexpr uint32_t kBufBT = kBufXW + 128 * kK * 2;   // 32768
constexpr uint32_t kBufP0 = kBufBT + kK * kC * 2;    // 49152: [64 zero rows | P] = 128 x 64
constexpr uint32_t kBufUP = kBufP0 + 128 * kC * 2;   // 65536: U' tile 64 x 32
constexpr uint32_t kBufGC = kBufUP + kC * kVT * 2;   // 69632
constexpr uint32_t kBufBytes = ((kBufGC + kK * 4) + 1023) / 1024 * 1024;
constexpr uint32_t kOffS = 2 * kBufBytes;            // S0 tile (bf16) as MMA1 operand: 32 x K
constexpr uint32_t kOffU = kOffS + kVT * kK * 2;     // U^T (bf16) as MMA2/3 operand: 32 x 64
constexpr uint32_t kStateSmem = kOffU + kVT * kC * 2;

// Shared memory of the intra kernel.
constexpr uint32_t kIntraG = 0;                          // fp32 [64][K]   cumulative gates
constexpr uint32_t kIntraA = kIntraG + kC * kK * 4;      // fp32 [64][64]  A
constexpr uint32_t kIntraX = kIntraA + kC * kC * 4;      // bf16 128 x K   [K.e^(G-R); Q.e^(G-R)]
constexpr uint32_t kIntraKi = kIntraX + 128 * kK * 2;    // bf16 64 x K    K.e^(R-G)
constexpr uint32_t kIntraWh = kIntraKi + kC * kK * 2;    // fp32 [64][K]   rows of W
constexpr uint32_t kIntraUh = kIntraWh + kC * kK * 4;    // fp32 [64][128] rows of U'
constexpr uint32_t kIntraSmem = kIntraUh + kC * 128 * 4;

__device__ __forceinline__ void st_bf16(void *p, float x) {
  *reinterpret_cast<bf16 *>(p) = __float2bfloat16_rn(x);
}
__device__ __forceinline__ float ld_bf16(const void *p) {
  return __bfloat162float(*reinterpret_cast<const bf16 *>(p));
}

// Last n in [0, N) with base[n] <= x.
__device__ __forceinline__ int last_le(const int32_t *base, int N, int x) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace

size_t prefill_tc_chunk_capacity(int N, int T) { return (size_t)T / kC + (size_t)N; }
size_t prefill_tc_block_bytes() { return kBlockBytes; }

// One warp: chunk_base[n] = number of 64-token chunks of sequences 0..n-1.  Any
// malformed cu_seqlens entry (negative, decreasing, beyond T) makes every count zero
// (nothing of the call is computed) and sets RSC_DEVERR_SEQ.
__global__ void prefill_chunk_table_kernel(const int32_t *__restrict__ cu, int N, int T,
                                           int32_t *__restrict__ chunk_base, int32_t *err) {
  const int lane = threadIdx.x;
  bool bad = false;
  for (int n = lane; n < N; n += 32) {
    const int a = cu[n], b = cu[n + 1];
    bad |= a < 0 || b < a || b > T;
  }
  bad = __any_sync(0xffffffffu, bad);
  if (bad && lane == 0) flag_error(err, RSC_DEVERR_SEQ);
  int carry = 0;
  if (lane == 0) chunk_base[0] = 0;
  for (int base = 0; base < N; base += 32) {
    const int n = base + lane;
    int cnt = 0;
    if (n < N && !bad) cnt = (cu[n + 1] - cu[n] + kC - 1) / kC;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (n < N) chunk_base[n + 1] = carry + incl;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// Intra-chunk work of one (chunk, head).  128 threads; thread `ch` owns key channel ch.
// The gate g is [T][H][K] (KDA) or [T][H] (GDN, one value for every channel of a head).
template <int V, int GATE>
__global__ void __launch_bounds__(128)
prefill_tc_intra_kernel(PoolView pv, const int32_t *__restrict__ cu,
                        const int32_t *__restrict__ chunk_base, int N, PrefillWs ws,
                        const float *__restrict__ g, const float *__restrict__ beta,
                        char *__restrict__ blocks) {
  extern __shared__ __align__(1024) unsigned char smem[];
  float *sG = reinterpret_cast<float *>(smem + kIntraG);
  float *sA = reinterpret_cast<float *>(smem + kIntraA);
  unsigned char *sX = smem + kIntraX;
  unsigned char *sKi = smem + kIntraKi;
  float *sWh = reinterpret_cast<float *>(smem + kIntraWh);
  float *sUh = reinterpret_cast<float *>(smem + kIntraUh);
  __shared__ uint32_t s_taddr;
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ float s_beta[kC];

  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
  const int H = pv.H;
  if (cid >= chunk_base[N]) return;
  const int n = last_le(chunk_base, N, cid);
  const int t0 = cu[n] + kC * (cid - chunk_base[n]);
  const int Lc = min(kC, cu[n + 1] - t0);
  char *blk = blocks + ((size_t)cid * H + h) * kBlockBytes;
  const int ch = tid;

  if (tid < kC) s_beta[tid] = tid < Lc ? beta[(size_t)(t0 + tid) * H + h] : 0.f;

  // cumulative gates and the per-channel reference point R (midpoint of G's range)
  float G = 0.f, gmin = 0.f, gmax = 0.f;
#pragma unroll 8
  for (int r = 0; r < kC; ++r) {
    if (r < Lc) {
      const size_t th = (size_t)(t0 + r) * H + h;
      G += GATE == RSC_GATE_KDA ? g[th * kK + ch] : g[th];
    }
    sG[r * kK + ch] = G;
    if (r == 0) { gmin = G; gmax = G; }
    else if (r < Lc) { gmin = fminf(gmin, G); gmax = fmaxf(gmax, G); }
  }
  if (gmax - gmin > kGateSpreadLimit) flag_error(pv.err, RSC_DEVERR_GATE);
  const float R = 0.5f * (gmin + gmax);
  const float Glast = sG[(Lc - 1) * kK + ch];
  reinterpret_cast<float *>(blk + kOffGC)[ch] = expf(Glast);
  __syncthreads();  // s_beta

  // operands of A / P (shared memory), the state-independent operands of the state pass
  // (workspace): Q.Gamma rows of [W; Q.Gamma] and (K.Gamma_c/Gamma)^T, and the right-hand
  // sides beta_r k_r Gamma_r, beta_r v_r of the forward substitution below (seeded into
  // the rows it overwrites in place, so that loop touches no global memory)
#pragma unroll 4
  for (int r = 0; r < kC; ++r) {
    float kr = 0.f, qr = 0.f, vr = 0.f;
    if (r < Lc) {
      const size_t th = (size_t)(t0 + r) * H + h;
      kr = ws.k[th * kK + ch];
      qr = ws.q[th * kK + ch];
      if (ch < V) vr = ws.v[th * V + ch];
    }
    const float Gr = sG[r * kK + ch];
    sWh[r * kK + ch] = s_beta[r] * kr * expf(Gr);
    if (ch < V) sUh[r * 128 + ch] = s_beta[r] * vr;
    const float ep = expf(Gr - R), en = expf(R - Gr);
    st_bf16(sX + tc::kmajor_offset(r, ch, kK), kr * ep);
    st_bf16(sX + tc::kmajor_offset(kC + r, ch, kK), qr * ep);
    st_bf16(sKi + tc::kmajor_offset(r, ch, kK), kr * en);
    st_bf16(blk + kOffXW + tc::kmajor_offset(kC + r, ch, kK), qr * expf(Gr));
    st_bf16(blk + kOffBT + tc::kmajor_offset(ch, r, kC), r < Lc ? kr * expf(Glast - Gr) : 0.f);
  }

  // MMA: [K.e^(G-R); Q.e^(G-R)] (128 x K) times (K.e^(R-G))^T -> 128 x 64 in TMEM
  tc::fence_smem_to_async();
  if (tid == 0) mbar_init(&s_bar, 1);
  if (warp == 0) { tc::tmem_alloc(&s_taddr, 64); tc::tmem_relinquish(); }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = s_taddr;
  if (tid == 0) {
#pragma unroll
    for (int ks = 0; ks < kK / 16; ++ks)
      tc::mma_bf16(taddr, tc::kmajor_desc(sX, kK, ks), tc::kmajor_desc(sKi, kK, ks),
                   tc::idesc_bf16<128, kC>(), ks > 0);
    tc::mma_commit(&s_bar);
  }
  const bool ok = __syncthreads_and(mbar_wait(&s_bar, 0));
  tc::fence_after_sync();
  if (ok) {
    // lane = row: rows 0..63 hold A' (warps 0, 1), rows 64..127 hold P' (warps 2, 3)
    const int row = tid;
#pragma unroll
    for (int q4 = 0; q4 < kC / 16; ++q4) {
      float d[16];
      tc::tmem_ld16(tc::tmem_addr(taddr, 32 * warp, 16 * q4), d);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = 16 * q4 + i;
        if (row < kC) {
          sA[row * kC + j] = (j < row && row < Lc) ? s_beta[row] * d[i] : 0.f;
        } else {
          const int r = row - kC;
          st_bf16(blk + kOffP + tc::kmajor_offset(r, j, kC), (j <= r && r < Lc) ? d[i] : 0.f);
        }
      }
    }
  } else if (tid == 0) {
    flag_error(pv.err, RSC_DEVERR_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(taddr, 64);
  if (!ok) return;

  // W = (I+A)^-1 Diag(beta) (K.Gamma) and U' = (I+A)^-1 Diag(beta) V by forward
  // substitution down the rows; thread ch owns column ch of both, so it only ever reads
  // its own earlier rows (no barrier inside the loop).
  for (int r = 0; r < kC; ++r) {
    float w = 0.f, u = 0.f;
    if (r < Lc) {
      w = sWh[r * kK + ch];
      if (ch < V) u = sUh[r * 128 + ch];
      float w2 = 0.f, u2 = 0.f;  // two accumulators for instruction-level parallelism
      int j = 0;
      for (; j + 1 < r; j += 2) {
        const float a0 = sA[r * kC + j], a1 = sA[r * kC + j + 1];
        w = fmaf(-a0, sWh[j * kK + ch], w);
        w2 = fmaf(-a1, sWh[(j + 1) * kK + ch], w2);
        if (ch < V) {
          u = fmaf(-a0, sUh[j * 128 + ch], u);
          u2 = fmaf(-a1, sUh[(j + 1) * 128 + ch], u2);
        }
      }
      if (j < r) {
        const float a0 = sA[r * kC + j];
        w = fmaf(-a0, sWh[j * kK + ch], w);
        if (ch < V) u = fmaf(-a0, sUh[j * 128 + ch], u);
      }
      w += w2;
      u += u2;
    }
    sWh[r * kK + ch] = w;
    st_bf16(blk + kOffXW + tc::kmajor_offset(r, ch, kK), w);
    if (ch < V) {
      sUh[r * 128 + ch] = u;
      st_bf16(blk + kOffUP + ((size_t)((ch / kVT) * kC + r) * kVT + (ch % kVT)) * 2, u);
    }
  }
}

// Sequential state pass of one (32-row tile, head, sequence).
template <typename IO, int V>
__global__ void __launch_bounds__(128)
prefill_tc_state_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                        const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_base,
                        int T, const uint8_t *__restrict__ has_init,
                        const char *__restrict__ blocks, IO *__restrict__ out) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ uint32_t s_taddr;
  __shared__ __align__(8) uint64_t s_lbar[2];
  __shared__ __align__(8) uint64_t s_bar1, s_bar2;
  const int vt = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = pv.H;

  const int start = cu[n], end = cu[n + 1];
  const int nch = chunk_base[n + 1] - chunk_base[n];
  if (start < 0 || end < start || end > T || nch != (end - start + kC - 1) / kC) return;  // flagged by the table
  const int slot = slots[n];
  if (slot < 0 || slot > pv.P) {
    if (tid == 0 && vt == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_SLOT);
    return;
  }
  const bool init = has_init == nullptr || has_init[n] != 0;
  const size_t prow = (size_t)layer * (pv.P + 1) + slot;
  bf16 *Sg = reinterpret_cast<bf16 *>(pv.ssm) + ((prow * H + h) * V + (size_t)vt * kVT) * kK;

  // state tile in registers, transposed: thread k holds S[v][k] for the tile's 32 rows v
  float S[kVT];
#pragma unroll
  for (int v = 0; v < kVT; ++v) S[v] = init ? __bfloat162float(Sg[(size_t)v * kK + tid]) : 0.f;

  // zero rows 0..63 of both [0; P] operands (the TMA fills rows 64..127)
  for (int i = tid; i < 2 * (kC * kC * 2 / 16); i += 128) {
    const int b = i / (kC * kC * 2 / 16), o = i % (kC * kC * 2 / 16);
    st16(smem + b * kBufBytes + kBufP0 + o * 16, make_uint4(0, 0, 0, 0));
  }
  if (tid == 0) {
    mbar_init(&s_lbar[0], 1);
    mbar_init(&s_lbar[1], 1);
    mbar_init(&s_bar1, 1);
    mbar_init(&s_bar2, 1);
  }
  if (warp == 0) { tc::tmem_alloc(&s_taddr, 128); tc::tmem_relinquish(); }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = s_taddr;
  const uint32_t tD1 = tm, tD2 = tm + 32, tD3 = tm + 64;
  unsigned char *sS = smem + kOffS, *sU = smem + kOffU;

  auto issue_load = [&](int c, int b) {
    const char *blk = blocks + ((size_t)(chunk_base[n] + c) * H + h) * kBlockBytes;
    unsigned char *dst = smem + b * kBufBytes;
    mbar_arrive_expect_tx(&s_lbar[b], 128 * kK * 2 + kK * kC * 2 + kC * kC * 2 + kC * kVT * 2 + kK * 4);
    bulk_g2s(dst + kBufXW, blk + kOffXW, 128 * kK * 2, &s_lbar[b]);
    bulk_g2s(dst + kBufBT, blk + kOffBT, kK * kC * 2, &s_lbar[b]);
    bulk_g2s(dst + kBufP0 + kC * kC * 2, blk + kOffP, kC * kC * 2, &s_lbar[b]);
    bulk_g2s(dst + kBufUP, blk + kOffUP + (size_t)vt * kC * kVT * 2, kC * kVT * 2, &s_lbar[b]);
    bulk_g2s(dst + kBufGC, blk + kOffGC, kK * 4, &s_lbar[b]);
  };
  int issued = 0;  // loads issued (tid 0's count; the loop below consumes them in order)
  if (tid == 0 && nch > 0) { issue_load(0, 0); }
  issued = nch > 0 ? 1 : 0;

  bool ok = true;
  int c = 0;
  for (; c < nch; ++c) {
    const int b = c & 1;
    const unsigned char *buf = smem + b * kBufBytes;
    const int t0 = start + kC * c, Lc = min(kC, end - t0);
    // S0 (bf16) as MMA1's B operand: element (v, k)
#pragma unroll
    for (int v = 0; v < kVT; ++v) st_bf16(sS + tc::kmajor_offset(v, tid, kK), S[v]);
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    ok = __syncthreads_and(mbar_wait(&s_lbar[b], (c >> 1) & 1));
    if (!ok) break;
    tc::fence_after_sync();
    // Prefetch chunk c+1 into the other buffer.  Its last readers (chunk c-1's MMAs and
    // every thread's reads of its U' tile and Gamma_c) are all behind the barrier above.
    if (c + 1 < nch) {
      if (tid == 0) issue_load(c + 1, b ^ 1);
      issued = c + 2;
    }
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kK / 16; ++ks)
        tc::mma_bf16(tD1, tc::kmajor_desc(buf + kBufXW, kK, ks), tc::kmajor_desc(sS, kK, ks),
                     tc::idesc_bf16<128, kVT>(), ks > 0);
      tc::mma_commit(&s_bar1);
    }
    ok = __syncthreads_and(mbar_wait(&s_bar1, c & 1));
    if (!ok) break;
    tc::fence_after_sync();
    float d[kVT];
    {
      float d0[16], d1[16];
      tc::tmem_ld16(tc::tmem_addr(tD1, 32 * warp, 0), d0);
      tc::tmem_ld16(tc::tmem_addr(tD1, 32 * warp, 16), d1);
#pragma unroll
      for (int i = 0; i < 16; ++i) { d[i] = d0[i]; d[16 + i] = d1[i]; }
    }
    if (warp < 2) {
      // rows 0..63: U = U' - W S0^T, stored transposed (element (v, r)) for MMA2 / MMA3
      const int r = tid;
      const unsigned char *up = buf + kBufUP + (size_t)r * kVT * 2;
#pragma unroll
      for (int v = 0; v < kVT; ++v) {
        const float u = r < Lc ? ld_bf16(up + v * 2) - d[v] : 0.f;
        st_bf16(sU + tc::kmajor_offset(v, r, kC), u);
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks)
        tc::mma_bf16(tD2, tc::kmajor_desc(buf + kBufBT, kC, ks), tc::kmajor_desc(sU, kC, ks),
                     tc::idesc_bf16<128, kVT>(), ks > 0);
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks)
        tc::mma_bf16(tD3, tc::kmajor_desc(buf + kBufP0, kC, ks), tc::kmajor_desc(sU, kC, ks),
                     tc::idesc_bf16<128, kVT>(), ks > 0);
      tc::mma_commit(&s_bar2);
    }
    ok = __syncthreads_and(mbar_wait(&s_bar2, c & 1));
    if (!ok) break;
    tc::fence_after_sync();
    if (warp >= 2) {
      // rows 64..127: O = (Q.Gamma) S0^T + P U for token r of the chunk
      const int r = tid - kC;
      float d0[16], d1[16];
      tc::tmem_ld16(tc::tmem_addr(tD3, 32 * warp, 0), d0);
      tc::tmem_ld16(tc::tmem_addr(tD3, 32 * warp, 16), d1);
      if (r < Lc) {
        IO *o = out + ((size_t)(t0 + r) * H + h) * V + (size_t)vt * kVT;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          o[i] = from_f32<IO>(d[i] + d0[i]);
          o[16 + i] = from_f32<IO>(d[16 + i] + d1[i]);
        }
      }
    }
    {
      // S_c^T[k][:] = Gamma_c[k] S0^T[k][:] + (K.Gamma_c/Gamma)^T U for this thread's k
      const float gc = reinterpret_cast<const float *>(buf + kBufGC)[tid];
      float d0[16], d1[16];
      tc::tmem_ld16(tc::tmem_addr(tD2, 32 * warp, 0), d0);
      tc::tmem_ld16(tc::tmem_addr(tD2, 32 * warp, 16), d1);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        S[i] = fmaf(gc, S[i], d0[i]);
        S[16 + i] = fmaf(gc, S[16 + i], d1[i]);
      }
    }
    tc::fence_before_sync();
  }
  if (!ok) {
    if (tid == 0) {
      flag_error(pv.err, RSC_DEVERR_TIMEOUT);
      // let every issued bulk copy land before the shared memory is released
      for (int k = c; k < issued; ++k) mbar_wait(&s_lbar[k & 1], (k >> 1) & 1);
    }
  } else {
#pragma unroll
    for (int v = 0; v < kVT; ++v) Sg[(size_t)v * kK + tid] = __float2bfloat16_rn(S[v]);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tm, 128);
}

// ---------------------------------------------------------------------------- launch

template <typename IO, int V, int GATE>
static int launch_tc_v(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N, int T,
                       const uint8_t *has_init, const PrefillWs &w, const float *g,
                       const float *beta, void *out, int32_t *chunk_base, char *blocks,
                       cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(prefill_tc_intra_kernel<V, GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kIntraSmem) != cudaSuccess ||
        cudaFuncSetAttribute(prefill_tc_state_kernel<IO, V>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStateSmem) != cudaSuccess)
      return RSC_ECUDA;
    attr = true;
  }
  const unsigned cap = (unsigned)prefill_tc_chunk_capacity(N, T);
  if (cap > 0 && T > 0) {
    prefill_tc_intra_kernel<V, GATE><<<dim3(cap, a.pv.H), 128, kIntraSmem, s>>>(a.pv, cu, chunk_base, N, w, g,
                                                                          beta, blocks);
    if (launch_status() != RSC_OK) return RSC_ECUDA;
  }
  prefill_tc_state_kernel<IO, V><<<dim3(V / kVT, a.pv.H, N), 128, kStateSmem, s>>>(
      a.pv, a.layer, slots, cu, chunk_base, T, has_init, blocks, static_cast<IO *>(out));
  return launch_status();
}

int launch_prefill_tc(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N, int T,
                      const uint8_t *has_init, const PrefillWs &w, const float *g,
                      const float *beta, void *out, int32_t *chunk_base, char *blocks,
                      cudaStream_t s) {
  prefill_chunk_table_kernel<<<1, 32, 0, s>>>(cu, N, T, chunk_base, a.pv.err);
  if (launch_status() != RSC_OK) return RSC_ECUDA;
  const bool kda = a.gate == RSC_GATE_KDA;
#define RSC_TC(IO_, V_)                                                                        \
  (kda ? launch_tc_v<IO_, V_, RSC_GATE_KDA>(a, slots, cu, N, T, has_init, w, g, beta, out,      \
                                            chunk_base, blocks, s)                             \
       : launch_tc_v<IO_, V_, RSC_GATE_GDN>(a, slots, cu, N, T, has_init, w, g, beta, out,      \
                                            chunk_base, blocks, s))
  if (a.io == RSC_BF16) return a.pv.V == 128 ? RSC_TC(bf16, 128) : RSC_TC(bf16, 64);
  return a.pv.V == 128 ? RSC_TC(float, 128) : RSC_TC(float, 64);
#undef RSC_TC
}

}  // namespace rsc

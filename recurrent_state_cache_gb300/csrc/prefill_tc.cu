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
// Launches:
//   chunk table  one warp: chunk_base[n] = chunks before sequence n (64-token chunks).
//   chunk        grid (chunk, head): everything that does not depend on the state, from
//                the raw projections (conv, L2 norm, gates, the A/P products as one
//                128x64x128 MMA with a per-channel midpoint reference R of the cumulative
//                gate so no split factor exceeds e^(range/2), W and U' by blocked forward
//                substitution).  Writes per (chunk, head) a block of bf16 tensor-core
//                operands already in the canonical shared-memory layout: [W; Q.Gamma]
//                (128xK), (K.Gamma_c/Gamma)^T (Kx64), P (64x64), U' by 32-column tiles,
//                and Gamma_c.
//   state        grid (32-row tile of S, head, sequence): walks the sequence's chunks in
//                order with the tile's state in fp32 registers (thread k holds column k)
//                and per chunk runs MMA1 = [W; Q.Gamma] S0^T (U correction and the
//                inter-chunk output in one 128x32x128 MMA), then MMA2 = (K.Gamma_c/
//                Gamma)^T U (state update) and MMA3 = [0; P] U (intra-chunk output).
//                The next chunk's operand block is fetched by TMA bulk copies into the
//                other half of a double buffer; a chunk's output is written while the
//                next chunk's first MMA runs.
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
constexpr uint32_t kOffS = 2 * kBufBytes;            // S0 tile (bf16), MMA1's B: 32 x K, MN-major
constexpr uint32_t kOffU = kOffS + kVT * kK * 2;     // U (bf16), MMA2/3's B: 32 x 64, MN-major
constexpr uint32_t kStateSmem = kOffU + kVT * kC * 2;

// Shared memory of the fused chunk kernel (bytes).  sQ becomes the W history and sV the
// U' history in place; sX becomes A once the MMA that reads it has completed.
constexpr uint32_t kChQ = 0;                         // bf16 [64][K]  q_hat   -> W rows
constexpr uint32_t kChK = kChQ + kC * kK * 2;        // bf16 [64][K]  k_hat
constexpr uint32_t kChV = kChK + kC * kK * 2;        // bf16 [64][128] beta.v -> U' rows
constexpr uint32_t kChX = kChV + kC * 128 * 2;       // bf16 128 x K  [K.e^(G-R); Q.e^(G-R)] -> fp32 A^T [64][64]
constexpr uint32_t kChKi = kChX + 128 * kK * 2;      // bf16 64 x K   K.e^(R-G)
// Before the operands exist, the same region stages the chunk's raw bf16 inputs: rows of
// sequence positions t0-3 .. t0+63, channels [q (K) | k (K) | v (V)] of the head.
constexpr int kStageRows = kC + 3;
constexpr uint32_t kChStage = kChX;
constexpr uint32_t kChStageBytes = kStageRows * (2 * kK + 128) * 2;
constexpr uint32_t kChSmem = kChX + (kChStageBytes > 128 * kK * 2 + kC * kK * 2
                                         ? kChStageBytes : 128 * kK * 2 + kC * kK * 2);  // ~100 KB: two CTAs per SM

__device__ __forceinline__ void st_bf16(void *p, float x) {
  *reinterpret_cast<bf16 *>(p) = __float2bfloat16_rn(x);
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

// Everything of one (chunk, head) that does not depend on the state, from the raw
// projections: 256 threads.
//   1. conv + L2 norm, one warp per token (8 tokens per warp), lane l owning channels
//      4l..4l+3 of the head's q, k and v blocks; the three previous inputs come from the
//      sequence, or for its first tokens from the slot's window (zeros for a fresh one).
//      q_hat, k_hat and beta.v land in shared memory as bf16.
//   2. cumulative gates in registers: thread t owns channel t % 128 for rows
//      32 (t / 128) .. +31; the per-channel midpoint R of G's range, Gamma_c.
//   3. operands: [K.e^(G-R); Q.e^(G-R)] and K.e^(R-G) for the A/P MMA (shared memory);
//      Q.Gamma rows of [W; Q.Gamma] and (K.Gamma_c/Gamma)^T straight to the block;
//      beta.k.Gamma (the right-hand side of W) over q_hat in place.
//   4. A and P with one 128x64x128 MMA; A (x beta, strictly lower) to shared memory over
//      the spent operand, P (lower incl. diagonal) to the block.
//   5. W = (I+A)^-1 [beta.k.Gamma] and U' = (I+A)^-1 [beta.v] by blocked forward
//      substitution: thread t owns one column (W for t < 128, U' above); per 16-row block
//      the earlier blocks' contribution with 16 independent accumulators, then the
//      triangular 16x16 solve.  Rows of earlier blocks are read back as bf16 (what the
//      state pass consumes anyway).
template <typename IO, int V, int GATE>
__global__ void __launch_bounds__(256, 2)
prefill_tc_chunk_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                        const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_base,
                        int N, const uint8_t *__restrict__ has_init, const IO *__restrict__ qkv,
                        const float *__restrict__ conv_w, const float *__restrict__ g,
                        const float *__restrict__ beta, char *__restrict__ blocks) {
  extern __shared__ __align__(1024) unsigned char smem[];
  bf16 *sQ = reinterpret_cast<bf16 *>(smem + kChQ);
  bf16 *sK = reinterpret_cast<bf16 *>(smem + kChK);
  bf16 *sV = reinterpret_cast<bf16 *>(smem + kChV);
  unsigned char *sX = smem + kChX;
  unsigned char *sKi = smem + kChKi;
  float *sA = reinterpret_cast<float *>(smem + kChX);
  __shared__ uint32_t s_taddr;
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ float s_beta[kC];
  __shared__ float s_half[kK], s_min[kK], s_max[kK], s_glast[kK];

  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int H = pv.H, D = pv.D;
  if (cid >= chunk_base[N]) return;
  const int n = last_le(chunk_base, N, cid);
  const int seq0 = cu[n];
  const int c_in_seq = cid - chunk_base[n];
  const int t0 = seq0 + kC * c_in_seq;
  const int Lc = min(kC, cu[n + 1] - t0);
  const int slot = slots[n];
  if (slot < 0 || slot > pv.P) return;  // flagged by the state pass
  const bool init = has_init == nullptr || has_init[n] != 0;
  char *blk = blocks + ((size_t)cid * H + h) * kBlockBytes;
  if (tid < kC) s_beta[tid] = tid < Lc ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
  __syncthreads();

  // the gates of this thread's rows, requested now so their latency hides behind the conv
  const int ch = tid & (kK - 1), half = tid >> 7, r0 = 32 * half;
  float G[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int r = r0 + i;
    const size_t th = (size_t)(t0 + r) * H + h;
    G[i] = r < Lc ? (GATE == RSC_GATE_KDA ? g[th * kK + ch] : g[th]) : 0.f;
  }

  // ---- 1. conv + L2 norm
  if constexpr (sizeof(IO) == 2) {
    // bf16 inputs: the chunk's rows (3 before it, from the sequence or the slot's window,
    // or zero for a fresh sequence) staged with cp.async, then a sliding window per
    // channel and a warp-per-token norm pass.
    constexpr int CH = 2 * kK + V;  // staged channels
    bf16 *stg = reinterpret_cast<bf16 *>(smem + kChStage);
    const IO *Wn = reinterpret_cast<const IO *>(pv.conv) +
                   ((size_t)layer * (pv.P + 1) + slot) * 3 * (size_t)D;
    const int p0 = t0 - seq0 - 3;   // sequence position of staged row 0
    for (int i = tid; i < kStageRows * (CH / 8); i += 256) {
      const int row = i / (CH / 8), c8 = (i % (CH / 8)) * 8;
      const int pos = p0 + row;
      const int src_c = c8 < kK ? h * kK + c8 : c8 < 2 * kK ? H * kK + h * kK + (c8 - kK)
                                                            : 2 * H * kK + h * V + (c8 - 2 * kK);
      bf16 *dst = stg + row * CH + c8;
      if (row - 3 >= Lc) {
        st16(dst, make_uint4(0, 0, 0, 0));
      } else if (pos >= 0) {
        cp_async16(dst, qkv + (size_t)(seq0 + pos) * D + src_c);
      } else if (init) {
        cp_async16(dst, Wn + (size_t)(3 + pos) * D + src_c);
      } else {
        st16(dst, make_uint4(0, 0, 0, 0));
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    for (int c = tid; c < CH; c += 256) {
      const int gc = c < kK ? h * kK + c : c < 2 * kK ? H * kK + h * kK + (c - kK)
                                                     : 2 * H * kK + h * V + (c - 2 * kK);
      const float4 w = reinterpret_cast<const float4 *>(conv_w)[gc];
      float x0 = __bfloat162float(stg[c]), x1 = __bfloat162float(stg[CH + c]);
      float x2 = __bfloat162float(stg[2 * CH + c]);
      bf16 *dst = c < kK ? sQ + c : c < 2 * kK ? sK + (c - kK) : sV + (c - 2 * kK);
      const int dstride = c < 2 * kK ? kK : 128;
#pragma unroll 8
      for (int r = 0; r < kC; ++r) {
        const float x3 = __bfloat162float(stg[(r + 3) * CH + c]);
        dst[r * dstride] = __float2bfloat16_rn(conv4(w, x0, x1, x2, x3));
        x0 = x1; x1 = x2; x2 = x3;
      }
    }
    __syncthreads();
    for (int r = warp; r < kC; r += 8) {
      float q[4], k[4], v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        q[e] = __bfloat162float(sQ[r * kK + 4 * lane + e]);
        k[e] = __bfloat162float(sK[r * kK + 4 * lane + e]);
        v[e] = 4 * lane < V ? __bfloat162float(sV[r * 128 + 4 * lane + e]) : 0.f;
      }
      float qq = q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3];
      float kk = k[0] * k[0] + k[1] * k[1] + k[2] * k[2] + k[3] * k[3];
      qq = group_sum<32>(qq);
      kk = group_sum<32>(kk);
      const bool live = r < Lc;
      const float rq = live ? 1.0f / sqrtf(qq + kNormEps) : 0.f;
      const float rk = live ? 1.0f / sqrtf(kk + kNormEps) : 0.f;
      const float br = s_beta[r];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sQ[r * kK + 4 * lane + e] = __float2bfloat16_rn(q[e] * rq);
        sK[r * kK + 4 * lane + e] = __float2bfloat16_rn(k[e] * rk);
        if (4 * lane < V) sV[r * 128 + 4 * lane + e] = __float2bfloat16_rn(live ? br * v[e] : 0.f);
      }
    }
  } else {
    // fp32 inputs: a warp per token straight from global memory (lane l owns channels
    // 4l..4l+3 of q, k, v).
    const int cq = h * kK + 4 * lane, ck = H * kK + h * kK + 4 * lane;
    const int cv = 2 * H * kK + h * V + 4 * lane;
    const bool has_v = 4 * lane < V;
    float4 wq[4], wk[4], wv[4];  // taps of the lane's 4 channels per block
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      wq[e] = reinterpret_cast<const float4 *>(conv_w)[cq + e];
      wk[e] = reinterpret_cast<const float4 *>(conv_w)[ck + e];
      wv[e] = has_v ? reinterpret_cast<const float4 *>(conv_w)[cv + e] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const IO *W = reinterpret_cast<const IO *>(pv.conv) +
                  ((size_t)layer * (pv.P + 1) + slot) * 3 * (size_t)D;
    auto load4 = [&](int pos, int c, float (&x)[4]) {  // input of sequence position pos
      if (pos >= 0) {
        const IO *p = qkv + (size_t)(seq0 + pos) * D + c;
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = to_f32(p[e]);
      } else if (init) {
        const IO *p = W + (size_t)(3 + pos) * D + c;
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = to_f32(p[e]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = 0.f;
      }
    };
    for (int r = warp; r < kC; r += 8) {
      float yq[4] = {0.f, 0.f, 0.f, 0.f}, yk[4] = {0.f, 0.f, 0.f, 0.f}, yv[4] = {0.f, 0.f, 0.f, 0.f};
      if (r < Lc) {
        const int pos = t0 - seq0 + r;
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // tap i on position pos - 3 + i
          float xq[4], xk[4], xv[4];
          load4(pos - 3 + i, cq, xq);
          load4(pos - 3 + i, ck, xk);
          if (has_v) load4(pos - 3 + i, cv, xv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float tq = i == 0 ? wq[e].x : i == 1 ? wq[e].y : i == 2 ? wq[e].z : wq[e].w;
            const float tk = i == 0 ? wk[e].x : i == 1 ? wk[e].y : i == 2 ? wk[e].z : wk[e].w;
            const float tv = i == 0 ? wv[e].x : i == 1 ? wv[e].y : i == 2 ? wv[e].z : wv[e].w;
            yq[e] = fmaf(tq, xq[e], yq[e]);
            yk[e] = fmaf(tk, xk[e], yk[e]);
            if (has_v) yv[e] = fmaf(tv, xv[e], yv[e]);
          }
        }
      }
      float qq = yq[0] * yq[0] + yq[1] * yq[1] + yq[2] * yq[2] + yq[3] * yq[3];
      float kk = yk[0] * yk[0] + yk[1] * yk[1] + yk[2] * yk[2] + yk[3] * yk[3];
      qq = group_sum<32>(qq);
      kk = group_sum<32>(kk);
      const float rq = 1.0f / sqrtf(qq + kNormEps), rk = 1.0f / sqrtf(kk + kNormEps);
      const float br = s_beta[r];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sQ[r * kK + 4 * lane + e] = __float2bfloat16_rn(yq[e] * rq);
        sK[r * kK + 4 * lane + e] = __float2bfloat16_rn(yk[e] * rk);
        if (has_v) sV[r * 128 + 4 * lane + e] = __float2bfloat16_rn(br * yv[e]);
      }
    }
  }

  // ---- 2. cumulative gates (registers), reference point, Gamma_c
#pragma unroll
  for (int i = 1; i < 32; ++i) G[i] += G[i - 1];
  if (half == 0) s_half[ch] = G[31];
  __syncthreads();
  if (half == 1) {
    const float off = s_half[ch];
#pragma unroll
    for (int i = 0; i < 32; ++i) G[i] += off;
  }
  float gmin = 3.0e38f, gmax = -3.0e38f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (r0 + i < Lc) { gmin = fminf(gmin, G[i]); gmax = fmaxf(gmax, G[i]); }
  if (half == 1) { s_min[ch] = gmin; s_max[ch] = gmax; }
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (r0 + i == Lc - 1) s_glast[ch] = G[i];
  __syncthreads();
  if (half == 0) {
    gmin = fminf(gmin, s_min[ch]);
    gmax = fmaxf(gmax, s_max[ch]);
    s_min[ch] = gmin;
    s_max[ch] = gmax;
    if (gmax - gmin > kGateSpreadLimit) flag_error(pv.err, RSC_DEVERR_GATE);
    reinterpret_cast<float *>(blk + kOffGC)[ch] = expf(s_glast[ch]);
  }
  __syncthreads();
  const float R = 0.5f * (s_min[ch] + s_max[ch]);
  const float Glast = s_glast[ch];

  // ---- 3. operands
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int r = r0 + i;
    const float kr = __bfloat162float(sK[r * kK + ch]);
    const float qr = __bfloat162float(sQ[r * kK + ch]);
    const float Gr = G[i];
    const float ep = expf(Gr - R), en = expf(R - Gr), gam = expf(Gr);
    st_bf16(sX + tc::kmajor_offset(r, ch, kK), kr * ep);
    st_bf16(sX + tc::kmajor_offset(kC + r, ch, kK), qr * ep);
    st_bf16(sKi + tc::kmajor_offset(r, ch, kK), kr * en);
    st_bf16(blk + kOffXW + tc::kmajor_offset(kC + r, ch, kK), qr * gam);
    st_bf16(blk + kOffBT + tc::kmajor_offset(ch, r, kC), r < Lc ? kr * expf(Glast - Gr) : 0.f);
    sQ[r * kK + ch] = __float2bfloat16_rn(s_beta[r] * kr * gam);  // right-hand side of W
  }

  // ---- 4. A and P: [K.e^(G-R); Q.e^(G-R)] (128 x K) times (K.e^(R-G))^T -> 128 x 64
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
    // warp w reads lanes 32 (w % 4) .. +31 (rows) and columns 32 (w / 4) .. +31
    const int row = 32 * (warp & 3) + lane, cbase = 32 * (warp >> 2);
    float d[32];
    {
      float d0[16], d1[16];
      tc::tmem_ld16(tc::tmem_addr(taddr, 32 * (warp & 3), cbase), d0);
      tc::tmem_ld16(tc::tmem_addr(taddr, 32 * (warp & 3), cbase + 16), d1);
#pragma unroll
      for (int i = 0; i < 16; ++i) { d[i] = d0[i]; d[16 + i] = d1[i]; }
    }
    tc::fence_before_sync();
    __syncthreads();  // every read of sX by the MMA is over; A may overwrite it
    if (row < kC) {
      const float br = s_beta[row];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int j = cbase + i;
        sA[j * kC + row] = (j < row && row < Lc) ? br * d[i] : 0.f;  // stored transposed
      }
    } else {
      const int r = row - kC;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int j = cbase + i;
        st_bf16(blk + kOffP + tc::kmajor_offset(r, j, kC), (j <= r && r < Lc) ? d[i] : 0.f);
      }
    }
  } else if (tid == 0) {
    flag_error(pv.err, RSC_DEVERR_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(taddr, 64);
  if (!ok) return;

  // ---- 5. blocked forward substitution, one column per thread
  const bool is_w = tid < kK;
  const int col = is_w ? tid : tid - kK;
  if (!is_w && col >= V) return;
  bf16 *hist = is_w ? sQ : sV;          // rows of W / U' (right-hand side until solved)
  const int hstride = is_w ? kK : 128;
#pragma unroll 1
  for (int I = 0; I < kC / 16; ++I) {
    float acc[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) acc[r] = __bfloat162float(hist[(16 * I + r) * hstride + col]);
#pragma unroll 2
    for (int j = 0; j < 16 * I; ++j) {  // earlier blocks, solved; A^T row j = 16 coefficients
      const float xj = __bfloat162float(hist[j * hstride + col]);
      const float4 *aj = reinterpret_cast<const float4 *>(sA + j * kC + 16 * I);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 a4 = aj[q];
        acc[4 * q] = fmaf(-a4.x, xj, acc[4 * q]);
        acc[4 * q + 1] = fmaf(-a4.y, xj, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(-a4.z, xj, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(-a4.w, xj, acc[4 * q + 3]);
      }
    }
#pragma unroll
    for (int j = 0; j < 15; ++j) {  // the block's own triangle, column by column
      const float *aj = sA + (16 * I + j) * kC + 16 * I;
#pragma unroll
      for (int r = j + 1; r < 16; ++r) acc[r] = fmaf(-aj[r], acc[j], acc[r]);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int row = 16 * I + r;
      const float x = row < Lc ? acc[r] : 0.f;
      hist[row * hstride + col] = __float2bfloat16_rn(x);
      if (is_w) st_bf16(blk + kOffXW + tc::kmajor_offset(row, col, kK), x);
      else st_bf16(blk + kOffUP + ((size_t)((col / kVT) * kC + row) * kVT + (col % kVT)) * 2, x);
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
  __shared__ __align__(8) uint64_t s_xbar[2];  // [W; Q.Gamma] of a buffer landed
  __shared__ __align__(8) uint64_t s_lbar[2];  // the rest of a buffer's block landed
  __shared__ __align__(8) uint64_t s_bar1, s_bar2, s_bar3;
  __shared__ volatile int s_fail;  // a bounded wait ran out somewhere; checked after barriers
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
    mbar_init(&s_xbar[0], 1);
    mbar_init(&s_xbar[1], 1);
    mbar_init(&s_lbar[0], 1);
    mbar_init(&s_lbar[1], 1);
    mbar_init(&s_bar1, 1);
    mbar_init(&s_bar2, 1);
    mbar_init(&s_bar3, 1);
    s_fail = 0;
  }
  if (warp == 0) { tc::tmem_alloc(&s_taddr, 128); tc::tmem_relinquish(); }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = s_taddr;
  const uint32_t tD1 = tm, tD2 = tm + 32, tD3 = tm + 64;
  unsigned char *sS = smem + kOffS, *sU = smem + kOffU;

  // [W; Q.Gamma] is all MMA1 needs: it is fetched two chunks ahead, into its buffer's
  // region as soon as MMA1 of the chunk before has read it; the rest one chunk ahead.
  auto issue_xw = [&](int c, int b) {
    const char *blk = blocks + ((size_t)(chunk_base[n] + c) * H + h) * kBlockBytes;
    mbar_arrive_expect_tx(&s_xbar[b], 128 * kK * 2);
    bulk_g2s(smem + b * kBufBytes + kBufXW, blk + kOffXW, 128 * kK * 2, &s_xbar[b]);
  };
  auto issue_load = [&](int c, int b) {
    const char *blk = blocks + ((size_t)(chunk_base[n] + c) * H + h) * kBlockBytes;
    unsigned char *dst = smem + b * kBufBytes;
    mbar_arrive_expect_tx(&s_lbar[b], kK * kC * 2 + kC * kC * 2 + kC * kVT * 2 + kK * 4);
    bulk_g2s(dst + kBufBT, blk + kOffBT, kK * kC * 2, &s_lbar[b]);
    bulk_g2s(dst + kBufP0 + kC * kC * 2, blk + kOffP, kC * kC * 2, &s_lbar[b]);
    bulk_g2s(dst + kBufUP, blk + kOffUP + (size_t)vt * kC * kVT * 2, kC * kVT * 2, &s_lbar[b]);
    bulk_g2s(dst + kBufGC, blk + kOffGC, kK * 4, &s_lbar[b]);
  };
  auto issue_mma1 = [&](int b) {  // tid 0: D1 = [W; Q.Gamma] S0^T
    const unsigned char *buf = smem + b * kBufBytes;
#pragma unroll
    for (int ks = 0; ks < kK / 16; ++ks)
      tc::mma_bf16(tD1, tc::kmajor_desc(buf + kBufXW, kK, ks), tc::mnmajor_desc(sS, kVT, ks),
                   tc::idesc_bf16_bmn<128, kVT>(), ks > 0);
    tc::mma_commit(&s_bar1);
  };
  auto write_s0 = [&]() {  // S0 (bf16) as MMA1's MN-major B operand: element (v, k = tid)
#pragma unroll
    for (int q = 0; q < kVT / 8; ++q) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = S[8 * q + e];
      st16(sS + tc::mnmajor_offset(8 * q, tid, kVT), pack16(x));
    }
  };
  auto wait = [&](uint64_t *bar, uint32_t phase) {
    if (!mbar_wait(bar, phase)) s_fail = 1;
  };

  // Pipeline of one chunk c (buffer b = c & 1):
  //   wait MMA1(c) -> U = U' - W S0^T into shared memory (rows 0..63), keep the inter-chunk
  //   output (rows 64..127) -> barrier -> MMA2 (state) and MMA3 (intra-chunk output), each
  //   with its own commit; prefetch chunk c+1's operands -> state update, S1 into shared
  //   memory -> barrier -> MMA1(c+1) -> output of chunk c written while MMA1(c+1) runs.
  //   Waits on mbarriers are per thread and bounded; a failed one sets s_fail, which
  //   every thread reads after the next barrier, so all leave the loop together.
  // counts of requested [W; Q.Gamma] parts and rest parts (tid 0 issues; every thread
  // keeps the counts, which depend only on the loop position)
  int issued_x = 0, issued = 0;
  bool ok = true;
  if (nch > 0) {
    if (tid == 0) {
      issue_xw(0, 0);
      if (nch > 1) issue_xw(1, 1);
      issue_load(0, 0);
    }
    issued_x = nch > 1 ? 2 : 1;
    issued = 1;
    write_s0();
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
      wait(&s_xbar[0], 0);
      if (!s_fail) issue_mma1(0);
    }
  }
  int c = 0;
  for (; c < nch; ++c) {
    const int b = c & 1;
    const unsigned char *buf = smem + b * kBufBytes;
    const int t0 = start + kC * c, Lc = min(kC, end - t0);
    wait(&s_bar1, c & 1);
    tc::fence_after_sync();
    // MMA1(c) has read buffer b's [W; Q.Gamma]: refill it with chunk c+2's
    if (c + 2 < nch) {
      if (tid == 0) issue_xw(c + 2, b);
      issued_x = c + 3;
    }
    float d[kVT];
    {
      float d0[16], d1[16];
      tc::tmem_ld16(tc::tmem_addr(tD1, 32 * warp, 0), d0);
      tc::tmem_ld16(tc::tmem_addr(tD1, 32 * warp, 16), d1);
#pragma unroll
      for (int i = 0; i < 16; ++i) { d[i] = d0[i]; d[16 + i] = d1[i]; }
    }
    wait(&s_lbar[b], (c >> 1) & 1);  // the operand block is visible to this thread
    if (warp < 2) {
      // rows 0..63: U = U' - W S0^T as MMA2/3's MN-major B operand: element (v, r = tid)
      const int r = tid;
      const uint4 *up = reinterpret_cast<const uint4 *>(buf + kBufUP + (size_t)r * kVT * 2);
#pragma unroll
      for (int q = 0; q < kVT / 8; ++q) {
        float u8[8];
        unpack16(up[q], u8);
#pragma unroll
        for (int e = 0; e < 8; ++e) u8[e] = r < Lc ? u8[e] - d[8 * q + e] : 0.f;
        st16(sU + tc::mnmajor_offset(8 * q, r, kVT), pack16(u8));
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    if (s_fail) { ok = false; break; }
    tc::fence_after_sync();
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks)
        tc::mma_bf16(tD2, tc::kmajor_desc(buf + kBufBT, kC, ks), tc::mnmajor_desc(sU, kVT, ks),
                     tc::idesc_bf16_bmn<128, kVT>(), ks > 0);
      tc::mma_commit(&s_bar2);
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks)
        tc::mma_bf16(tD3, tc::kmajor_desc(buf + kBufP0, kC, ks), tc::mnmajor_desc(sU, kVT, ks),
                     tc::idesc_bf16_bmn<128, kVT>(), ks > 0);
      tc::mma_commit(&s_bar3);
    }
    // Every thread is past chunk c-1, so the rest of the other buffer is free for c+1.
    if (c + 1 < nch) {
      if (tid == 0) issue_load(c + 1, b ^ 1);
      issued = c + 2;
    }
    wait(&s_bar2, c & 1);
    tc::fence_after_sync();
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
    if (c + 1 < nch) {
      write_s0();
      tc::fence_smem_to_async();
    }
    float o[kVT];
    if (warp >= 2) {
      wait(&s_bar3, c & 1);
      tc::fence_after_sync();
      float d0[16], d1[16];
      tc::tmem_ld16(tc::tmem_addr(tD3, 32 * warp, 0), d0);
      tc::tmem_ld16(tc::tmem_addr(tD3, 32 * warp, 16), d1);
#pragma unroll
      for (int i = 0; i < 16; ++i) { o[i] = d[i] + d0[i]; o[16 + i] = d[16 + i] + d1[i]; }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (s_fail) { ok = false; break; }
    tc::fence_after_sync();
    if (c + 1 < nch && tid == 0) {
      wait(&s_xbar[b ^ 1], ((c + 1) >> 1) & 1);
      if (!s_fail) issue_mma1(b ^ 1);  // a failure here surfaces after the next barrier
    }
    if (warp >= 2) {
      // rows 64..127: O = (Q.Gamma) S0^T + P U of token r, written while MMA1(c+1) runs
      const int r = tid - kC;
      if (r < Lc) {
        IO *op = out + ((size_t)(t0 + r) * H + h) * V + (size_t)vt * kVT;
        constexpr int EPV = 16 / sizeof(IO);
#pragma unroll
        for (int q = 0; q < kVT / EPV; ++q) {
          float x[EPV];
#pragma unroll
          for (int e = 0; e < EPV; ++e) x[e] = o[EPV * q + e];
          st16(op + EPV * q, pack16(x));
        }
      }
    }
  }
  if (nch > 0 && s_fail) ok = false;
  if (!ok) {
    if (tid == 0) {
      flag_error(pv.err, RSC_DEVERR_TIMEOUT);
      // let every issued bulk copy land before the shared memory is released
      for (int k = c; k < issued_x; ++k) mbar_wait(&s_xbar[k & 1], (k >> 1) & 1);
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
                       const uint8_t *has_init, const void *qkv, const float *conv_w,
                       const float *g, const float *beta, void *out, int32_t *chunk_base,
                       char *blocks, cudaStream_t s) {
  auto chunk_kernel = prefill_tc_chunk_kernel<IO, V, GATE>;
  auto state_kernel = prefill_tc_state_kernel<IO, V>;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kChSmem) != cudaSuccess ||
        cudaFuncSetAttribute(state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStateSmem) != cudaSuccess)
      return RSC_ECUDA;
    attr = true;
  }
  const unsigned cap = (unsigned)prefill_tc_chunk_capacity(N, T);
  if (cap > 0 && T > 0) {
    chunk_kernel<<<dim3(cap, a.pv.H), 256, kChSmem, s>>>(a.pv, a.layer, slots, cu, chunk_base, N,
                                                          has_init, static_cast<const IO *>(qkv),
                                                          conv_w, g, beta, blocks);
    if (launch_status() != RSC_OK) return RSC_ECUDA;
  }
  state_kernel<<<dim3(V / kVT, a.pv.H, N), 128, kStateSmem, s>>>(
      a.pv, a.layer, slots, cu, chunk_base, T, has_init, blocks, static_cast<IO *>(out));
  return launch_status();
}

int launch_prefill_tc(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N, int T,
                      const uint8_t *has_init, const void *qkv, const float *conv_w,
                      const float *g, const float *beta, void *out, int32_t *chunk_base,
                      char *blocks, cudaStream_t s) {
  prefill_chunk_table_kernel<<<1, 32, 0, s>>>(cu, N, T, chunk_base, a.pv.err);
  if (launch_status() != RSC_OK) return RSC_ECUDA;
  const bool kda = a.gate == RSC_GATE_KDA;
#define RSC_TC(IO_, V_)                                                                        \
  (kda ? launch_tc_v<IO_, V_, RSC_GATE_KDA>(a, slots, cu, N, T, has_init, qkv, conv_w, g, beta, \
                                            out, chunk_base, blocks, s)                        \
       : launch_tc_v<IO_, V_, RSC_GATE_GDN>(a, slots, cu, N, T, has_init, qkv, conv_w, g, beta, \
                                            out, chunk_base, blocks, s))
  if (a.io == RSC_BF16) return a.pv.V == 128 ? RSC_TC(bf16, 128) : RSC_TC(bf16, 64);
  return a.pv.V == 128 ? RSC_TC(float, 128) : RSC_TC(float, 64);
#undef RSC_TC
}

}  // namespace rsc

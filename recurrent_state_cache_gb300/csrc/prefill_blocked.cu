// prefill_blocked.cu -- prefill of every pool the tensor-core form does not take (fp32 state,
// or head_k 64): the exact recurrence taken eight tokens at a time in closed form, in fp32.
//
// Sources: "SGLang之KV Cache内存池机制" §8.5 forward_extend (each sequence starts from its
// slot's state or from zero, the final state goes back to the slot; sequences packed by
// cu_seqlens) and "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理", ReplaySSM section
// (the recurrence over several tokens unrolled into one closed form from the first state).
//
// The closed form.  Within a block of tokens 0..c-1 of one sequence, with S0 the state
// before the block and Gam_t the cumulative log-decay from the block start up to and
// including token t (per key channel for KDA, per head for GDN):
//   S_{t-1} Diag(alpha_t) = S0 Diag(e^Gam_t) + sum_{s<t} d_s (k_s . e^(Gam_t - Gam_s))^T
// so every state row's u_t = a_t + sum_{s<t} A[t][s] d_s and o_t = b_t + sum_{s<=t} P[t][s] d_s
// with a_t = S0 (k_t . e^Gam_t), b_t = S0 (q_t . e^Gam_t), A[t][s] = sum_k k_s k_t e^(Gam_t - Gam_s)
// and P[t][s] = sum_k k_s q_t e^(Gam_t - Gam_s); d_t = beta_t (v_t - u_t) is then a forward
// substitution, and S_end = S0 Diag(e^Gam_end) + sum_s d_s (k_s . e^(Gam_end - Gam_s))^T.
// This is exact algebra: the result is the token-by-token recurrence up to rounding order.
//
// Three launches:
//   blk        grid (block, head): conv and L2 norms of the block's tokens, then its scaled
//              keys and queries, the end-scaled keys, e^Gam_end and the A / P rows, written
//              with beta and the values as one contiguous record per (block, head).  The
//              2 x 32 sums over channels are one butterfly reduce-scatter per warp and a
//              4-warp add (a shared-memory transpose instead costs the CTAs per SM that this
//              latency-bound kernel needs).
//   recurrent  grid (row tile, head, sequence): S in registers across the sequence; per
//              block the 16 row dots of every row (one butterfly reduce-scatter: 16 shuffles
//              where the token loop spends 80), the 8x8 forward substitution, the outputs
//              and the block-end state.  Each block's record is staged by two bulk copies
//              (TMA) from one thread, a few blocks ahead.
//   window     (prefill.cu) the slot's window becomes the sequence's last three inputs.
// Blocks start at each sequence start, so a sequence of n tokens has ceil(n / 8) blocks;
// block b of the grid belongs to the last sequence i with cu[i] / 8 + i <= b (these bases are
// strictly increasing and leave room for every block of each sequence).
#include "rsc_internal.h"
#include "rsc_step.cuh"

namespace rsc {

namespace {

constexpr int TS = 8;      // tokens per block
constexpr int NCO = 16;    // per token: its A row (8), then its P row (8)
constexpr float kMaxRise = 80.f;  // largest growth of a log gate within a block

// One record per (block, head) in the workspace, fp32, in the order the recurrence stages it:
// scaled keys (rows 0-7) and queries (rows 8-15) [16][K], end-scaled keys [8][K], e^Gam_end
// [K], the A rows then the P rows [8][16], beta [8] (+8 zero), then the values [V][8] (value
// channel-major, so a row tile's values are one contiguous run).  Rows past the sequence end
// are zero, which makes their deltas zero.
template <int K>
struct Rec {
  static constexpr int KQ = 0;
  static constexpr int KE = KQ + 2 * TS * K;
  static constexpr int EG = KE + TS * K;
  static constexpr int CO = EG + K;
  static constexpr int B = CO + TS * NCO;
  static constexpr int V = B + 2 * TS;  // also the floats of the shared part of a record
  static_assert((V * 4) % 16 == 0, "16-byte bulk copies");
  __host__ __device__ static constexpr int floats(int Vd) { return V + TS * Vd; }
};

// Pair indices of the 64 coefficient sums: A[t][s] (s < t) at t(t-1)/2 + s, then P[t][s]
// (s <= t) at 28 + t(t+1)/2 + s.
__host__ __device__ constexpr int ia(int t, int s) { return t * (t - 1) / 2 + s; }
__host__ __device__ constexpr int ip(int t, int s) { return 28 + t * (t + 1) / 2 + s; }

// Per (block, head): the conv of the head's q / k / v channels over the block's tokens (thread
// k owns key channel k when k < K and value channel k when k < V), the L2 norms of q and k,
// then the block's operands.  A thread reads its channels' 11 inputs once (3 before the
// block: the sequence, the slot's window before the sequence start, or zero for a fresh
// sequence) where a conv per token would read 32.
template <typename IO, int K, int V, int GATE>
__global__ void __launch_bounds__(128)
prefill_blk_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                   const int32_t *__restrict__ cu, int N, int T,
                   const uint8_t *__restrict__ has_init, const IO *__restrict__ qkv,
                   const float *__restrict__ conv_w, const float *__restrict__ g,
                   const float *__restrict__ beta, float *__restrict__ recs) {
  using L = Rec<K>;
  static_assert(K <= 128 && V <= 128, "a thread per channel");
  __shared__ float red[4][64];
  __shared__ float nrm[2 * TS];  // 1/|q_t|, 1/|k_t|
  const int b = blockIdx.x, h = blockIdx.y, k = threadIdx.x, lane = k & 31, warp = k >> 5;
  const int H = pv.H, D = pv.D;
  if (b == 0 && h == 0 && k == 0 && (cu[0] != 0 || cu[N] != T)) flag_error(pv.err, RSC_DEVERR_SEQ);
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] / TS + mid <= b) lo = mid; else hi = mid - 1;
  }
  const int start = cu[lo], end = cu[lo + 1];
  if (start < 0 || end < start || end > T) return;  // flagged by the recurrence
  const int t0 = start + TS * (b - (start / TS + lo));
  if (t0 < start || t0 >= end) return;
  const int cnt = min(TS, end - t0);
  const int slot = slots[lo];
  if (slot < 0 || slot > pv.P) return;  // flagged by the recurrence
  const bool init = has_init == nullptr || has_init[lo] != 0;
  const IO *W = reinterpret_cast<const IO *>(pv.conv) + ((size_t)layer * (pv.P + 1) + slot) * 3 * (size_t)D;
  float *rec = recs + ((size_t)b * H + h) * L::floats(V);

  auto conv_rows = [&](int c, float (&y)[TS]) {
    float x[TS + 3];  // inputs at tokens t0 - 3 .. t0 + 7 (oldest first)
#pragma unroll
    for (int i = 0; i < TS + 3; ++i) {
      const int pos = t0 - start + i - 3;  // position within the sequence
      x[i] = 0.f;
      if (i < cnt + 3)
        x[i] = pos >= 0 ? to_f32(qkv[(size_t)(start + pos) * D + c])
                        : (init ? to_f32(W[(size_t)(3 + pos) * D + c]) : 0.f);
    }
    const float4 wc = *reinterpret_cast<const float4 *>(conv_w + 4 * (size_t)c);
#pragma unroll
    for (int t = 0; t < TS; ++t) y[t] = t < cnt ? conv4(wc, x[t], x[t + 1], x[t + 2], x[t + 3]) : 0.f;
  };
  const bool key = k < K;  // this thread's key channel; threads past K add zeros
  float q[TS], kk[TS];
#pragma unroll
  for (int t = 0; t < TS; ++t) q[t] = kk[t] = 0.f;
  if (key) {
    conv_rows(h * K + k, q);
    conv_rows(H * K + h * K + k, kk);
  }
  if (k < V) {
    float y[TS];
    conv_rows(2 * H * K + h * V + k, y);
    float4 *dv = reinterpret_cast<float4 *>(rec + L::V + TS * k);
    dv[0] = make_float4(y[0], y[1], y[2], y[3]);
    dv[1] = make_float4(y[4], y[5], y[6], y[7]);
  }
  {
    float sq[2 * TS];  // |q_t|^2, then |k_t|^2, summed over the head's channels
#pragma unroll
    for (int t = 0; t < TS; ++t) {
      sq[t] = q[t] * q[t];
      sq[TS + t] = kk[t] * kk[t];
    }
    float v16 = group_reduce_scatter<2 * TS>(sq);  // lane i: entry i & 15 over its half-warp
    v16 += __shfl_xor_sync(0xffffffffu, v16, 16);
    if (lane < 2 * TS) red[warp][lane] = v16;
    __syncthreads();
    if (k < 2 * TS) nrm[k] = 1.0f / sqrtf(red[0][k] + red[1][k] + red[2][k] + red[3][k] + kNormEps);
    __syncthreads();
#pragma unroll
    for (int t = 0; t < TS; ++t) {
      q[t] *= nrm[t];
      kk[t] *= nrm[TS + t];
    }
  }

  // Decays alpha_t = e^(g_t) (1 past the sequence end); every factor e^(Gam_t - Gam_s) below
  // is a product of alphas, the token recurrence's own arithmetic, to at most 7 roundings.
  float al[TS];
  float acc = 0.f, low = 0.f, rise = 0.f;
#pragma unroll
  for (int t = 0; t < TS; ++t) {
    al[t] = 1.f;
    if (t < cnt && key) {
      const size_t th = (size_t)(t0 + t) * H + h;
      const float gt = GATE == RSC_GATE_KDA ? g[th * K + k] : g[th];
      al[t] = expf(gt);
      acc += gt;
      rise = fmaxf(rise, acc - low);
      low = fminf(low, acc);
    }
  }
  if (rise > kMaxRise) flag_error(pv.err, RSC_DEVERR_GATE);
  float eg[TS], ee[TS];  // e^Gam_t, e^(Gam_end - Gam_t)
  {
    float f = 1.f, b2 = 1.f;
#pragma unroll
    for (int t = 0; t < TS; ++t) { f *= al[t]; eg[t] = f; }
#pragma unroll
    for (int t = TS - 1; t >= 0; --t) { ee[t] = b2; b2 *= al[t]; }
  }
  if (key) {
#pragma unroll
    for (int t = 0; t < TS; ++t) {  // zero past the sequence end: q, k are
      rec[L::KQ + t * K + k] = kk[t] * eg[t];
      rec[L::KQ + (TS + t) * K + k] = q[t] * eg[t];
      rec[L::KE + t * K + k] = kk[t] * ee[t];
    }
    rec[L::EG + k] = eg[TS - 1];
  }
  if (k < 2 * TS) rec[L::B + k] = k < cnt ? beta[(size_t)(t0 + k) * H + h] : 0.f;

  // this channel's terms of the 64 sums (rows t >= cnt come out zero: their q, k are zero)
  float x[64];
#pragma unroll
  for (int s2 = 0; s2 < TS; ++s2) {
    x[ip(s2, s2)] = kk[s2] * q[s2];
    float f = kk[s2];
#pragma unroll
    for (int t = s2 + 1; t < TS; ++t) {
      f *= al[t];  // k_s e^(Gam_t - Gam_s)
      x[ia(t, s2)] = f * kk[t];
      x[ip(t, s2)] = f * q[t];
    }
  }
  float lo32[32], hi32[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) { lo32[i] = x[i]; hi32[i] = x[32 + i]; }
  red[warp][lane] = group_reduce_scatter<32>(lo32);
  red[warp][32 + lane] = group_reduce_scatter<32>(hi32);
  __syncthreads();
  static_assert(TS * NCO == 128, "a thread per coefficient");
  {
    const int t = k / NCO, c = k % NCO;
    float v = 0.f;
    if (c < TS) {
      if (c < t) { const int e = ia(t, c); v = red[0][e] + red[1][e] + red[2][e] + red[3][e]; }
    } else if (c - TS <= t) {
      const int e = ip(t, c - TS);
      v = red[0][e] + red[1][e] + red[2][e] + red[3][e];
    }
    rec[L::CO + k] = v;  // rows past the end: zero sums
  }
}

// One stage of block operands in shared memory: the record's shared part and this tile's
// values, each one bulk copy.
template <int K, int VT>
struct Stage {
  float rec[Rec<K>::V];
  float v[VT][TS];  // values of the tile's rows, [row][token]
};

// E consecutive fp32 values (E = 2 or 4, 8- or 16-byte aligned) as E/2 pairs.
template <int E>
__device__ __forceinline__ void ld_pairs(const float *p, float2 (&d)[E / 2]) {
  if constexpr (E == 4) {
    const float4 x = *reinterpret_cast<const float4 *>(p);
    d[0] = make_float2(x.x, x.y);
    d[1] = make_float2(x.z, x.w);
  } else {
    d[0] = *reinterpret_cast<const float2 *>(p);
  }
}
// A lane's E state entries in the state dtype.
template <typename ST, int E>
__device__ __forceinline__ void ld_state(const ST *p, float2 (&d)[E / 2]) {
  if constexpr (sizeof(ST) == 4) {
    ld_pairs<E>(reinterpret_cast<const float *>(p), d);
  } else if constexpr (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    d[0] = make_float2(bf16lo(u.x), bf16hi(u.x));
    d[1] = make_float2(bf16lo(u.y), bf16hi(u.y));
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
    d[0] = make_float2(bf16lo(u), bf16hi(u));
  }
}
template <typename ST, int E>
__device__ __forceinline__ void st_state(ST *p, const float2 (&d)[E / 2]) {
  if constexpr (sizeof(ST) == 4) {
    if constexpr (E == 4)
      st16_stream(p, make_uint4(__float_as_uint(d[0].x), __float_as_uint(d[0].y),
                                __float_as_uint(d[1].x), __float_as_uint(d[1].y)));
    else
      *reinterpret_cast<float2 *>(p) = d[0];
  } else if constexpr (E == 4) {
    *reinterpret_cast<uint2 *>(p) =
        make_uint2(pack_bf16x2(d[0].x, d[0].y), pack_bf16x2(d[1].x, d[1].y));
  } else {
    *reinterpret_cast<uint32_t *>(p) = pack_bf16x2(d[0].x, d[0].y);
  }
}

// One CTA: rows [j VT, (j+1) VT) of head h of sequence n's state, VT = NW R: NW warps of R
// rows each, a row across a whole warp (lane i holds key channels E i .. E i + E - 1, E =
// K / 32).  Thread 0 stages each block's record with two bulk copies (TMA) NS - 1 blocks
// ahead, completing on that stage's mbarrier.  Per block a lane loads its channels of the
// block's scaled keys, queries and end-scaled keys into registers once and applies them to
// its R rows.  Per row: the 16 row dots, one butterfly reduce-scatter (lane t then holds a_t,
// lane 8+t holds b_t), the 8 a's gathered, the forward substitution, o_t written by lane 8+t,
// the row moved to the block end.  The state stays in fp32 registers for the whole call and
// is rounded to the state dtype once, at the end.
template <typename ST, typename IO, int K, int V, int NW, int R, int NS>
__global__ void __launch_bounds__(32 * NW)
prefill_blocked_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                       const int32_t *__restrict__ cu, int T, const uint8_t *__restrict__ has_init,
                       const float *__restrict__ recs, IO *__restrict__ out) {
  using L = Rec<K>;
  constexpr int VT = NW * R, E = K / 32, E2 = E / 2;
  constexpr uint32_t kBytesRec = L::V * 4, kBytesV = VT * TS * 4;
  static_assert(V % VT == 0 && kBytesV % 16 == 0 && (E == 2 || E == 4), "row tile, lanes");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Stage<K, VT> *stg = reinterpret_cast<Stage<K, VT> *>(smem_raw);
  __shared__ __align__(8) uint64_t s_bar[NS];

  const int j = blockIdx.x, h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5, k0 = E * lane;
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
  float2 s[R][E2];  // rows warp R + p, channels k0 .. k0 + E - 1
#pragma unroll
  for (int p = 0; p < R; ++p) {
    if (init) {
      ld_state<ST, E>(S + (size_t)(warp * R + p) * K + k0, s[p]);
    } else {
#pragma unroll
      for (int e = 0; e < E2; ++e) s[p][e] = make_float2(0.f, 0.f);
    }
  }

  const int nb = (end - start + TS - 1) / TS;
  const float *rec0 = recs + ((size_t)(start / TS + n) * H + h) * L::floats(V);
  auto issue = [&](int i) {  // thread 0: block i of the sequence into stage i % NS
    Stage<K, VT> &st = stg[i % NS];
    const float *rec = rec0 + (size_t)i * H * L::floats(V);
    mbar_arrive_expect_tx(&s_bar[i % NS], kBytesRec + kBytesV);
    bulk_g2s(st.rec, rec, kBytesRec, &s_bar[i % NS]);
    bulk_g2s(st.v, rec + L::V + (size_t)j * VT * TS, kBytesV, &s_bar[i % NS]);
  };
  int issued = 0;
  if (tid == 0) {
    for (int b = 0; b < NS; ++b) mbar_init(&s_bar[b], 1);
    for (; issued < NS - 1 && issued < nb; ++issued) issue(issued);
  }
  __syncthreads();

  const int to = lane & 7;  // lanes 8-15 end with b_to
  const int perm = lane & 15;
  bool ok = true;
  int i = 0;
  for (; i < nb; ++i) {
    // block i landed; everyone is done with the stage of block i - 1
    ok = __syncthreads_and(mbar_wait(&s_bar[i % NS], (i / NS) & 1));
    if (!ok) break;
    if (tid == 0 && issued < nb) issue(issued++);
    const Stage<K, VT> &st = stg[i % NS];
    const float *rc = st.rec;
    const int t0 = start + i * TS, cnt = min(TS, end - t0);
    float A[TS][TS], bt[TS], Pr[TS];  // 16-byte loads: A rows, beta, this lane's P row
    auto ld = [](const float *p, float *d) {
      const float4 x = *reinterpret_cast<const float4 *>(p);
      d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
    };
    ld(rc + L::B, bt);
    ld(rc + L::B + 4, bt + 4);
    ld(rc + L::CO + to * NCO + TS, Pr);  // P[to][t]
    ld(rc + L::CO + to * NCO + TS + 4, Pr + 4);
#pragma unroll
    for (int t = 1; t < TS; ++t) {
      ld(rc + L::CO + t * NCO, A[t]);
      if (t > 4) ld(rc + L::CO + t * NCO + 4, A[t] + 4);
    }
    // Slot q of this lane holds operand row q ^ (lane & 15) (a scaled key for rows < 8, a
    // scaled query above): then at every level of the reduce-scatter below the values this
    // lane keeps sit in the lower slots and the ones it hands over in the upper slots, for
    // every lane, so the butterfly needs no per-lane selects.
    float2 kq[2 * TS][E2], ke[TS][E2], eg[E2];
#pragma unroll
    for (int q = 0; q < 2 * TS; ++q) ld_pairs<E>(rc + L::KQ + (q ^ perm) * K + k0, kq[q]);
#pragma unroll
    for (int t = 0; t < TS; ++t) ld_pairs<E>(rc + L::KE + t * K + k0, ke[t]);
    ld_pairs<E>(rc + L::EG + k0, eg);
#pragma unroll
    for (int p = 0; p < R; ++p) {
      const int row = warp * R + p;
      float x[2 * TS];  // x[q]: this lane's part of the dot with operand row q ^ perm
#pragma unroll
      for (int q = 0; q < 2 * TS; ++q) {
        float2 u = __fmul2_rn(s[p][0], kq[q][0]);
#pragma unroll
        for (int e = 1; e < E2; ++e) u = __ffma2_rn(s[p][e], kq[q][e], u);
        x[q] = u.x + u.y;
      }
#pragma unroll
      for (int m = TS; m >= 1; m >>= 1)
#pragma unroll
        for (int q = 0; q < m; ++q) x[q] += __shfl_xor_sync(0xffffffffu, x[q + m], m);
      // lane q (and q + 16) now holds the whole dot with row q: a_q for q < 8, b_(q-8) above
      const float val = x[0] + __shfl_xor_sync(0xffffffffu, x[0], 16);
      float r[TS], d[TS];
      ld(st.v[row], r);
      ld(st.v[row] + 4, r + 4);
#pragma unroll
      for (int t = 0; t < TS; ++t) r[t] -= __shfl_sync(0xffffffffu, val, t);
#pragma unroll
      for (int u = 0; u < TS; ++u) {
        d[u] = bt[u] * r[u];
#pragma unroll
        for (int t = u + 1; t < TS; ++t) r[t] = fmaf(-A[t][u], d[u], r[t]);
      }
      if (lane >= TS && lane < 2 * TS && to < cnt) {
        float o = val;
#pragma unroll
        for (int u = 0; u < TS; ++u) o = fmaf(Pr[u], d[u], o);
        out[((size_t)(t0 + to) * H + h) * V + (size_t)j * VT + row] = from_f32<IO>(o);
      }
#pragma unroll
      for (int e = 0; e < E2; ++e) s[p][e] = __fmul2_rn(s[p][e], eg[e]);
#pragma unroll
      for (int u = 0; u < TS; ++u) {
        const float2 du = make_float2(d[u], d[u]);
#pragma unroll
        for (int e = 0; e < E2; ++e) s[p][e] = __ffma2_rn(du, ke[u][e], s[p][e]);
      }
    }
  }
  if (!ok) {
    if (tid == 0) {
      flag_error(pv.err, RSC_DEVERR_TIMEOUT);
      // let every requested bulk copy land before the shared memory is released
      for (int k = i; k < issued; ++k) mbar_wait(&s_bar[k % NS], (k / NS) & 1);
    }
    return;  // the slot's rows stay as they were
  }
#pragma unroll
  for (int p = 0; p < R; ++p) st_state<ST, E>(S + (size_t)(warp * R + p) * K + k0, s[p]);
}

#ifndef RSC_BLK_STAGES
#define RSC_BLK_STAGES 3
#endif

template <typename ST, typename IO, int K, int V, int NW, int R>
int run_blocked(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N, int T,
                const uint8_t *has_init, const float *recs, void *out, cudaStream_t s) {
  constexpr int VT = NW * R, NS = RSC_BLK_STAGES;
  static_assert(NS >= 2 && sizeof(Stage<K, VT>) % 16 == 0, "stages");
  constexpr size_t smem = NS * sizeof(Stage<K, VT>);
  auto *kern = prefill_blocked_kernel<ST, IO, K, V, NW, R, NS>;
  static PerDeviceFlag attr;
  const int rc = once_per_device(attr, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
                   cudaSuccess
               ? RSC_OK
               : RSC_ECUDA;
  });
  if (rc != RSC_OK) return rc;
  kern<<<dim3(V / VT, a.pv.H, N), 32 * NW, smem, s>>>(a.pv, a.layer, slots, cu, T, has_init, recs,
                                                      static_cast<IO *>(out));
  return launch_status();
}

// Row tiles: few (sequence, head) pairs get small tiles so that the grid still spreads over
// the GPU; many get wide ones (fewer copies of each block's operands staged).
#ifndef RSC_BLOCKED_MIN_CTAS
#define RSC_BLOCKED_MIN_CTAS 304
#endif
#ifndef RSC_BLK_SMALL_NW
#define RSC_BLK_SMALL_NW 2
#endif
#ifndef RSC_BLK_SMALL_R
#define RSC_BLK_SMALL_R 2
#endif
#ifndef RSC_BLK_WIDE_NW
#define RSC_BLK_WIDE_NW 4
#endif
#ifndef RSC_BLK_WIDE_R
#define RSC_BLK_WIDE_R 8
#endif

template <typename ST, typename IO, int K, int V, int GATE>
struct BlockedLaunch {
  static int run(const LayerArgs *a, const int32_t *slots, const int32_t *cu, int N, int T,
                 const uint8_t *has_init, const void *qkv, const float *conv_w, const float *g,
                 const float *beta, void *out, float *recs, cudaStream_t s) {
    if (T > 0) {
      prefill_blk_kernel<IO, K, V, GATE><<<dim3((unsigned)(T / TS + N), a->pv.H), 128, 0, s>>>(
          a->pv, a->layer, slots, cu, N, T, has_init, static_cast<const IO *>(qkv), conv_w, g,
          beta, recs);
      if (launch_status() != RSC_OK) return RSC_ECUDA;
    }
    const long wide = (long)(V / 32) * a->pv.H * N;
    const int rc =
        wide >= RSC_BLOCKED_MIN_CTAS
            ? run_blocked<ST, IO, K, V, RSC_BLK_WIDE_NW, RSC_BLK_WIDE_R>(*a, slots, cu, N, T,
                                                                          has_init, recs, out, s)
            : run_blocked<ST, IO, K, V, RSC_BLK_SMALL_NW, RSC_BLK_SMALL_R>(*a, slots, cu, N, T,
                                                                            has_init, recs, out, s);
    if (rc != RSC_OK) return rc;
    return launch_prefill_window(*a, slots, cu, N, T, has_init, qkv, s);
  }
};

}  // namespace

// Blocks of the grid: sequence i's ceil(len_i / 8) blocks start at floor(cu[i] / 8) + i, so
// floor(T / 8) + N records per head cover every block.
size_t prefill_blocked_bytes(const PoolView &pv, int N, int T) {
  const size_t rec = pv.K == 64 ? Rec<64>::floats(pv.V) : Rec<128>::floats(pv.V);
  return ((size_t)T / TS + N) * pv.H * rec * 4;
}

int launch_prefill_blocked(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N,
                           int T, const uint8_t *has_init, const void *qkv,
                           const float *conv_w, const float *g, const float *beta, void *out,
                           void *ws, cudaStream_t s) {
  float *recs = static_cast<float *>(ws);
  if (a.st == RSC_F32)
    return a.io == RSC_F32
               ? dispatch_k<BlockedLaunch, float, float>(a.pv.K, a.pv.V, a.gate, &a, slots, cu, N,
                                                          T, has_init, qkv, conv_w, g, beta, out,
                                                          recs, s)
               : dispatch_k<BlockedLaunch, float, bf16>(a.pv.K, a.pv.V, a.gate, &a, slots, cu, N,
                                                         T, has_init, qkv, conv_w, g, beta, out,
                                                         recs, s);
  // bf16 state: head_k 64 here, head_k 128 takes the tensor-core form
  if (a.pv.K != 64) return RSC_EDTYPE;
  return a.io == RSC_F32
             ? dispatch_v<BlockedLaunch, bf16, float, 64>(a.pv.V, a.gate, &a, slots, cu, N, T,
                                                          has_init, qkv, conv_w, g, beta, out,
                                                          recs, s)
             : dispatch_v<BlockedLaunch, bf16, bf16, 64>(a.pv.V, a.gate, &a, slots, cu, N, T,
                                                         has_init, qkv, conv_w, g, beta, out,
                                                         recs, s);
}

}  // namespace rsc

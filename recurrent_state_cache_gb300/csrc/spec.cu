// spec.cu -- speculative verify (T tokens per request, every intermediate state and
// window saved) and commit (the accepted entry gathered back into the slot).
//
// Source: "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理", speculative-decoding
// conv-state section: the verify pass stores the conv window after each token into a
// per-step cache and the commit scatters the snapshot of the last accepted step into
// the persistent state; the intermediate SSM cache does the same for S.
//
// VERIFY runs the delta rule T times with the state tile held in registers (fp32) across
// tokens; the slot is only read.  The per-token inputs (q/k channels of the head, the
// tile's value channels, gate, beta) are staged into shared memory eight tokens at a
// time with cp.async, one block ahead; conv, L2 norms and exp(g) of a whole block are
// computed before its token loop, so that loop has no barrier and never waits on HBM.  Each CTA keeps its own copy
// of the head's q/k windows plus its value rows' windows in registers and rolls them
// token by token, so no CTA ever writes memory another one reads: no cluster needed.
// Each window channel of a cache entry is written by exactly one CTA (q/k channels
// partitioned over the NVT tiles of the head, value channels by tile), each S entry
// tile by its owner.
//
// REPLAY (ReplaySSM, same page, ReplaySSM section): the same pass, but instead of S_t each
// token leaves its records in the slot's rings at entry (pos + t) mod depth: the delta d
// (rows of the tile, by their owner), the normalised key, the pre-norm key (the CTA owning
// the key channels' windows), the log-decay and beta (tile 0).  No intermediate state is
// stored, so the token loop is replaced by a closed form per block of eight tokens (every
// row's outputs and deltas from the tile at the block start: 16 independent row dots, one
// butterfly reduction, an 8x8 triangular solve; see replay_block), on a whole head per CTA.
// COMMIT of the replay path replays the accepted tokens from the slot state out of those
// records.
#include "rsc_internal.h"
#include "rsc_step.cuh"
#include "rsc_tc.cuh"

namespace rsc {

// Replay commit: 64 state rows and 4 warps per CTA, compiled for 4 resident CTAs per SM (128
// registers); measured 23.8 against 25.3 us with a whole head per CTA.  At accept 0 / 7 for
// every request: 15.0 / 27.0 us; 32-row tiles at 6 or 7 CTAs per SM 14.3-14.8 / 29.0; 64 rows at
// 3 CTAs per SM 17.4 / 29.5.
#ifndef RSC_COMMIT_ROWS
#define RSC_COMMIT_ROWS 64
#endif
#ifndef RSC_COMMIT_WARPS
#define RSC_COMMIT_WARPS 4
#endif
#ifndef RSC_COMMIT_MINB
#define RSC_COMMIT_MINB 4
#endif
// Snapshot verify: a whole head per CTA (8 warps) compiled for 2 resident CTAs per SM (128
// registers).  B=64, T=8, H=12: 51.0 us; 64 rows x 4 warps 63.9 us unbounded (168 registers,
// 3 CTAs per SM) and 61.4 us at 4 CTAs per SM; a whole head at 1 CTA per SM 66.5 us; a whole
// head on 16 warps 81 us at 1 or 2 CTAs per SM.
#ifndef RSC_SNAPSHOT_ROWS
#define RSC_SNAPSHOT_ROWS 128
#endif
#ifndef RSC_SNAPSHOT_WARPS
#define RSC_SNAPSHOT_WARPS 8
#endif
#ifndef RSC_SNAPSHOT_MINB
#define RSC_SNAPSHOT_MINB 2
#endif
// Record-mode verify: state rows and warps per CTA (rows = 16 x warps, so that the block's
// row dots reduce to one value per lane), and the resident CTAs it is compiled for.  A whole
// head per CTA does the head's conv, norms, records and coefficients once instead of once
// per row tile.
#ifndef RSC_REPLAY_ROWS
#define RSC_REPLAY_ROWS 128
#endif
#ifndef RSC_REPLAY_WARPS
#define RSC_REPLAY_WARPS 8
#endif
#ifndef RSC_REPLAY_MINB
#define RSC_REPLAY_MINB 2
#endif

template <typename ST, typename IO, int K, int V, int NVT, int NW, int GATE, bool REPLAY>
__global__ void __launch_bounds__(NW * 32, REPLAY ? RSC_REPLAY_MINB * RSC_REPLAY_WARPS / NW
                                                   : RSC_SNAPSHOT_MINB)
kda_spec_verify_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots, int T,
                       int L, ST *__restrict__ spec_ssm, IO *__restrict__ spec_conv,
                       const IO *__restrict__ qkv, const float *__restrict__ conv_w,
                       const float *__restrict__ g, const float *__restrict__ beta,
                       IO *__restrict__ out, RingView rv, const int32_t *__restrict__ pos) {
  constexpr int VT = V / NVT;
  // one 16-byte vector per lane and pass (two were measured slower: 109 vs 66 us at the
  // speculative workload)
  constexpr int VPL = 1;
  constexpr int NT = NW * 32;
  using G = TileGeom<ST, K, VT, NW, VPL>;
  constexpr int QK_T = (2 * K + NT - 1) / NT;
  constexpr int OWN = 2 * K / NVT;
  constexpr int TS = 8;                       // tokens per staged block
  constexpr int GW = GATE == RSC_GATE_KDA ? K : 1;
  constexpr int XV = 16 / sizeof(IO);         // io elements per 16-byte copy
  static_assert((2 * K) % XV == 0 && VT % XV == 0, "16-byte staging");
  static_assert(VT <= NT, "one value row per thread");

  // Per-token inputs of TS tokens, double-buffered: this head's q/k channels, this tile's
  // value channels, the gate and beta.  Staged with cp.async one block ahead.
  __shared__ __align__(16) IO s_xqk[2][TS][2 * K];
  __shared__ __align__(16) IO s_xv[2][TS][VT];
  __shared__ __align__(16) float s_g[2][TS][GW];
  __shared__ float s_b[2][TS];
  // Per-token operands of the current block, computed before its token loop: q_hat then
  // k_hat (in place of the conv outputs), the value rows, alpha = exp(g), k_hat . q_hat.
  __shared__ __align__(16) float s_qk[TS][2 * K];
  __shared__ float s_v[TS][VT];
  __shared__ __align__(16) float s_al[REPLAY ? 1 : TS][GW];
  __shared__ float s_kq[TS];
  // Record mode only (the block in closed form, see below): cumulative log-decays of the
  // block G_t, the decayed keys and queries k_hat_t . e^G_t and q_hat_t . e^G_t, the keys
  // decayed to the block's last token k_hat_t . e^(G_last - G_t), and the coefficients
  // A[t][s] = sum_k k_hat_s k_hat_t e^(G_t - G_s), P[t][s] = sum_k k_hat_s q_hat_t e^(G_t - G_s).
  constexpr int RS = REPLAY ? TS : 1;
  __shared__ __align__(16) float s_G[RS][GW];
  __shared__ __align__(16) float s_kk[RS][K];
  __shared__ __align__(16) float s_qq[RS][K];
  __shared__ __align__(16) float s_c[RS][K];
  __shared__ float s_A[RS][TS], s_P[RS][TS];
  __shared__ float s_d[RS][VT];  // the block's deltas by row, for the tile update at its end

  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = pv.H, D = pv.D;

  const int slot = slots[b];
  if (slot < 0 || slot > pv.P) {
    if (tid == 0 && j == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_SLOT);
    return;
  }
  const size_t prow = (size_t)layer * (pv.P + 1) + slot;
  int p0 = 0;  // ring entry of token 0 (replay)
  if constexpr (REPLAY) {
    p0 = pos[b];
    if (p0 < 0 || p0 >= rv.depth) {
      if (tid == 0 && j == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_RING);
      return;
    }
  }
  // ring entry of token t of this (layer, slot, head)
  auto ent = [&](int t) { return (prow * H + h) * (size_t)rv.depth + ((p0 + t) & (rv.depth - 1)); };

  auto stage = [&](int buf, int t0) {
    const int cnt = min(TS, T - t0);
    for (int i = tid; i < cnt * (2 * K / XV); i += NT) {
      const int tau = i / (2 * K / XV), c = (i % (2 * K / XV)) * XV;
      const int src = c < K ? h * K + c : H * K + h * K + (c - K);
      cp_async16(&s_xqk[buf][tau][c], qkv + ((size_t)b * T + t0 + tau) * D + src);
    }
    for (int i = tid; i < cnt * (VT / XV); i += NT) {
      const int tau = i / (VT / XV), c = (i % (VT / XV)) * XV;
      cp_async16(&s_xv[buf][tau][c],
                 qkv + ((size_t)b * T + t0 + tau) * D + 2 * H * K + h * V + j * VT + c);
    }
    if (GATE == RSC_GATE_KDA) {
      for (int i = tid; i < cnt * (K / 4); i += NT) {
        const int tau = i / (K / 4), c = (i % (K / 4)) * 4;
        cp_async16(&s_g[buf][tau][c], g + (((size_t)b * T + t0 + tau) * H + h) * K + c);
      }
    } else if (tid < cnt) {
      cp_async4(&s_g[buf][tid][0], g + ((size_t)b * T + t0 + tid) * H + h);
    }
    if (tid < cnt) cp_async4(&s_b[buf][tid], beta + ((size_t)b * T + t0 + tid) * H + h);
    cp_async_commit();
  };
  stage(0, 0);

  const ST *S = reinterpret_cast<const ST *>(pv.ssm) + ((prow * H + h) * V + (size_t)j * VT) * K;
  Tile2<ST, K, VT, NW, VPL> s;
  tile_load2<ST, K, VT, VPL, NW>(S, s);

  // Window registers (raw io values, row 0 oldest) and taps of this thread's channels.
  const IO *W = reinterpret_cast<const IO *>(pv.conv) + prow * 3 * (size_t)D;
  IO win[QK_T][3];
  float4 wt[QK_T];
  int cqk[QK_T];
#pragma unroll
  for (int u = 0; u < QK_T; ++u) {
    const int i2 = tid + u * NT;
    cqk[u] = i2 < K ? h * K + i2 : H * K + h * K + (i2 - K);
    if (i2 < 2 * K) {
      wt[u] = *reinterpret_cast<const float4 *>(conv_w + 4 * (size_t)cqk[u]);
      win[u][0] = W[cqk[u]]; win[u][1] = W[D + cqk[u]]; win[u][2] = W[2 * D + cqk[u]];
    }
  }
  IO winv[3];
  float4 wtv = make_float4(0.f, 0.f, 0.f, 0.f);
  const int cv = 2 * H * K + h * V + j * VT + tid;
  if (tid < VT) {
    wtv = *reinterpret_cast<const float4 *>(conv_w + 4 * (size_t)cv);
    winv[0] = W[cv]; winv[1] = W[D + cv]; winv[2] = W[2 * D + cv];
  }

  const int k0 = G::kofs();
  int cur = 0;

  // Record mode: the block's tokens in closed form.  With G_t the cumulative log-decay from
  // the block start and S0 the tile at the block start,
  //   S_{t-1} Diag(alpha_t) = S0 Diag(e^G_t) + sum_{s<t} d_s (k_hat_s . e^(G_t - G_s))^T,
  // so every row's u_t = a_t + sum_{s<t} A[t][s] d_s with a_t = S0 (k_hat_t . e^G_t), and
  // o_t = S_t q_hat_t = b_t + sum_{s<=t} P[t][s] d_s with b_t = S0 (q_hat_t . e^G_t).  The 2 TS
  // row dots of the block are independent of each other (one butterfly reduction for all
  // of them instead of two per token), then d_t = beta_t (v_t - u_t) is an 8x8 triangular
  // solve per row.  The tile itself changes only at the block end, if another block follows:
  //   S <- S0 Diag(e^G_last) + sum_s d_s (k_hat_s . e^(G_last - G_s))^T.
  auto replay_block = [&](int t0, int cnt) {
    constexpr int LPR = G::LPR, NP = G::NP, E2 = G::EPL / 2;
    static_assert(!REPLAY || 2 * NP == LPR, "the reduction leaves one value per lane");
    const bool more = t0 + TS < T;
    auto gk = [](int k) { return GW == 1 ? 0 : k; };
    // exponentials of log-decay sums over at most eight tokens (arguments of moderate size,
    // non-positive for decaying gates): the fast intrinsic, ~1e-6 relative
    for (int i = tid; i < cnt * K; i += NT) {
      const int tau = i / K, k = i % K;
      const float Gt = s_G[tau][gk(k)];
      const float e = __expf(Gt);
      s_kk[tau][k] = s_qk[tau][K + k] * e;
      s_qq[tau][k] = s_qk[tau][k] * e;
      if (more) s_c[tau][k] = s_qk[tau][K + k] * __expf(s_G[cnt - 1][gk(k)] - Gt);
    }
    {
      // the pairs (t, s), s < t, PPW per warp (pair PPW warp + i) over all warps; a lane
      // covers CPL consecutive channels of one half of K (lanes 0-15 the first half, 16-31
      // the second), so a warp's shared-memory reads are contiguous
      constexpr int PPW = NW >= 7 ? 4 : 8;
      static_assert(!REPLAY || NW * PPW >= TS * (TS - 1) / 2, "pairs per warp");
      constexpr int CPL = K / 32;
      static_assert(CPL == 2 || CPL == 4, "channels per lane");
      const int c0 = (lane >> 4) * (K / 2) + CPL * (lane & 15);
      auto ldv = [&](const float *p, float (&v)[CPL]) {
        if constexpr (CPL == 4) {
          const float4 u = *reinterpret_cast<const float4 *>(p);
          v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
        } else {
          const float2 u = *reinterpret_cast<const float2 *>(p);
          v[0] = u.x; v[1] = u.y;
        }
      };
      auto pair_of = [](int pi, int &t, int &s2) {
        t = 1;
        while (t * (t + 1) / 2 <= pi) ++t;
        s2 = pi - t * (t - 1) / 2;
      };
      float x[2 * PPW];  // A of the warp's pairs, then P
#pragma unroll
      for (int i = 0; i < PPW; ++i) {
        int t, s2;
        pair_of(PPW * warp + i, t, s2);
        float a = 0.f, p = 0.f;
        if (PPW * warp + i < TS * (TS - 1) / 2 && t < cnt) {  // uniform over the warp
          float ks[CPL], kt[CPL], qt[CPL], gt[CPL], gs[CPL];
          ldv(&s_qk[s2][K + c0], ks);
          ldv(&s_qk[t][K + c0], kt);
          ldv(&s_qk[t][c0], qt);
          if constexpr (GW == 1) {
#pragma unroll
            for (int e = 0; e < CPL; ++e) { gt[e] = s_G[t][0]; gs[e] = s_G[s2][0]; }
          } else {
            ldv(&s_G[t][c0], gt);
            ldv(&s_G[s2][c0], gs);
          }
#pragma unroll
          for (int e = 0; e < CPL; ++e) {
            const float kd = ks[e] * __expf(gt[e] - gs[e]);
            a = fmaf(kd, kt[e], a);
            p = fmaf(kd, qt[e], p);
          }
        }
        x[i] = a;
        x[PPW + i] = p;
      }
      // the 2 PPW sums over each half's 16 lanes, then over the two halves
      float r;
      if constexpr (PPW == 8) {
        r = group_reduce_scatter<16>(x);
      } else {
        float y[2 * PPW];
#pragma unroll
        for (int i = 0; i < 2 * PPW; ++i) y[i] = x[i] + __shfl_xor_sync(0xffffffffu, x[i], 8);
        r = group_reduce_scatter<2 * PPW>(y);
      }
      r += __shfl_xor_sync(0xffffffffu, r, 16);
      if (lane < 2 * PPW) {  // lane i: entry i (A of pair i, then P of pair i - PPW)
        const int i = lane % PPW;
        int t, s2;
        pair_of(PPW * warp + i, t, s2);
        if (PPW * warp + i < TS * (TS - 1) / 2 && t < cnt) (lane < PPW ? s_A : s_P)[t][s2] = r;
      }
    }
    __syncthreads();
    // the row dots: lane i of a row group ends with entry i, a_t of pass i (i < NP) or b_t
    // of pass i - NP
    const int li = lane & (LPR - 1);
    const bool is_a = li < NP;
    const int row = G::row(is_a ? li : li - NP);
    float val[TS];
#pragma unroll
    for (int t = 0; t < TS; ++t) {
      val[t] = 0.f;
      if (t < cnt) {
        float2 kv[E2], qv[E2];
#pragma unroll
        for (int e = 0; e < E2; ++e) {
          kv[e] = *reinterpret_cast<const float2 *>(&s_kk[t][k0 + 2 * e]);
          qv[e] = *reinterpret_cast<const float2 *>(&s_qq[t][k0 + 2 * e]);
        }
        // first butterfly level (lanes NP apart) as each pass's pair of dots completes,
        // so the 2 NP partials never live at once: lanes with bit NP keep the b half
        float y[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          float2 u = make_float2(0.f, 0.f), w = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < E2; ++e) {
            u = __ffma2_rn(s[p][e], kv[e], u);
            w = __ffma2_rn(s[p][e], qv[e], w);
          }
          const float pa = u.x + u.y, pb = w.x + w.y;
          y[p] = (is_a ? pa : pb) + __shfl_xor_sync(0xffffffffu, is_a ? pb : pa, NP);
        }
        val[t] = group_reduce_scatter<NP>(y);
      }
    }
    // deltas (meaningful on the a lanes), then handed to the b lane of the same row
    float d[TS];
#pragma unroll
    for (int t = 0; t < TS; ++t) {
      d[t] = 0.f;
      if (t < cnt) {
        float u = val[t];
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) u = fmaf(s_A[t][s2], d[s2], u);
        d[t] = s_b[cur][t] * (s_v[t][row] - u);
      }
    }
#pragma unroll
    for (int t = 0; t < TS; ++t) {
      const float da = __shfl_up_sync(0xffffffffu, d[t], NP, LPR);
      if (!is_a) d[t] = da;
    }
    // records (a lanes) and outputs (b lanes)
#pragma unroll
    for (int t = 0; t < TS; ++t) {
      if (t < cnt) {
        if (is_a) {
          static_cast<ST *>(rv.d)[ent(t0 + t) * V + (size_t)j * VT + row] = from_f32<ST>(d[t]);
          if (more) s_d[t][row] = d[t];
        } else {
          float o = fmaf(s_kq[t], d[t], val[t]);
#pragma unroll
          for (int s2 = 0; s2 < t; ++s2) o = fmaf(s_P[t][s2], d[s2], o);
          out[(((size_t)b * T + t0 + t) * H + h) * V + (size_t)j * VT + row] = from_f32<IO>(o);
        }
      }
    }
    if (more) {
      // the tile at the block end; each row's deltas from its a lane, through shared memory
      // (the rows of a lane group are written by a lanes of the same warp)
      __syncwarp();
      float2 gl[E2];
#pragma unroll
      for (int e = 0; e < E2; ++e)
        gl[e] = make_float2(expf(s_G[cnt - 1][gk(k0 + 2 * e)]), expf(s_G[cnt - 1][gk(k0 + 2 * e + 1)]));
#pragma unroll
      for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int e = 0; e < E2; ++e) s[p][e] = __fmul2_rn(s[p][e], gl[e]);
#pragma unroll 1
      for (int t = 0; t < cnt; ++t) {
        {
          float2 c[E2];
#pragma unroll
          for (int e = 0; e < E2; ++e) c[e] = *reinterpret_cast<const float2 *>(&s_c[t][k0 + 2 * e]);
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            const float dp = s_d[t][G::row(p)];
            const float2 d2 = make_float2(dp, dp);
#pragma unroll
            for (int e = 0; e < E2; ++e) s[p][e] = __ffma2_rn(d2, c[e], s[p][e]);
          }
        }
      }
    }
  };

  for (int t0 = 0; t0 < T; t0 += TS) {
    cp_async_wait_all();
    __syncthreads();  // block `cur` landed; every reader of block cur^1 and of s_qk is done
    if (t0 + TS < T) stage(cur ^ 1, t0 + TS);
    const int cnt = min(TS, T - t0);

    // conv of the block's tokens: each thread rolls its own channels' windows, writes the
    // window after every token into the cache entry (channels it owns) and the conv output
    for (int tau = 0; tau < cnt; ++tau) {
      IO *E = spec_conv + ((size_t)b * L + t0 + tau) * 3 * (size_t)D;
#pragma unroll
      for (int u = 0; u < QK_T; ++u) {
        const int i2 = tid + u * NT;
        if (i2 >= 2 * K) continue;
        const IO xc = s_xqk[cur][tau][i2];
        const float y = conv4(wt[u], to_f32(win[u][0]), to_f32(win[u][1]), to_f32(win[u][2]),
                              to_f32(xc));
        s_qk[tau][i2] = y;
        win[u][0] = win[u][1]; win[u][1] = win[u][2]; win[u][2] = xc;
        if (i2 >= j * OWN && i2 < (j + 1) * OWN) {
          E[cqk[u]] = win[u][0]; E[D + cqk[u]] = win[u][1]; E[2 * D + cqk[u]] = win[u][2];
          if constexpr (REPLAY)
            if (i2 >= K) static_cast<ST *>(rv.rawk)[ent(t0 + tau) * K + (i2 - K)] = from_f32<ST>(y);
        }
      }
      if (tid < VT) {
        const IO xc = s_xv[cur][tau][tid];
        const float y = conv4(wtv, to_f32(winv[0]), to_f32(winv[1]), to_f32(winv[2]), to_f32(xc));
        s_v[tau][tid] = y;
        winv[0] = winv[1]; winv[1] = winv[2]; winv[2] = xc;
        E[cv] = winv[0]; E[D + cv] = winv[1]; E[2 * D + cv] = winv[2];
        if constexpr (REPLAY)
          static_cast<ST *>(rv.rawv)[ent(t0 + tau) * V + (size_t)j * VT + tid] = from_f32<ST>(y);
      }
    }
    if constexpr (REPLAY) {
      for (int c = tid; c < GW; c += NT) {  // G_t = g_0 + ... + g_t, a thread per channel
        float acc = 0.f;
        for (int tau = 0; tau < cnt; ++tau) {
          acc += s_g[cur][tau][c];
          s_G[tau][c] = acc;
        }
      }
    } else if (GATE == RSC_GATE_KDA) {
      for (int i = tid; i < cnt * K; i += NT) s_al[i / K][i % K] = expf(s_g[cur][i / K][i % K]);
    } else if (tid < cnt) {
      s_al[tid][0] = expf(s_g[cur][tid][0]);
    }
    __syncthreads();
    // L2 norms, a warp per token: lane l holds channels l, l+32, ... of q and of k
    for (int tau = warp; tau < cnt; tau += NW) {
      float qq = 0.f, kk = 0.f, qk = 0.f;
#pragma unroll
      for (int e = 0; e < K / 32; ++e) {
        const float a = s_qk[tau][lane + 32 * e], c = s_qk[tau][K + lane + 32 * e];
        qq = fmaf(a, a, qq); kk = fmaf(c, c, kk); qk = fmaf(a, c, qk);
      }
      qq = group_sum<32>(qq); kk = group_sum<32>(kk); qk = group_sum<32>(qk);
      const float rq = 1.0f / sqrtf(qq + kNormEps), rk = 1.0f / sqrtf(kk + kNormEps);
#pragma unroll
      for (int e = 0; e < K / 32; ++e) {
        s_qk[tau][lane + 32 * e] *= rq;
        s_qk[tau][K + lane + 32 * e] *= rk;
      }
      if (lane == 0) s_kq[tau] = qk * rq * rk;
    }
    __syncthreads();
    if constexpr (REPLAY) {
      // the block's normalised keys (owner of the key channels), log-decays and betas (tile 0)
      for (int i = tid; i < cnt * 2 * K; i += NT) {
        const int tau = i / (2 * K), i2 = i % (2 * K);
        if (i2 >= K && i2 >= j * OWN && i2 < (j + 1) * OWN)
          static_cast<ST *>(rv.k)[ent(t0 + tau) * K + (i2 - K)] = from_f32<ST>(s_qk[tau][i2]);
      }
      if (j == 0) {
        for (int i = tid; i < cnt * GW; i += NT)
          rv.g[ent(t0 + i / GW) * GW + i % GW] = s_g[cur][i / GW][i % GW];
        if (tid < cnt) rv.beta[ent(t0 + tid)] = s_b[cur][tid];
      }
    }

    if constexpr (REPLAY) {
      replay_block(t0, cnt);
    } else {
      // the block's tokens: delta rule on the register tile, no barrier inside
      for (int tau = 0; tau < cnt; ++tau) {
        const int t = t0 + tau;
        const size_t bt = (size_t)b * T + t;
        float2 qh[G::EPL / 2], kh[G::EPL / 2], al[G::EPL / 2];
#pragma unroll
        for (int e = 0; e < G::EPL / 2; ++e) {
          qh[e] = *reinterpret_cast<const float2 *>(&s_qk[tau][k0 + 2 * e]);
          kh[e] = *reinterpret_cast<const float2 *>(&s_qk[tau][K + k0 + 2 * e]);
          al[e] = GATE == RSC_GATE_KDA ? *reinterpret_cast<const float2 *>(&s_al[tau][k0 + 2 * e])
                                       : make_float2(s_al[tau][0], s_al[tau][0]);
        }
        float o[G::NP];
        delta_rule_tile2<ST, K, VT, VPL, NW>(s, qh, kh, al, s_b[cur][tau], s_kq[tau], s_v[tau], o, nullptr);
        ST *Se = spec_ssm + ((((size_t)b * L + t) * H + h) * V + (size_t)j * VT) * K;
        tile_store2<ST, K, VT, VPL, NW>(Se, s);
        if (k0 == 0) {
          IO *ob = out + (bt * H + h) * V + (size_t)j * VT;
#pragma unroll
          for (int p = 0; p < G::NP; ++p) ob[G::row(p)] = from_f32<IO>(o[p]);
        }
      }
    }
    cur ^= 1;
  }
}


template <typename ST, typename IO, int K, int V, int GATE>
struct VerifyLaunch {
  static int run(const LayerArgs *a, const int32_t *slots, int B, int T, int L,
                 void *spec_ssm, void *spec_conv, const void *qkv, const float *conv_w,
                 const float *g, const float *beta, void *out, cudaStream_t s) {
    constexpr int NVT = V / (RSC_SNAPSHOT_ROWS < V ? RSC_SNAPSHOT_ROWS : V);
    constexpr int NW = RSC_SNAPSHOT_WARPS;
    dim3 grid(NVT, a->pv.H, B);
    kda_spec_verify_kernel<ST, IO, K, V, NVT, NW, GATE, false><<<grid, NW * 32, 0, s>>>(
        a->pv, a->layer, slots, T, L, static_cast<ST *>(spec_ssm),
        static_cast<IO *>(spec_conv), static_cast<const IO *>(qkv), conv_w, g, beta,
        static_cast<IO *>(out), RingView{}, nullptr);
    return launch_status();
  }
};

int launch_spec_verify(const LayerArgs &a, const int32_t *slots, int B, int T, int L,
                       void *spec_ssm, void *spec_conv, const void *qkv,
                       const float *conv_w, const float *g, const float *beta, void *out,
                       cudaStream_t s) {
  return dispatch_all<VerifyLaunch>(a.st, a.io, a.pv.K, a.pv.V, a.gate, &a, slots, B, T, L,
                                    spec_ssm, spec_conv, qkv, conv_w, g, beta, out, s);
}

// Record-mode verify on the tensor cores: bf16 state, K = V = 128, one block of T <= 8
// tokens (the pages' draft of seven tokens plus the anchor), one CTA per (head, request).
// The same closed form as replay_block, with the 2 T row dots of the block as one tcgen05
// product: D = S0 [k_hat_t . e^G_t | q_hat_t . e^G_t]^T (M = 128 state rows, N = 16,
// K = 128), S0 the slot's tile (exactly bf16, copied into the canonical operand layout by
// cp.async) and the 16 vectors as bf16 high and low parts (two accumulating products, so
// the dots keep ~16 bits of the fp32 vectors).  Thread v (warps 0-3) then reads row v's 16
// dots from tensor memory and runs the 8x8 triangular solve of its row.  No state tile in
// registers: 256 threads at three CTAs per SM.
namespace rtc {
constexpr int K = 128, V = 128, TS = 8, CH = 2 * K + V, NT = 256;
constexpr uint32_t kS0 = 0;                       // S0  bf16 K-major, 128 rows x K
constexpr uint32_t kXH = kS0 + V * K * 2;         // X   bf16 K-major, 16 rows x K (high part)
constexpr uint32_t kXL = kXH + 16 * K * 2;        //     low part
constexpr uint32_t kSx = kXL + 16 * K * 2;        // raw inputs of the block [TS][CH] (io dtype)
constexpr uint32_t kSy = kSx + TS * CH * 4;       // conv outputs fp32 [TS][CH]: q_hat | k_hat | v
constexpr uint32_t kSg = kSy + TS * CH * 4;       // log-decays fp32 [TS][K]
constexpr uint32_t kSG = kSg + TS * K * 4;        // cumulative log-decays fp32 [TS][K]
constexpr uint32_t kSmem = kSG + TS * K * 4;      // 72 KB: three CTAs per SM
}  // namespace rtc

template <typename IO, int GATE>
__global__ void __launch_bounds__(rtc::NT, 3)
kda_replay_verify_tc_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots, int T,
                            IO *__restrict__ spec_conv, const IO *__restrict__ qkv,
                            const float *__restrict__ conv_w, const float *__restrict__ g,
                            const float *__restrict__ beta, IO *__restrict__ out, RingView rv,
                            const int32_t *__restrict__ pos) {
  using namespace rtc;
  using bf16_t = bf16;
  constexpr int GW = GATE == RSC_GATE_KDA ? K : 1;
  constexpr int XV = 16 / sizeof(IO);
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ float s_b[TS], s_kq[TS], s_A[TS][TS], s_P[TS][TS];
  __shared__ uint32_t s_taddr;
  __shared__ __align__(8) uint64_t s_bar;
  IO *sx = reinterpret_cast<IO *>(smem + kSx);
  float *sy = reinterpret_cast<float *>(smem + kSy);
  float *sg = reinterpret_cast<float *>(smem + kSg);
  float *sG = reinterpret_cast<float *>(smem + kSG);
  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = pv.H, D = pv.D;

  const int slot = slots[b];
  if (slot < 0 || slot > pv.P) {
    if (tid == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_SLOT);
    return;
  }
  const int p0 = pos[b];
  if (p0 < 0 || p0 >= rv.depth) {
    if (tid == 0 && h == 0) flag_error(pv.err, RSC_DEVERR_RING);
    return;
  }
  const size_t prow = (size_t)layer * (pv.P + 1) + slot;
  auto ent = [&](int t) { return (prow * H + h) * (size_t)rv.depth + ((p0 + t) & (rv.depth - 1)); };
  // channel c of the head (q | k | v) -> column of the projections and of the window
  auto col = [&](int c) {
    return c < K ? h * K + c : c < 2 * K ? H * K + h * K + (c - K) : 2 * H * K + h * V + (c - 2 * K);
  };

  if (tid == 0) mbar_init(&s_bar, 1);
  if (warp == 0) { tc::tmem_alloc(&s_taddr, 32); tc::tmem_relinquish(); }

  // 1. copies in two groups: the block's raw inputs, gates and betas (waited for before the
  //    conv), then the slot's tile into the operand layout (8 lanes with the same 16-byte
  //    column take 8 consecutive rows: distinct bank groups), waited for only before the
  //    product, so its latency hides behind the conv, the norms and the coefficients
  for (int i = tid; i < T * (CH / XV); i += NT) {
    const int t = i / (CH / XV), c = (i % (CH / XV)) * XV;
    cp_async16(sx + t * CH + c, qkv + ((size_t)b * T + t) * D + col(c));
  }
  if constexpr (GW == K) {
    for (int i = tid; i < T * (K / 4); i += NT) {
      const int t = i / (K / 4), c = (i % (K / 4)) * 4;
      cp_async16(sg + t * K + c, g + (((size_t)b * T + t) * H + h) * K + c);
    }
  } else if (tid < T) {
    cp_async4(sg + tid * K, g + ((size_t)b * T + tid) * H + h);
  }
  if (tid < T) cp_async4(&s_b[tid], beta + ((size_t)b * T + tid) * H + h);
  cp_async_commit();
  const bf16_t *Sg = reinterpret_cast<const bf16_t *>(pv.ssm) + (prow * H + h) * (size_t)V * K;
  for (int i = tid; i < V * K / 8; i += NT) {
    const int v = ((i >> 7) << 3) | (i & 7), kc = (i >> 3) & 15;
    cp_async16(smem + kS0 + tc::kmajor_offset(v, 8 * kc, K), Sg + (size_t)v * K + 8 * kc);
  }
  cp_async_commit();
  // taps and window rows of this thread's channels (tid, and tid + 256 below 384)
  const IO *W = reinterpret_cast<const IO *>(pv.conv) + prow * 3 * (size_t)D;
  float4 wt[2];
  IO win[2][3];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int c = tid + u * NT;
    if (c < CH) {
      const int cc = col(c);
      wt[u] = *reinterpret_cast<const float4 *>(conv_w + 4 * (size_t)cc);
      win[u][0] = W[cc]; win[u][1] = W[D + cc]; win[u][2] = W[2 * D + cc];
    }
  }
  asm volatile("cp.async.wait_group 1;\n" ::: "memory");  // the inputs (the tile may be in flight)
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = s_taddr;

  // 2. conv of every token (each thread rolls its channels' windows, writes the window after
  //    every token into the cache entry, rawk / rawv records), cumulative log-decays
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int c = tid + u * NT;
    if (c >= CH) continue;
    const int cc = col(c);
    for (int t = 0; t < T; ++t) {
      const IO xc = sx[t * CH + c];
      const float y = conv4(wt[u], to_f32(win[u][0]), to_f32(win[u][1]), to_f32(win[u][2]), to_f32(xc));
      sy[t * CH + c] = y;
      win[u][0] = win[u][1]; win[u][1] = win[u][2]; win[u][2] = xc;
      IO *E = spec_conv + ((size_t)b * rv.depth + t) * 3 * (size_t)D;
      E[cc] = win[u][0]; E[D + cc] = win[u][1]; E[2 * D + cc] = win[u][2];
      if (c >= 2 * K) static_cast<bf16_t *>(rv.rawv)[ent(t) * V + (c - 2 * K)] = __float2bfloat16_rn(y);
      else if (c >= K) static_cast<bf16_t *>(rv.rawk)[ent(t) * K + (c - K)] = __float2bfloat16_rn(y);
    }
  }
  if (tid < GW) {
    float acc = 0.f;
    for (int t = 0; t < T; ++t) {
      const float x = sg[t * K + tid];
      acc += x;
      sG[t * K + tid] = acc;
      rv.g[ent(t) * GW + tid] = x;
    }
  }
  if (tid < T) rv.beta[ent(tid)] = s_b[tid];
  __syncthreads();

  // 3. L2 norms, a warp per token (lane l: channels l, l+32, l+64, l+96 of q and of k);
  //    the normalised key's record
  for (int t = warp; t < T; t += NT / 32) {
    float *yq = sy + t * CH, *yk = yq + K;
    float qq = 0.f, kk = 0.f, qk = 0.f;
#pragma unroll
    for (int e = 0; e < K / 32; ++e) {
      const float a = yq[lane + 32 * e], c = yk[lane + 32 * e];
      qq = fmaf(a, a, qq); kk = fmaf(c, c, kk); qk = fmaf(a, c, qk);
    }
    qq = group_sum<32>(qq); kk = group_sum<32>(kk); qk = group_sum<32>(qk);
    const float rq = 1.0f / sqrtf(qq + kNormEps), rk = 1.0f / sqrtf(kk + kNormEps);
#pragma unroll
    for (int e = 0; e < K / 32; ++e) {
      yq[lane + 32 * e] *= rq;
      const float kh = yk[lane + 32 * e] * rk;
      yk[lane + 32 * e] = kh;
      static_cast<bf16_t *>(rv.k)[ent(t) * K + lane + 32 * e] = __float2bfloat16_rn(kh);
    }
    if (lane == 0) s_kq[t] = qk * rq * rk;
  }
  __syncthreads();

  // 4. the product's B operand, rows n < 8: k_hat_n . e^G_n, rows 8 + n: q_hat_n . e^G_n (zero
  //    beyond the block), as bf16 high and low parts; item i: row i % 16, eight channels
  //    8 (i / 16) .. +7
  {
    const int n = tid & 15, kc = tid >> 4, t = n & 7;
    float hi[8], lo[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float x = 0.f;
      if (t < T) {
        const int k = 8 * kc + e;
        const float Gt = sG[t * K + (GW == 1 ? 0 : k)];
        x = sy[t * CH + (n < 8 ? K : 0) + k] * __expf(Gt);
      }
      hi[e] = __bfloat162float(__float2bfloat16_rn(x));
      lo[e] = x - hi[e];
    }
    const uint32_t off = tc::kmajor_offset(n, 8 * kc, K);
    st16(smem + kXH + off, pack16(hi));
    st16(smem + kXL + off, pack16(lo));
  }
  // coefficients of the pairs s < t: A[t][s] = sum_k k_s k_t e^(G_t - G_s), P[t][s] = sum_k
  // k_s q_t e^(G_t - G_s); warp w takes pairs w, w + 8, ..., lane l channels 4l .. 4l+3
  for (int pi = warp; pi < TS * (TS - 1) / 2; pi += NT / 32) {
    int t = 1;
    while (t * (t + 1) / 2 <= pi) ++t;
    const int s2 = pi - t * (t - 1) / 2;
    if (t >= T) continue;  // uniform over the warp
    const float *ks = sy + s2 * CH + K, *kt = sy + t * CH + K, *qt = sy + t * CH;
    float a = 0.f, p = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = 4 * lane + e;
      const float dg = GW == 1 ? sG[t * K] - sG[s2 * K] : sG[t * K + k] - sG[s2 * K + k];
      const float kd = ks[k] * __expf(dg);
      a = fmaf(kd, kt[k], a);
      p = fmaf(kd, qt[k], p);
    }
    a = group_sum<32>(a);
    p = group_sum<32>(p);
    if (lane == 0) { s_A[t][s2] = a; s_P[t][s2] = p; }
  }
  cp_async_wait_all();        // this thread's pieces of the tile
  tc::fence_smem_to_async();  // the tile and X are read by the tensor core
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // 5. D = S0 X^T on the tensor core (high part, then low part accumulated)
  if (tid == 0) {
    constexpr uint32_t idesc = tc::idesc_bf16<128, 16>();
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks)
      tc::mma_bf16(taddr, tc::kmajor_desc(smem + kS0, K, ks), tc::kmajor_desc(smem + kXH, K, ks),
                   idesc, ks > 0);
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks)
      tc::mma_bf16(taddr, tc::kmajor_desc(smem + kS0, K, ks), tc::kmajor_desc(smem + kXL, K, ks),
                   idesc, true);
    tc::mma_commit(&s_bar);
  }
  bool ok = true;
  if (warp < 4) {
    ok = mbar_wait(&s_bar, 0);
    tc::fence_after_sync();
  }
  ok = __syncthreads_and(ok);
  // 6. row v = tid (warps 0-3, their own lane quadrant): a_t, b_t; the triangular solve
  //    d_t = beta_t (v_t - a_t - sum_{s<t} A[t][s] d_s), o_t = b_t + sum_{s<=t} P[t][s] d_s
  if (ok && warp < 4) {
    float dv[16];
    tc::tmem_ld16(tc::tmem_addr(taddr, 32 * warp, 0), dv);
    const int v = tid;
    float d[TS];
#pragma unroll
    for (int t = 0; t < TS; ++t) {
      d[t] = 0.f;
      if (t < T) {
        float u = dv[t];
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) u = fmaf(s_A[t][s2], d[s2], u);
        d[t] = s_b[t] * (sy[t * CH + 2 * K + v] - u);
        float o = fmaf(s_kq[t], d[t], dv[8 + t]);
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) o = fmaf(s_P[t][s2], d[s2], o);
        static_cast<bf16_t *>(rv.d)[ent(t) * V + v] = __float2bfloat16_rn(d[t]);
        out[(((size_t)b * T + t) * H + h) * V + v] = from_f32<IO>(o);
      }
    }
  } else if (!ok && tid == 0) {
    flag_error(pv.err, RSC_DEVERR_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(taddr, 32);
}

template <typename IO, int GATE>
static int launch_replay_verify_tc(const LayerArgs &a, const RingView &rv, const int32_t *slots,
                                   const int32_t *pos, int B, int T, void *spec_conv,
                                   const void *qkv, const float *conv_w, const float *g,
                                   const float *beta, void *out, cudaStream_t s) {
  auto kern = kda_replay_verify_tc_kernel<IO, GATE>;
  static PerDeviceFlag attr;
  const int rc = once_per_device(attr, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)rtc::kSmem) == cudaSuccess ? RSC_OK : RSC_ECUDA;
  });
  if (rc != RSC_OK) return rc;
  kern<<<dim3(a.pv.H, B), rtc::NT, rtc::kSmem, s>>>(
      a.pv, a.layer, slots, T, static_cast<IO *>(spec_conv), static_cast<const IO *>(qkv),
      conv_w, g, beta, static_cast<IO *>(out), rv, pos);
  return launch_status();
}

template <typename ST, typename IO, int K, int V, int GATE>
struct ReplayVerifyLaunch {
  static int run(const LayerArgs *a, const RingView *rv, const int32_t *slots, const int32_t *pos,
                 int B, int T, void *spec_conv, const void *qkv, const float *conv_w,
                 const float *g, const float *beta, void *out, cudaStream_t s) {
    constexpr int ROWS = RSC_REPLAY_ROWS < V ? RSC_REPLAY_ROWS : V;
    constexpr int NVT = V / ROWS;
    constexpr int NW = ROWS / 16;
    static_assert(RSC_REPLAY_ROWS == 16 * RSC_REPLAY_WARPS, "rows = 16 x warps");
    dim3 grid(NVT, a->pv.H, B);
    kda_spec_verify_kernel<ST, IO, K, V, NVT, NW, GATE, true><<<grid, NW * 32, 0, s>>>(
        a->pv, a->layer, slots, T, rv->depth, nullptr, static_cast<IO *>(spec_conv),
        static_cast<const IO *>(qkv), conv_w, g, beta, static_cast<IO *>(out), *rv, pos);
    return launch_status();
  }
};

int launch_replay_verify(const LayerArgs &a, const RingView &rv, const int32_t *slots,
                         const int32_t *pos, int B, int T, void *spec_conv, const void *qkv,
                         const float *conv_w, const float *g, const float *beta, void *out,
                         cudaStream_t s) {
  if (a.st == RSC_BF16 && a.pv.K == 128 && a.pv.V == 128 && T >= 1 && T <= rtc::TS) {
    const bool kda = a.gate == RSC_GATE_KDA;
    if (a.io == RSC_BF16)
      return kda ? launch_replay_verify_tc<bf16, RSC_GATE_KDA>(a, rv, slots, pos, B, T, spec_conv,
                                                               qkv, conv_w, g, beta, out, s)
                 : launch_replay_verify_tc<bf16, RSC_GATE_GDN>(a, rv, slots, pos, B, T, spec_conv,
                                                               qkv, conv_w, g, beta, out, s);
    return kda ? launch_replay_verify_tc<float, RSC_GATE_KDA>(a, rv, slots, pos, B, T, spec_conv,
                                                              qkv, conv_w, g, beta, out, s)
               : launch_replay_verify_tc<float, RSC_GATE_GDN>(a, rv, slots, pos, B, T, spec_conv,
                                                              qkv, conv_w, g, beta, out, s);
  }
  return dispatch_all<ReplayVerifyLaunch>(a.st, a.io, a.pv.K, a.pv.V, a.gate, &a, &rv, slots,
                                          pos, B, T, spec_conv, qkv, conv_w, g, beta, out, s);
}

// ReplaySSM COMMIT: one CTA per (row tile, head, request).  The tile of the slot's state is
// loaded into registers, tokens 0..accept[b] are replayed from the rings eight at a time
// (their pre-norm keys, log-decays, this tile's value rows and betas staged by cp.async; the
// key norms and exp(g) of the block computed before its token loop), and the tile is stored
// back.  The CTA also restores its share of the window from snapshot accept[b] (the same
// channel ownership as the verify pass), so every byte of the slot has one writer.
template <typename ST, typename IO, int K, int V, int NVT, int NW, int GATE>
__global__ void __launch_bounds__(NW * 32, RSC_COMMIT_MINB)
kda_replay_commit_kernel(PoolView pv, RingView rv, int layer, const int32_t *__restrict__ slots,
                         const int32_t *__restrict__ pos, int T, const IO *__restrict__ spec_conv,
                         const int32_t *__restrict__ accept) {
  constexpr int VT = V / NVT;
  constexpr int VPL = 1;
  constexpr int NT = NW * 32;
  using G = TileGeom<ST, K, VT, NW, VPL>;
  constexpr int OWN = 2 * K / NVT;
  constexpr int TS = 8;
  constexpr int GW = GATE == RSC_GATE_KDA ? K : 1;
  constexpr int XS = 16 / sizeof(ST);  // state-dtype elements per 16-byte copy
  static_assert(K % XS == 0 && VT % XS == 0, "16-byte staging");
  __shared__ __align__(16) ST s_rk[TS][K];
  __shared__ __align__(16) ST s_rv[TS][VT];
  __shared__ __align__(16) float s_g[TS][GW];
  __shared__ float s_b[TS];
  __shared__ __align__(16) float s_kh[TS][K];
  __shared__ float s_v[TS][VT];
  __shared__ __align__(16) float s_al[TS][GW];

  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = pv.H, D = pv.D;
  const int slot = slots[b], acc = accept[b], p0 = pos[b];
  const bool bad_slot = slot < 0 || slot > pv.P, bad_acc = acc < 0 || acc >= T;
  const bool bad_pos = p0 < 0 || p0 >= rv.depth;
  if (bad_slot || bad_acc || bad_pos) {
    if (tid == 0 && j == 0 && h == 0)
      flag_error(pv.err, (bad_slot ? RSC_DEVERR_SLOT : 0) | (bad_acc ? RSC_DEVERR_ACCEPT : 0) |
                             (bad_pos ? RSC_DEVERR_RING : 0));
    return;
  }
  const size_t prow = (size_t)layer * (pv.P + 1) + slot;
  auto ent = [&](int t) { return (prow * H + h) * (size_t)rv.depth + ((p0 + t) & (rv.depth - 1)); };
  const int n = acc + 1;  // tokens to replay

  // the records of tokens t0 .. t0 + cnt - 1 into shared memory (cp.async, one group)
  auto stage = [&](int t0, int cnt) {
    for (int i = tid; i < cnt * (K / XS); i += NT) {
      const int tau = i / (K / XS), c = (i % (K / XS)) * XS;
      cp_async16(&s_rk[tau][c], static_cast<const ST *>(rv.rawk) + ent(t0 + tau) * K + c);
    }
    for (int i = tid; i < cnt * (VT / XS); i += NT) {
      const int tau = i / (VT / XS), c = (i % (VT / XS)) * XS;
      cp_async16(&s_rv[tau][c], static_cast<const ST *>(rv.rawv) + ent(t0 + tau) * V + (size_t)j * VT + c);
    }
    if (GATE == RSC_GATE_KDA) {
      for (int i = tid; i < cnt * (K / 4); i += NT) {
        const int tau = i / (K / 4), c = (i % (K / 4)) * 4;
        cp_async16(&s_g[tau][c], rv.g + ent(t0 + tau) * K + c);
      }
    } else if (tid < cnt) {
      cp_async4(&s_g[tid][0], rv.g + ent(t0 + tid));
    }
    if (tid < cnt) cp_async4(&s_b[tid], rv.beta + ent(t0 + tid));
    cp_async_commit();
  };
  // the first block's records are requested before the state tile, which is needed only
  // after their norms: the two latencies overlap
  stage(0, min(TS, n));
  ST *S = reinterpret_cast<ST *>(pv.ssm) + ((prow * H + h) * V + (size_t)j * VT) * K;
  Tile2<ST, K, VT, NW, VPL> s;
  tile_load2<ST, K, VT, VPL, NW>(S, s);
  const int k0 = G::kofs();
  // the window snapshot accept[b]: this CTA's q/k channels of the head and its value channels,
  // requested now and written back at the end (its latency hides behind the replay)
  const IO *E = spec_conv + ((size_t)b * rv.depth + acc) * 3 * (size_t)D;
  IO *W = reinterpret_cast<IO *>(pv.conv) + prow * 3 * (size_t)D;
  constexpr int NWIN = (3 * (OWN + VT) + NT - 1) / NT;
  IO wsnap[NWIN];
  auto win_index = [&](int i) {  // element i of this CTA's share -> offset in a [3][D] window
    const int row = i / (OWN + VT), c = i % (OWN + VT);
    const int i2 = j * OWN + c;
    const int ch = c < OWN ? (i2 < K ? h * K + i2 : H * K + h * K + (i2 - K))
                           : 2 * H * K + h * V + j * VT + (c - OWN);
    return (size_t)row * D + ch;
  };
#pragma unroll
  for (int u = 0; u < NWIN; ++u) {
    const int i = tid + u * NT;
    if (i < 3 * (OWN + VT)) wsnap[u] = E[win_index(i)];
  }

  for (int t0 = 0; t0 < n; t0 += TS) {
    const int cnt = min(TS, n - t0);
    if (t0 > 0) {
      __syncthreads();  // the previous block's readers are done
      stage(t0, cnt);
    }
    cp_async_wait_all();
    __syncthreads();
    // normalised keys (a warp per token), alpha = exp(g), value rows to fp32
    for (int tau = warp; tau < cnt; tau += NW) {
      float kk = 0.f;
#pragma unroll
      for (int e = 0; e < K / 32; ++e) {
        const float x = to_f32(s_rk[tau][lane + 32 * e]);
        kk = fmaf(x, x, kk);
      }
      kk = group_sum<32>(kk);
      const float rk = 1.0f / sqrtf(kk + kNormEps);
#pragma unroll
      for (int e = 0; e < K / 32; ++e) s_kh[tau][lane + 32 * e] = to_f32(s_rk[tau][lane + 32 * e]) * rk;
    }
    if (GATE == RSC_GATE_KDA) {
      for (int i = tid; i < cnt * K; i += NT) s_al[i / K][i % K] = expf(s_g[i / K][i % K]);
    } else if (tid < cnt) {
      s_al[tid][0] = expf(s_g[tid][0]);
    }
    for (int i = tid; i < cnt * VT; i += NT) s_v[i / VT][i % VT] = to_f32(s_rv[i / VT][i % VT]);
    __syncthreads();
    for (int tau = 0; tau < cnt; ++tau) {
      float2 kh[G::EPL / 2], al[G::EPL / 2];
#pragma unroll
      for (int e = 0; e < G::EPL / 2; ++e) {
        kh[e] = *reinterpret_cast<const float2 *>(&s_kh[tau][k0 + 2 * e]);
        al[e] = GATE == RSC_GATE_KDA ? *reinterpret_cast<const float2 *>(&s_al[tau][k0 + 2 * e])
                                     : make_float2(s_al[tau][0], s_al[tau][0]);
      }
      delta_rule_tile2<ST, K, VT, VPL, NW, false>(s, kh, kh, al, s_b[tau], 0.f, s_v[tau], nullptr, nullptr);
    }
  }
  tile_store2<ST, K, VT, VPL, NW>(S, s);
  // window <- snapshot acc
#pragma unroll
  for (int u = 0; u < NWIN; ++u) {
    const int i = tid + u * NT;
    if (i < 3 * (OWN + VT)) W[win_index(i)] = wsnap[u];
  }
}

template <typename ST, typename IO, int K, int V, int GATE>
struct ReplayCommitLaunch {
  static int run(const LayerArgs *a, const RingView *rv, const int32_t *slots, const int32_t *pos,
                 int B, int T, const void *spec_conv, const int32_t *accept, cudaStream_t s) {
    constexpr int NVT = V / (RSC_COMMIT_ROWS < V ? RSC_COMMIT_ROWS : V);
    constexpr int NW = RSC_COMMIT_WARPS;
    dim3 grid(NVT, a->pv.H, B);
    kda_replay_commit_kernel<ST, IO, K, V, NVT, NW, GATE><<<grid, NW * 32, 0, s>>>(
        a->pv, *rv, a->layer, slots, pos, T, static_cast<const IO *>(spec_conv), accept);
    return launch_status();
  }
};

int launch_replay_commit(const LayerArgs &a, const RingView &rv, const int32_t *slots,
                         const int32_t *pos, int B, int T, const void *spec_conv,
                         const int32_t *accept, cudaStream_t s) {
  return dispatch_all<ReplayCommitLaunch>(a.st, a.io, a.pv.K, a.pv.V, a.gate, &a, &rv, slots,
                                          pos, B, T, spec_conv, accept, s);
}

// COMMIT: slot <- cache entry accept[b], the state rows (blockIdx.z == 0) and the window
// rows (blockIdx.z == 1) in one launch.  Grid (chunks of kCopyChunk bytes of the longer
// row, batch, 2).  A bad slot or accept count skips the row and sets the error word.
__global__ void __launch_bounds__(128)
kda_spec_commit_kernel(PoolView pv, int layer, size_t ssm_row_bytes, size_t conv_row_bytes,
                       const int32_t *__restrict__ slots, int T, int L,
                       const char *__restrict__ spec_ssm, const char *__restrict__ spec_conv,
                       const int32_t *__restrict__ accept) {
  const int b = blockIdx.y, which = blockIdx.z;
  const int slot = slots[b], a = accept[b];
  const bool bad_slot = slot < 0 || slot > pv.P, bad_acc = a < 0 || a >= T;
  if (bad_slot || bad_acc) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && which == 0)
      flag_error(pv.err, (bad_slot ? RSC_DEVERR_SLOT : 0) | (bad_acc ? RSC_DEVERR_ACCEPT : 0));
    return;
  }
  const size_t row_bytes = which == 0 ? ssm_row_bytes : conv_row_bytes;
  const size_t off = (size_t)blockIdx.x * kCopyChunk;
  if (off >= row_bytes) return;
  char *base = reinterpret_cast<char *>(which == 0 ? pv.ssm : pv.conv);
  char *dst = base + ((size_t)layer * (pv.P + 1) + slot) * row_bytes;
  const char *src = (which == 0 ? spec_ssm : spec_conv) + ((size_t)b * L + a) * row_bytes;
  copy_chunk(dst, src, row_bytes, off);
}

int launch_spec_commit(const LayerArgs &a, const int32_t *slots, int B, int T, int L,
                       const void *spec_ssm, const void *spec_conv, const int32_t *accept,
                       cudaStream_t s) {
  const size_t ssz = a.st == RSC_F32 ? 4 : 2, csz = a.io == RSC_F32 ? 4 : 2;
  const size_t sb = (size_t)a.pv.H * a.pv.V * a.pv.K * ssz;
  const size_t cb = (size_t)3 * a.pv.D * csz;
  const size_t longest = sb > cb ? sb : cb;
  dim3 grid((unsigned)((longest + kCopyChunk - 1) / kCopyChunk), B, 2);
  kda_spec_commit_kernel<<<grid, 128, 0, s>>>(a.pv, a.layer, sb, cb, slots, T, L,
                                              static_cast<const char *>(spec_ssm),
                                              static_cast<const char *>(spec_conv), accept);
  return launch_status();
}

}  // namespace rsc

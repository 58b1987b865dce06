// rsc_step.cuh -- the per-token delta-rule update of one CTA's tile of S rows.
//
// A CTA of 128 threads owns VT consecutive rows of one head's state S[V][K] (K
// contiguous).  Each row is covered by LPR lanes holding one 16-byte vector each (EPL
// elements), so a warp touches RPW whole rows per pass and a pass of the CTA covers
// RPP rows: every global access of S is a fully coalesced 16-byte vector access.  Rows
// of S evolve independently under the gated delta rule (the update acts on S from the
// right), which is what lets a head be split across CTAs by rows.
#pragma once

#include "rsc_common.cuh"

namespace rsc {

template <typename ST, int K, int VT, int NW = 4, int VPL = 1>
struct TileGeom {
  static constexpr int EPL = VPL * VecTraits<ST>::N;  // elements per lane (VPL 16-byte vectors)
  static constexpr int LPR = K / EPL;                 // lanes per row
  static constexpr int RPW = 32 / LPR;                // rows per warp per pass
  static constexpr int RPP = NW * RPW;                // rows per CTA per pass
  static constexpr int NP = VT / RPP;                 // passes
  static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row must fit a warp");
  static_assert(NP >= 1 && NP * RPP == VT, "tile rows must be whole passes");
  __device__ static __forceinline__ int row(int p) {
    return p * RPP + (threadIdx.x >> 5) * RPW + (threadIdx.x & 31) / LPR;
  }
  __device__ static __forceinline__ int kofs() { return ((threadIdx.x & 31) % LPR) * EPL; }
};

// Load / store this thread's part of the tile (rows base[row(p)*K + kofs()]): VPL
// consecutive 16-byte vectors per lane and pass.
template <typename ST, int K, int VT, int VPL = 1, int NW = 4>
__device__ __forceinline__ void tile_load(const ST *base, float (&s)[TileGeom<ST, K, VT, NW, VPL>::NP][TileGeom<ST, K, VT, NW, VPL>::EPL]) {
  using G = TileGeom<ST, K, VT, NW, VPL>;
  constexpr int N16 = VecTraits<ST>::N;
#pragma unroll
  for (int p = 0; p < G::NP; ++p)
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      float x[N16];
      unpack16(ld16_stream(base + (size_t)G::row(p) * K + G::kofs() + v * N16), x);
#pragma unroll
      for (int e = 0; e < N16; ++e) s[p][v * N16 + e] = x[e];
    }
}

template <typename ST, int K, int VT, int VPL = 1, int NW = 4>
__device__ __forceinline__ void tile_store(ST *base, const float (&s)[TileGeom<ST, K, VT, NW, VPL>::NP][TileGeom<ST, K, VT, NW, VPL>::EPL]) {
  using G = TileGeom<ST, K, VT, NW, VPL>;
  constexpr int N16 = VecTraits<ST>::N;
#pragma unroll
  for (int p = 0; p < G::NP; ++p)
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      float x[N16];
#pragma unroll
      for (int e = 0; e < N16; ++e) x[e] = s[p][v * N16 + e];
      st16(base + (size_t)G::row(p) * K + G::kofs() + v * N16, pack16(x));
    }
}

// One token of the gated delta rule on one row segment held by this lane (EPL elements
// of row r; the LPR lanes of the row together hold the whole row):
//   s <- s . alpha            (decay, S Diag(alpha))
//   u  = s . k_hat ;  w = s . q_hat          (one pass, two row dots)
//   d  = beta (v_r - u)
//   s <- s + d k_hat          (rank-1 write)
//   o_r = w + d (k_hat . q_hat)
// The last line is S_new q_hat written out: (S Diag(alpha) + d k^T) q = w + d (k.q), so
// the output of the updated state costs no second pass over the row.
template <int EPL, int LPR>
__device__ __forceinline__ float delta_rule_row(float (&s)[EPL], const float (&qh)[EPL],
                                                const float (&kh)[EPL], const float (&al)[EPL],
                                                float beta, float kq, float v_r) {
  float u = 0.f, w = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    s[e] *= al[e];
    u = fmaf(s[e], kh[e], u);
    w = fmaf(s[e], qh[e], w);
  }
  u = group_sum<LPR>(u);
  w = group_sum<LPR>(w);
  const float d = beta * (v_r - u);
#pragma unroll
  for (int e = 0; e < EPL; ++e) s[e] = fmaf(d, kh[e], s[e]);
  return fmaf(d, kq, w);
}

// delta_rule_row on fp32 pairs (the packed fp32 instructions: two lanes of arithmetic per
// issue); the same update, the sums taken pairwise.
template <int E2, int LPR>
__device__ __forceinline__ float delta_rule_row2(float2 (&s)[E2], const float2 (&qh)[E2],
                                                 const float2 (&kh)[E2], const float2 (&al)[E2],
                                                 float beta, float kq, float v_r) {
  float2 u2 = make_float2(0.f, 0.f), w2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < E2; ++e) {
    s[e] = __fmul2_rn(s[e], al[e]);
    u2 = __ffma2_rn(s[e], kh[e], u2);
    w2 = __ffma2_rn(s[e], qh[e], w2);
  }
  const float u = group_sum<LPR>(u2.x + u2.y);
  const float w = group_sum<LPR>(w2.x + w2.y);
  const float d = beta * (v_r - u);
  const float2 d2 = make_float2(d, d);
#pragma unroll
  for (int e = 0; e < E2; ++e) s[e] = __ffma2_rn(d2, kh[e], s[e]);
  return fmaf(d, kq, w);
}

// The same for every row of a register-held tile (rows G::row(p), p < NP).
template <typename ST, int K, int VT, int VPL = 1, int NW = 4>
__device__ __forceinline__ void delta_rule_tile(
    float (&s)[TileGeom<ST, K, VT, NW, VPL>::NP][TileGeom<ST, K, VT, NW, VPL>::EPL],
    const float (&qh)[TileGeom<ST, K, VT, NW, VPL>::EPL],
    const float (&kh)[TileGeom<ST, K, VT, NW, VPL>::EPL],
    const float (&al)[TileGeom<ST, K, VT, NW, VPL>::EPL], float beta, float kq,
    const float *v_rows, float (&o)[TileGeom<ST, K, VT, NW, VPL>::NP]) {
  using G = TileGeom<ST, K, VT, NW, VPL>;
#pragma unroll
  for (int p = 0; p < G::NP; ++p)
    o[p] = delta_rule_row<G::EPL, G::LPR>(s[p], qh, kh, al, beta, kq, v_rows[G::row(p)]);
}

// ---- the same on a tile held as fp32 pairs: each lane's EPL elements of a row as EPL/2
// float2, updated with the packed fp32 instructions (two lanes of arithmetic per issue).
template <typename ST, int K, int VT, int NW = 4, int VPL = 1>
using Tile2 = float2[TileGeom<ST, K, VT, NW, VPL>::NP][TileGeom<ST, K, VT, NW, VPL>::EPL / 2];

template <typename ST, int K, int VT, int VPL = 1, int NW = 4>
__device__ __forceinline__ void tile_load2(const ST *base, Tile2<ST, K, VT, NW, VPL> &s) {
  using G = TileGeom<ST, K, VT, NW, VPL>;
  constexpr int N16 = VecTraits<ST>::N;
#pragma unroll
  for (int p = 0; p < G::NP; ++p)
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      float x[N16];
      unpack16(ld16_stream(base + (size_t)G::row(p) * K + G::kofs() + v * N16), x);
#pragma unroll
      for (int e = 0; e < N16 / 2; ++e) s[p][v * N16 / 2 + e] = make_float2(x[2 * e], x[2 * e + 1]);
    }
}

// Streaming (evict-first) stores: a stored tile is not read again soon (a spec cache entry
// until its commit, a committed slot until that layer's next step).
template <typename ST, int K, int VT, int VPL = 1, int NW = 4>
__device__ __forceinline__ void tile_store2(ST *base, const Tile2<ST, K, VT, NW, VPL> &s) {
  using G = TileGeom<ST, K, VT, NW, VPL>;
  constexpr int N16 = VecTraits<ST>::N;
#pragma unroll
  for (int p = 0; p < G::NP; ++p)
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      float x[N16];
#pragma unroll
      for (int e = 0; e < N16 / 2; ++e) {
        x[2 * e] = s[p][v * N16 / 2 + e].x;
        x[2 * e + 1] = s[p][v * N16 / 2 + e].y;
      }
      st16_stream(base + (size_t)G::row(p) * K + G::kofs() + v * N16, pack16(x));
    }
}

// One token on every row of a pair tile.  Returns o (row outputs, S_new q_hat) and, when
// dd is given, each row's delta.  qh/kh/al are this lane's EPL/2 pairs of q_hat, k_hat, alpha.
template <typename ST, int K, int VT, int VPL = 1, int NW = 4, bool WITH_Q = true>
__device__ __forceinline__ void delta_rule_tile2(
    Tile2<ST, K, VT, NW, VPL> &s, const float2 (&qh)[TileGeom<ST, K, VT, NW, VPL>::EPL / 2],
    const float2 (&kh)[TileGeom<ST, K, VT, NW, VPL>::EPL / 2],
    const float2 (&al)[TileGeom<ST, K, VT, NW, VPL>::EPL / 2], float beta, float kq,
    const float *v_rows, float *o, float *dd) {
  using G = TileGeom<ST, K, VT, NW, VPL>;
  constexpr int E2 = G::EPL / 2;
#pragma unroll
  for (int p = 0; p < G::NP; ++p) {
    float2 u2 = make_float2(0.f, 0.f), w2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < E2; ++e) {
      s[p][e] = __fmul2_rn(s[p][e], al[e]);
      u2 = __ffma2_rn(s[p][e], kh[e], u2);
      if (WITH_Q) w2 = __ffma2_rn(s[p][e], qh[e], w2);
    }
    const float u = group_sum<G::LPR>(u2.x + u2.y);
    const float d = beta * (v_rows[G::row(p)] - u);
    const float2 d2 = make_float2(d, d);
#pragma unroll
    for (int e = 0; e < E2; ++e) s[p][e] = __ffma2_rn(d2, kh[e], s[p][e]);
    if (WITH_Q) o[p] = fmaf(d, kq, group_sum<G::LPR>(w2.x + w2.y));
    if (dd) dd[p] = d;
  }
}

// Butterfly reduce-scatter over the M lanes of an aligned lane group (M a power of two, at
// most 32): on entry every lane holds M partial values x[0..M); on return lane i of the group
// holds the sum over the group of entry i.  M - 1 shuffles in all, where M separate group
// sums take M log2(M).  x is clobbered.
template <int M>
__device__ __forceinline__ float group_reduce_scatter(float (&x)[M]) {
  const int li = threadIdx.x & (M - 1);
#pragma unroll
  for (int n = M; n > 1; n >>= 1) {
    const int m = n >> 1;
    const bool up = (li & m) != 0;  // this lane keeps the upper half of the current list
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float send = up ? x[i] : x[i + m];
      const float keep = up ? x[i + m] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  return x[0];
}

// The conv of one channel: taps 0..2 on the window rows (oldest first), tap 3 on x.
__device__ __forceinline__ float conv4(const float4 &w, float w0, float w1, float w2, float x) {
  return fmaf(w.w, x, fmaf(w.z, w2, fmaf(w.y, w1, w.x * w0)));
}

}  // namespace rsc

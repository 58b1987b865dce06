// prefill_tc.cu -- chunked prefill in the chunkwise (WY / UT) form on the tcgen05 tensor
// cores, for bf16-state pools with K = 128.
//
// Source: "SGLang之KV Cache内存池机制" §8.5 (chunk-based extend with chunk 64: an
// inter-chunk recurrence plus intra-chunk parallel work) and the unrolled closed form of
// the recurrence printed in "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理"
// (ReplaySSM section).  The pages give no more than that; the algebra below is derived
// from the recurrence and is checked against it by the oracle's own chunkwise form.
//
// For a chunk of c <= 64 tokens starting from state S0 (V x K), with per-channel cumulative
// log gates G_r = sum_{i<=r} g_i, Gamma_r = exp(G_r) and Gamma_c = Gamma of its last token:
//   A[r][j]  = beta_r sum_k k_r[k] k_j[k] exp(G_r[k] - G_j[k])   (j < r)
//   P[r][j]  =        sum_k q_r[k] k_j[k] exp(G_r[k] - G_j[k])   (j <= r)
//   W  = (I + A)^-1 Diag(beta) (K . Gamma),   U' = (I + A)^-1 Diag(beta) V
//   U  = U' - W S0^T              (row r of U is the delta d_r of token r)
//   O  = (Q . Gamma) S0^T + P U
//   S_c = S0 Diag(Gamma_c) + U^T B,           B = K . Gamma_c / Gamma
// Everything but S0 is known before the state is.  With
//   Z = B^T W (K x K),   N^T = B^T U' (K x V),   E = Q . Gamma - P W (c x K),   F = P U' (c x V)
// the two lines that involve the state become
//   S_c^T = Diag(Gamma_c) S0^T - Z S0^T + N^T,      O = E S0^T + F,
// so the sequential pass over chunks needs one tensor-core product per chunk.
//
// Launches:
//   chunk table  one warp: chunk_base[n] = chunks before sequence n (64-token chunks).
//   chunk        grid (chunk, head), 256 threads, two CTAs per SM: everything that does not
//                depend on the state, from the raw projections.  Conv and L2 norm; the gate
//                cumsum with one reference point per 16-token sub-chunk (every factor on
//                the tensor cores has an exponent <= 0 for a decaying gate; a sub-chunk
//                whose own spread is too wide gets its diagonal block in fp32); A and P as
//                one MMA; (I + A)^-1 by 16x16 blocks in fp32; [W | U'] as one MMA of
//                (I + A)^-1 Diag(beta) (split into bf16 high and low parts) with [K.Gamma | V];
//                [Z | N^T] = B^T [W | U'] and [P W | F] = P [W | U'] as two more MMAs.  Writes
//                per (chunk, head) a block of Z and E in the canonical K-major operand
//                layout, N^T and F by 32-column tiles, and Gamma_c.
//   state        grid (32-row tile of S, head, sequence): walks the sequence's chunks in
//                order with the tile's state in fp32 registers (thread k holds column k); per
//                chunk one MMA Z S0^T (Z the A operand in tensor memory), then the state
//                update; S0 of every chunk goes to the chunk's block.  Operand blocks arrive
//                by TMA bulk copies three chunks ahead.
//                The state pass also writes the slot's new conv window.
//   output       grid (chunk, head): O = E S0^T + F, one MMA per chunk and head.
#include "rsc_internal.h"
#include "rsc_step.cuh"
#include "rsc_tc.cuh"

namespace rsc {

namespace {

constexpr int kC = 64;      // chunk length
constexpr int kK = 128;     // key dim of the tensor-core path
constexpr int kVmax = 128;  // largest value dim
constexpr int kVT = 32;     // state rows per state-pass CTA
constexpr int kSub = 16;    // rows of a sub-chunk block (four per chunk)
// A diagonal 16-row block pairs k_r e^(G_r - Gb) with k_j e^(Gb - G_j), Gb the cumulative
// gate at the block's first row: the second factor grows with the block's own spread of the
// cumulative log gate.  Up to this spread (e^64 ~ 6e27, far inside the fp32 / bf16 range,
// and so is e^-64) the block stays on the tensor core; a wider block is recomputed in fp32
// from the exponent differences.
constexpr float kDiagSpread = 64.f;
constexpr float kMaxInv = 1e30f;  // clamp of e^(Gb - G_j) in a block beyond kDiagSpread
// A growing gate (g > 0) turns the references' exponents positive; beyond this exponent the
// chunk is flagged (RSC_DEVERR_GATE).  A decaying gate never reaches it.
constexpr float kGrowLimit = 60.f;
constexpr float kLog2e = 1.4426950408889634f;
// Layout of the A / P product.  Rows (tensor-memory lanes): block I's 16 key rows, then its 16
// query rows, at 32 I -- so lane quadrant I holds block I alone.  Columns: one segment per row
// block, at ap_seg(I), holding token j = 0 .. 16 I + 15 at ap_seg(I) + j: the earlier blocks'
// tokens (factors k_j h_j t, exponents <= 0) and then block I's own (k_j / f_j).  A row of block
// I reads its entries from one contiguous, warp-uniform window.
__host__ __device__ constexpr int ap_seg(int I) { return 8 * I * (I + 1); }
constexpr int kApN = ap_seg(4);  // 160 columns
__host__ __device__ constexpr int ap_row(int r, int is_q) { return 32 * (r >> 4) + 16 * is_q + (r & 15); }

// Per (chunk, head) operand block in the workspace (bytes).
constexpr size_t kOffZ = 0;                          // Z   128 x K  bf16, K-major (KD = K)
constexpr size_t kOffE = kOffZ + kK * kK * 2;        // E   64 x K   bf16, K-major (KD = K)
constexpr size_t kOffN = kOffE + kC * kK * 2;        // N^T as [V/32][K][32] bf16
constexpr size_t kOffF = kOffN + kK * kVmax * 2;     // F   as [V/32][64][32] bf16
constexpr size_t kOffGC = kOffF + kC * kVmax * 2;    // Gamma_c [K] fp32
// S0 of the chunk (bf16, V x K), written by the state pass for the output kernel: the
// MN-major B operand of E S0^T (n = v, contraction k), N = V.
constexpr size_t kOffS0 = ((kOffGC + kK * 4) + 1023) / 1024 * 1024;
constexpr size_t kBlockBytes = kOffS0 + kVmax * kK * 2;

// ---- chunk kernel shared memory (bytes)
// Phase 1: the chunk's raw rows (positions t0-3 .. t0+63, channels [q | k | v] of the
// head) and the conv outputs of its 64 tokens (q_hat | k_hat after the norm), rows padded.
constexpr int kStageRows = kC + 3;
constexpr int kRowElems = (2 * kK + kVmax) + 8;           // 392 bf16 = 784 bytes per row
constexpr uint32_t kChStg = 0;
constexpr uint32_t kChY = 53248;                           // >= 67 * 784
// Phase 2: tensor-core operands (overlaying phase 1; the V half of KV is written by the
// norm pass, once the staged rows are dead).
constexpr uint32_t kChKV = 0;        // [K.Gamma | V]        MN-major B, N = K + V, KD = 64
constexpr uint32_t kChX = 32768;     // [K.f; Q.f]             K-major 128 x K
constexpr uint32_t kChKc = 65536;    // columns of A / P       K-major 160 x K
// Written once the A / P product has completed (over its spent column operand); B^T leaves
// the registers it was formed in then.
constexpr uint32_t kChBT = 73728;    // B^T                    K-major K x 64
constexpr uint32_t kChPP = 90112;    // P                      K-major 64 x 64
// Phase 1 also: the conv taps of the head's channels (float4 each), transposed so that the
// lanes of a warp read consecutive vectors: the taps of channel 8 g + e at [e][g].
constexpr uint32_t kChW = 106496;
constexpr uint32_t kChSmem = kChW + (2 * kK + kVmax) * 16;  // 112640: two CTAs per SM
// Wide diagonal blocks (between the norm pass and the operands): the block's exponents
// G_r - Gb in fp32 (over the dead staged rows), and the exact diagonal-block values of A and
// P (over the dead taps; per block 120 strictly lower A entries, then 136 P entries).
constexpr int kGS = kK + 4;          // fp32 row stride of the staged exponents
constexpr uint32_t kChG = 32768;
constexpr uint32_t kChFb = kChW;
// Phase 3 (over X and Ki once the A/P product has completed).
constexpr int kAS = 68;                                  // fp32 row stride of A
constexpr uint32_t kChA = 32768;     // A, then (I + A)^-1 in place, fp32 [64][68]
constexpr int kSS = 52;                                  // fp32 row stride of the partials
constexpr uint32_t kChSt = kChA + kC * kAS * 4;          // block-row partial products [16][52]
constexpr uint32_t kChTH = 54272;    // (I + A)^-1 Diag(beta), high bf16 part, K-major 64 x 64
constexpr uint32_t kChTL = kChTH + kC * kC * 2;          // low part
// Phase 4 (over phase 3 once the [W | U'] product has completed).
constexpr uint32_t kChWU = 32768;    // [W | U']               MN-major B, N = K + V, KD = 64
constexpr uint32_t kChQG = 0;        // Q.Gamma back from the block, K-major 64 x K (over KV)
static_assert(kChY >= kStageRows * kRowElems * 2, "staging");
static_assert(kChY + kC * kRowElems * 2 <= kChSmem, "conv outputs");
static_assert(kChKV + kC * (kK + kVmax) * 2 <= kChY, "V half of KV beside the conv outputs");
static_assert(kChSt + 16 * kSS * 4 <= kChTH && kChTL + kC * kC * 2 <= kChBT, "phase 3");
static_assert(kChWU + kC * (kK + kVmax) * 2 <= kChBT, "phase 4");
static_assert(kChKc + kApN * kK * 2 == kChW && kChPP + kC * kC * 2 <= kChW, "A / P columns");
static_assert(kChBT + kK * kC * 2 <= kChPP && kChX + 2 * kC * kK * 2 == kChKc, "operands");
static_assert(kChG + kSub * kGS * 4 <= kChY && kChFb + 4 * 256 * 4 <= kChSmem, "wide blocks");

// ---- state pass shared memory (bytes): four operand buffers and two S0 buffers
constexpr uint32_t kSbZ = 0;                          // Z        128 x K K-major
constexpr uint32_t kSbN = kSbZ + kK * kK * 2;         // N^T tile [K][32]
constexpr uint32_t kSbGC = kSbN + kK * kVT * 2;       // Gamma_c  [K] fp32
constexpr uint32_t kSBuf = ((kSbGC + kK * 4) + 1023) / 1024 * 1024;
constexpr int kNBuf = 4;                              // operands fetched 3 chunks ahead
constexpr uint32_t kStS = kNBuf * kSBuf;              // S0 (bf16) x 2, MN-major B, N = 32, KD = K
constexpr uint32_t kSBytes = kVT * kK * 2;
constexpr uint32_t kStateSmem = kStS + 2 * kSBytes;
constexpr uint32_t kLoadBytes = kK * kK * 2 + kK * kVT * 2 + kK * 4;

// ---- output kernel shared memory (bytes)
constexpr uint32_t kOuE = 0;                          // E   64 x K K-major
constexpr uint32_t kOuS = kOuE + kC * kK * 2;         // S0  MN-major, N = V, KD = K
constexpr uint32_t kOuF = kOuS + kVmax * kK * 2;      // F   [V/32][64][32]
constexpr uint32_t kOutSmem = kOuF + kC * kVmax * 2;

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

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void fma4(float4 &acc, float a, const float4 &b) {
  acc.x = fmaf(a, b.x, acc.x); acc.y = fmaf(a, b.y, acc.y);
  acc.z = fmaf(a, b.z, acc.z); acc.w = fmaf(a, b.w, acc.w);
}

// Stage I of the blocked inverse: rows 16I .. 16I+15 of T = (I + A)^-1, columns below 16I.
// sA holds T in its rows < 16I (zeros above the diagonal), T's diagonal 16x16 blocks, and
// A in rows >= 16I.  The partials A[16I.., 0..16I) T[0..16I, 0..16I) go to sSt, then
// T[16I.., c] = -T_II (partials).  Writes the T rows into sA and T Diag(beta) as bf16
// high and low parts.
template <int I>
__device__ __forceinline__ void inverse_stage(float *sA, float *sSt, unsigned char *sTH,
                                              unsigned char *sTL, const float *s_beta, int tid) {
  constexpr int NQ = 4 * I;  // column quads per row
  const bool busy = tid < 16 * NQ;
  const int rr = tid / NQ, c = 4 * (tid % NQ);
  if (busy) {
    const float *arow = sA + (16 * I + rr) * kAS;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16 * I; m += 4) {
      const float4 a = ld4(arow + m);
      fma4(acc, a.x, ld4(sA + (m + 0) * kAS + c));
      fma4(acc, a.y, ld4(sA + (m + 1) * kAS + c));
      fma4(acc, a.z, ld4(sA + (m + 2) * kAS + c));
      fma4(acc, a.w, ld4(sA + (m + 3) * kAS + c));
    }
    st4(sSt + rr * kSS + c, acc);
  }
  __syncthreads();
  if (busy) {
    const float *trow = sA + (16 * I + rr) * kAS + 16 * I;  // row rr of T_II
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; m += 4) {
      const float4 a = ld4(trow + m);
      fma4(acc, a.x, ld4(sSt + (m + 0) * kSS + c));
      fma4(acc, a.y, ld4(sSt + (m + 1) * kSS + c));
      fma4(acc, a.z, ld4(sSt + (m + 2) * kSS + c));
      fma4(acc, a.w, ld4(sSt + (m + 3) * kSS + c));
    }
    const float t[4] = {-acc.x, -acc.y, -acc.z, -acc.w};
    st4(sA + (16 * I + rr) * kAS + c, make_float4(t[0], t[1], t[2], t[3]));
    float hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = t[e] * s_beta[c + e];
      hi[e] = __bfloat162float(__float2bfloat16_rn(x));
      lo[e] = x - hi[e];
    }
    const uint32_t off = tc::kmajor_offset(16 * I + rr, c, kC);  // 4 elements, 8 bytes
    *reinterpret_cast<uint2 *>(sTH + off) = make_uint2(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]));
    *reinterpret_cast<uint2 *>(sTL + off) = make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
  }
  __syncthreads();
}

// One lane's row rr of A (rows < 64 of the product) or of P, columns j0 .. j0+N-1, from N
// accumulator values d.  A: beta_r x value below the diagonal, fp32 rows of sA; P: the value
// on and below the diagonal of a live row, bf16 K-major.  In a block beyond kDiagSpread
// (WIDE) the row's own-block entries come from the exact values in fb.
struct ApRow {
  int rr, rb;
  bool isP, rwide, live;
  float br;
};
template <int N, bool WIDE>
__device__ __forceinline__ void ap_emit(const float *d, int j0, const ApRow &w, const float *fb,
                                        float *sA, unsigned char *sPP) {
#pragma unroll
  for (int g8 = 0; g8 < N / 8; ++g8) {
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = j0 + 8 * g8 + e;
      float x = d[8 * g8 + e];
      if constexpr (WIDE) {
        if ((j >> 4) == w.rb && j <= w.rr) {
          const int r = w.rr & 15, c = j & 15;
          x = w.isP ? fb[w.rb * 256 + 120 + r * (r + 1) / 2 + c]
                    : (c < r ? fb[w.rb * 256 + r * (r - 1) / 2 + c] : 0.f);
        }
      }
      v[e] = w.isP ? (j <= w.rr && w.live ? x : 0.f) : (j < w.rr ? w.br * x : 0.f);
    }
    const int j = j0 + 8 * g8;
    if (w.isP) {
      st16(sPP + tc::kmajor_offset(w.rr, j, kC), pack16(v));
    } else {
      st4(sA + w.rr * kAS + j, make_float4(v[0], v[1], v[2], v[3]));
      st4(sA + w.rr * kAS + j + 4, make_float4(v[4], v[5], v[6], v[7]));
    }
  }
}

// Exact diagonal block bI of A (raw, before beta) and P for a block beyond kDiagSpread, from
// the block's rows of q_hat | k_hat (Y, bf16) and its exponents x = G - Gb (sG, fp32):
// A[r][j] (j < r) = sum_c k_r k_j e^(x_r - x_j), P[r][j] (j <= r) = sum_c q_r k_j e^(x_r - x_j)
// (every exponent <= 0 for a decaying gate).  Thread pair (2p, 2p+1) sums pair p of the strictly
// lower triangle over the two channel halves; threads 240.. the P diagonal.  Out of line: the
// rare path stays out of the kernel's instruction stream.
__device__ __noinline__ void diag_block_exact(const bf16 *Y, const float *sG, float *fbb, int bI,
                                              int tid) {
  const int p = tid >> 1, hc = tid & 1;
  int r = 1;
  while ((r + 1) * r / 2 <= p) ++r;
  const int j = p - r * (r - 1) / 2;
  float a = 0.f, pp = 0.f;
  if (p < 120) {
    const bf16 *yr = Y + (kSub * bI + r) * kRowElems, *yj = Y + (kSub * bI + j) * kRowElems;
    const float *gr = sG + r * kGS, *gj = sG + j * kGS;
#pragma unroll 2
    for (int c = 64 * hc; c < 64 * hc + 64; c += 8) {
      float qr[8], kr[8], kj[8];
      unpack16(ld16(yr + c), qr);
      unpack16(ld16(yr + kK + c), kr);
      unpack16(ld16(yj + kK + c), kj);
      const float4 ra = ld4(gr + c), rb = ld4(gr + c + 4), ja = ld4(gj + c), jb = ld4(gj + c + 4);
      const float dx[8] = {ra.x - ja.x, ra.y - ja.y, ra.z - ja.z, ra.w - ja.w,
                           rb.x - jb.x, rb.y - jb.y, rb.z - jb.z, rb.w - jb.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float w = exp2f(dx[e] * kLog2e);
        a = fmaf(kr[e] * kj[e], w, a);
        pp = fmaf(qr[e] * kj[e], w, pp);
      }
    }
  } else {
    const bf16 *yr = Y + (kSub * bI + (tid - 240)) * kRowElems;
#pragma unroll 2
    for (int c = 0; c < kK; c += 8) {
      float qr[8], kr[8];
      unpack16(ld16(yr + c), qr);
      unpack16(ld16(yr + kK + c), kr);
#pragma unroll
      for (int e = 0; e < 8; ++e) pp = fmaf(qr[e], kr[e], pp);
    }
  }
  const float a2 = __shfl_xor_sync(0xffffffffu, a, 1);
  const float p2 = __shfl_xor_sync(0xffffffffu, pp, 1);
  if (p < 120) {
    if (hc == 0) {
      fbb[r * (r - 1) / 2 + j] = a + a2;
      fbb[120 + r * (r + 1) / 2 + j] = pp + p2;
    }
  } else {
    const int rd = tid - 240;
    fbb[120 + rd * (rd + 1) / 2 + rd] = pp;
  }
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

// Everything of one (chunk, head) that does not depend on the state: 256 threads.
//   1. conv + L2 norm: q_hat | k_hat rows (bf16) in shared memory, v straight into the V
//      half of the [K.Gamma | V] operand.
//   2. gates, in the layout of step 3 (thread t: channels 8 (t / 16) .. +7, rows
//      4 (t % 16) .. +3): cumsum by a 16-lane scan, per-channel midpoint R, Gamma_c.
//   3. operands, 16-byte stores: [K.e^(G-R); Q.e^(G-R)] and K.e^(R-G) for the A/P MMA,
//      K.Gamma for the W/U' MMA, B^T, and Q.Gamma (parked in the block's E slot).
//   4. A and P with one 128x64x128 MMA; A (x beta, strictly lower) to fp32, P to bf16.
//   5. T = (I + A)^-1 by 16x16 blocks; T Diag(beta) as bf16 high + low parts.
//   6. [W | U'] = T Diag(beta) [K.Gamma | V] (two accumulating MMAs), to shared memory.
//   7. [Z | N^T] = B^T [W | U'] -> block.   8. [P W | F] = P [W | U'] -> E = Q.Gamma - P W, F.
template <typename IO, int V, int GATE>
__global__ void __launch_bounds__(256, 2)
prefill_tc_chunk_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                        const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_base,
                        int N, const uint8_t *__restrict__ has_init, const IO *__restrict__ qkv,
                        const float *__restrict__ conv_w, const float *__restrict__ g,
                        const float *__restrict__ beta, char *__restrict__ blocks) {
  constexpr int NKV = kK + V;     // columns of [K.Gamma | V] and [W | U']
  constexpr int CH = 2 * kK + V;  // channels of one head
  extern __shared__ __align__(1024) unsigned char smem[];
  bf16 *Y = reinterpret_cast<bf16 *>(smem + kChY);
  unsigned char *sKV = smem + kChKV, *sX = smem + kChX;
  unsigned char *sBT = smem + kChBT, *sPP = smem + kChPP, *sWU = smem + kChWU;
  unsigned char *sTH = smem + kChTH, *sTL = smem + kChTL, *sQG = smem + kChQG;
  float *sA = reinterpret_cast<float *>(smem + kChA);
  float *sSt = reinterpret_cast<float *>(smem + kChSt);
  __shared__ uint32_t s_taddr;
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ __align__(8) uint64_t s_sbar;  // the staged rows (bulk copies)
  __shared__ float s_beta[kC];
  __shared__ int s_wide, s_grow;  // blocks beyond kDiagSpread (bit per block); a growing gate

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
  // tensor memory and the MMA barrier, ready long before the first product
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    mbar_init(&s_sbar, 1);
    s_wide = 0;
    s_grow = 0;
  }
  if (warp == 0) { tc::tmem_alloc(&s_taddr, 256); tc::tmem_relinquish(); }
  bool staged = true;  // the staging barrier completed (false: it timed out)

  // the gates of this thread's rows and channels: their lines are prefetched into L2 at once,
  // the registers filled after the q/k conv pass
  const int kg = tid >> 4, rsub = tid & 15;
  float G[4][8];
  if (GATE == RSC_GATE_KDA && (kg & 3) == 0) {  // the rows' gate lines into L2 meanwhile
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (4 * rsub + i < Lc) prefetch_l2(g + ((size_t)(t0 + 4 * rsub + i) * H + h) * kK + 8 * kg);
  }
  auto load_gates = [&]() {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * rsub + i;
    const size_t th = (size_t)(t0 + r) * H + h;
    if (r < Lc) {
      if constexpr (GATE == RSC_GATE_KDA) {
        const float4 a = ld4(g + th * kK + 8 * kg), b = ld4(g + th * kK + 8 * kg + 4);
        G[i][0] = a.x; G[i][1] = a.y; G[i][2] = a.z; G[i][3] = a.w;
        G[i][4] = b.x; G[i][5] = b.y; G[i][6] = b.z; G[i][7] = b.w;
      } else {
        const float x = g[th];
#pragma unroll
        for (int e = 0; e < 8; ++e) G[i][e] = x;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) G[i][e] = 0.f;
    }
  }
  };

  // ---- 1. conv + L2 norm -> Y rows 0..63: q_hat | k_hat; v (zero beyond the chunk) -> KV
  auto src_channel = [&](int c) {  // channel c of the head -> column of the projections
    return c < kK ? h * kK + c : c < 2 * kK ? H * kK + h * kK + (c - kK)
                                           : 2 * H * kK + h * V + (c - 2 * kK);
  };
  if constexpr (sizeof(IO) == 2) {
    // bf16 inputs: the chunk's rows (3 before it, from the sequence or the slot's window,
    // or zero for a fresh sequence) staged by bulk copies, three contiguous runs a row (the
    // head's q, k and v channels), completing on one barrier; then a sliding window per
    // (channel, half of the rows).  (Per-thread 16-byte copies took 3216 requests a chunk.)
    bf16 *stg = reinterpret_cast<bf16 *>(smem + kChStg);
    const IO *Wn = reinterpret_cast<const IO *>(pv.conv) +
                   ((size_t)layer * (pv.P + 1) + slot) * 3 * (size_t)D;
    const int p0 = t0 - seq0 - 3;   // sequence position of staged row 0
    auto copied = [&](int row) { return row - 3 < Lc && (p0 + row >= 0 || init); };
    __syncthreads();  // the staging barrier is initialised before any copy names it
    if (tid == 0) {
      uint32_t bytes = 0;
      for (int row = 0; row < kStageRows; ++row)
        if (copied(row)) bytes += CH * 2;
      mbar_arrive_expect_tx(&s_sbar, bytes);
    }
    for (int i = tid; i < kStageRows * 3; i += 256) {
      const int row = i / 3, c0 = (i % 3) * kK;  // runs start at channels 0, K, 2K
      const uint32_t nbytes = (c0 < 2 * kK ? kK : V) * 2;
      const int pos = p0 + row;
      bf16 *dst = stg + row * kRowElems + c0;
      if (copied(row)) {
        const IO *src = pos >= 0 ? qkv + (size_t)(seq0 + pos) * D : Wn + (size_t)(3 + pos) * D;
        bulk_g2s(dst, src + src_channel(c0), nbytes, &s_sbar);
      } else {
        for (uint32_t o = 0; o < nbytes; o += 16) st16(reinterpret_cast<char *>(dst) + o, make_uint4(0, 0, 0, 0));
      }
    }
    float4 *sW = reinterpret_cast<float4 *>(smem + kChW);
    for (int c = tid; c < CH; c += 256)
      cp_async16(sW + (c % 8) * (CH / 8) + c / 8, conv_w + 4 * (size_t)src_channel(c));
    cp_async_commit();
    cp_async_wait_all();
    staged = mbar_wait(&s_sbar, 0);
    __syncthreads();
    // q and k, conv and L2 norm in one pass: warp w takes tokens 8w .. 8w+7, lane l the eight
    // channels 8l .. 8l+7 of [q | k] (lanes 0-15 q, 16-31 k, so each row's sum of squares is
    // one reduction over a half warp); the fp32 conv outputs are normalised before rounding
    {
      const int g = lane;
      float4 w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = sW[e * (CH / 8) + g];
      const int r0 = 8 * warp;
      float x0[8], x1[8], x2[8];
      unpack16(ld16(stg + r0 * kRowElems + 8 * g), x0);
      unpack16(ld16(stg + (r0 + 1) * kRowElems + 8 * g), x1);
      unpack16(ld16(stg + (r0 + 2) * kRowElems + 8 * g), x2);
#pragma unroll
      for (int r = r0; r < r0 + 8; ++r) {
        float x3[8], y[8];
        unpack16(ld16(stg + (r + 3) * kRowElems + 8 * g), x3);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          y[e] = conv4(w[e], x0[e], x1[e], x2[e], x3[e]);
          ss = fmaf(y[e], y[e], ss);
          x0[e] = x1[e]; x1[e] = x2[e]; x2[e] = x3[e];
        }
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float rn = r < Lc ? rsqrtf(ss + kNormEps) : 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] *= rn;
        st16(Y + r * kRowElems + 8 * g, pack16(y));
      }
    }
    load_gates();  // after the q/k pass, whose registers they would crowd
    // v: thread (g, s) = (tid % 16, tid / 16) takes channels 8g .. 8g+7 of v on tokens
    // 4s .. 4s+3 (zero beyond the chunk)
    if (8 * (tid & 15) < V) {
      const int g = tid & 15, r0 = 4 * (tid >> 4);
      float4 w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = sW[e * (CH / 8) + 2 * kK / 8 + g];
      const bf16 *xs = stg + 2 * kK + 8 * g;
      float x0[8], x1[8], x2[8];
      unpack16(ld16(xs + r0 * kRowElems), x0);
      unpack16(ld16(xs + (r0 + 1) * kRowElems), x1);
      unpack16(ld16(xs + (r0 + 2) * kRowElems), x2);
#pragma unroll
      for (int r = r0; r < r0 + 4; ++r) {
        float x3[8], y[8];
        unpack16(ld16(xs + (r + 3) * kRowElems), x3);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          y[e] = r < Lc ? conv4(w[e], x0[e], x1[e], x2[e], x3[e]) : 0.f;
          x0[e] = x1[e]; x1[e] = x2[e]; x2[e] = x3[e];
        }
        st16(Y + r * kRowElems + 2 * kK + 8 * g, pack16(y));
      }
    }
    __syncthreads();  // the staged rows are dead from here
    // v into the V half of [K.Gamma | V] (over the staged rows): 16-byte pieces, token r,
    // columns K + 8g .. +7
    for (int i = tid; i < kC * (V / 8); i += 256) {
      const int r = i / (V / 8), g = i % (V / 8);
      st16(sKV + tc::mnmajor_offset(kK + 8 * g, r, NKV), ld16(Y + r * kRowElems + 2 * kK + 8 * g));
    }
  } else {
    // fp32 inputs: a warp per token straight from global memory (lane l owns channels
    // 4l..4l+3 of q, k, v).
    __syncthreads();  // the flags of step 2 are initialised
    load_gates();
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
      const float qq = group_sum<32>(yq[0] * yq[0] + yq[1] * yq[1] + yq[2] * yq[2] + yq[3] * yq[3]);
      const float kk = group_sum<32>(yk[0] * yk[0] + yk[1] * yk[1] + yk[2] * yk[2] + yk[3] * yk[3]);
      const bool live = r < Lc;
      const float rq = live ? 1.0f / sqrtf(qq + kNormEps) : 0.f;
      const float rk = live ? 1.0f / sqrtf(kk + kNormEps) : 0.f;
      bf16 *yr = Y + r * kRowElems;
      *reinterpret_cast<uint2 *>(yr + 4 * lane) =
          make_uint2(pack_bf16x2(yq[0] * rq, yq[1] * rq), pack_bf16x2(yq[2] * rq, yq[3] * rq));
      *reinterpret_cast<uint2 *>(yr + kK + 4 * lane) =
          make_uint2(pack_bf16x2(yk[0] * rk, yk[1] * rk), pack_bf16x2(yk[2] * rk, yk[3] * rk));
      if (has_v)
        *reinterpret_cast<uint2 *>(sKV + tc::mnmajor_offset(kK + 4 * lane, r, NKV)) =
            make_uint2(pack_bf16x2(yv[0], yv[1]), pack_bf16x2(yv[2], yv[3]));
    }
  }

  // ---- 2. cumulative gates: this thread's 4 rows by a local prefix, across the 16 lanes
  // of its half-warp (rows 4 rsub .. 4 rsub + 3) by a scan
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    G[1][e] += G[0][e];
    G[2][e] += G[1][e];
    G[3][e] += G[2][e];
  }
  {
    float incl[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) incl[e] = G[3][e];
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float y = __shfl_up_sync(0xffffffffu, incl[e], o, 16);
        if (rsub >= o) incl[e] += y;
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float ex = __shfl_up_sync(0xffffffffu, incl[e], 1, 16);
      if (rsub == 0) ex = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) G[i][e] += ex;
    }
  }
  // Sub-chunk references.  The chunk's rows form four 16-row blocks; this thread's rows lie
  // in block I = rsub / 4.  With Gb(J) the cumulative gate at the first row of block J and
  // G_last that of the chunk's last token, the factors
  //   f_r = e^(G_r - Gb(I)),   h_r = e^(Gb(I+1) - G_r)   (block 3: e^(G_last - G_r))
  // and, per channel, e^Gb(I), s = e^(G_last - Gb(I+1)), t_m = e^(Gb(I+m) - Gb(I+1)) all have
  // exponents <= 0 for a decaying gate.  From them:
  //   A / P rows          k_r f_r, q_r f_r
  //   own-block columns   k_j / f_j           (the block's spread; see kDiagSpread)
  //   earlier-block cols  k_j h_j t           (row block I' > J: t = e^(Gb(I') - Gb(J+1)))
  //   K.Gamma, Q.Gamma    k_r f_r e^Gb(I), q_r f_r e^Gb(I)
  //   B                   k_r h_r s
  // A pair of different blocks multiplies two factors <= 1, so nothing overflows and what
  // underflows is below fp32 range in the exact value too.  G is replaced by G - Gb(I).
  const int I = rsub >> 2;
  float d1[8], eGb[8], s1[8], t2[8], t3[8];
  {
    const int last = Lc - 1, src = last >> 2, il = last & 3;
    const int sb1 = 4 * min(I + 1, 3), sb2 = 4 * min(I + 2, 3);
    bool wide = false, grow = false;
    float gc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float gv = il == 0 ? G[0][e] : il == 1 ? G[1][e] : il == 2 ? G[2][e] : G[3][e];
      const float gl = __shfl_sync(0xffffffffu, gv, src, 16);
      const float gb0 = __shfl_sync(0xffffffffu, G[0][e], 4 * I, 16);
      const float gn = __shfl_sync(0xffffffffu, G[0][e], sb1, 16);
      const float gb2 = __shfl_sync(0xffffffffu, G[0][e], sb2, 16);
      const float gb3 = __shfl_sync(0xffffffffu, G[0][e], 12, 16);
      const float gb1 = I == 3 ? gl : gn;
      d1[e] = gb1 - gb0;
      eGb[e] = exp2f(gb0 * kLog2e);
      s1[e] = exp2f((gl - gb1) * kLog2e);
      t2[e] = exp2f((gb2 - gb1) * kLog2e);
      t3[e] = exp2f((gb3 - gb1) * kLog2e);
      gc[e] = expf(gl);
      grow |= gb0 > kGrowLimit || gl - gb1 > kGrowLimit || (I < 2 && gb2 - gb1 > kGrowLimit) ||
              (I == 0 && gb3 - gb1 > kGrowLimit);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float x = G[i][e] - gb0;
        G[i][e] = x;
        wide |= -x > kDiagSpread;
        grow |= x > kGrowLimit || d1[e] - x > kGrowLimit;
      }
    }
    if (wide) atomicOr(&s_wide, 1 << I);
    if (grow) s_grow = 1;
    if (rsub == 0) {
      float *gp = reinterpret_cast<float *>(blk + kOffGC) + 8 * kg;
      st4(gp, make_float4(gc[0], gc[1], gc[2], gc[3]));
      st4(gp + 4, make_float4(gc[4], gc[5], gc[6], gc[7]));
    }
  }

  // ---- 3. operands
  __syncthreads();  // the norm pass is complete; s_wide and s_grow are final
  const int wide_blocks = s_wide;
  if (tid == 0 && s_grow) flag_error(pv.err, RSC_DEVERR_GATE);
  float *fb = reinterpret_cast<float *>(smem + kChFb);
  if (wide_blocks) {
    // Diagonal blocks beyond kDiagSpread, exactly (diag_block_exact), one block at a time:
    // its exponents x = G - Gb staged in fp32, then the block's A and P entries into fb.
    float *sG = reinterpret_cast<float *>(smem + kChG);
    for (int bI = 0; bI < 4; ++bI) {
      if (!((wide_blocks >> bI) & 1)) continue;
      if (I == bI) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float *gp = sG + (4 * (rsub & 3) + i) * kGS + 8 * kg;
          st4(gp, make_float4(G[i][0], G[i][1], G[i][2], G[i][3]));
          st4(gp + 4, make_float4(G[i][4], G[i][5], G[i][6], G[i][7]));
        }
      }
      __syncthreads();
      diag_block_exact(Y, sG, fb + bI * 256, bI, tid);
      __syncthreads();  // the staged exponents are reused by the next wide block
    }
  }
  uint4 qv[4], kv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bf16 *yr = Y + (4 * rsub + i) * kRowElems;
    qv[i] = ld16(yr + 8 * kg);
    kv[i] = ld16(yr + kK + 8 * kg);
  }
  __syncthreads();  // Y is dead; the operands overlay it
  unsigned char *sKc = smem + kChKc;
  uint32_t btp[2][8];  // B^T of the thread's rows, bf16 pairs (rows 4 rsub + 2 ip, + 1)
#pragma unroll
  for (int ip = 0; ip < 4; ip += 2) {  // rows in pairs: B^T takes two rows per 4-byte store
    float bt[8][2];
#pragma unroll
    for (int i = ip; i < ip + 2; ++i) {
      const int r = 4 * rsub + i;
      const bool live = r < Lc;
      float q8[8], k8[8], xk[8], xq[8], kd[8], kh[8], kgm[8], qgm[8];
      unpack16(qv[i], q8);
      unpack16(kv[i], k8);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = G[i][e] * kLog2e;
        const float f = exp2f(x), hh = exp2f(d1[e] * kLog2e - x);
        const float fi = fminf(exp2f(-x), kMaxInv), gam = f * eGb[e];
        xk[e] = k8[e] * f;
        xq[e] = q8[e] * f;
        kd[e] = k8[e] * fi;
        kh[e] = k8[e] * hh;
        kgm[e] = k8[e] * gam;
        qgm[e] = q8[e] * gam;
        bt[e][i - ip] = live ? kh[e] * s1[e] : 0.f;
      }
      st16(sX + tc::kmajor_offset(ap_row(r, 0), 8 * kg, kK), pack16(xk));
      st16(sX + tc::kmajor_offset(ap_row(r, 1), 8 * kg, kK), pack16(xq));
      st16(sKc + tc::kmajor_offset(ap_seg(I) + r, 8 * kg, kK), pack16(kd));
      if (I < 3) st16(sKc + tc::kmajor_offset(ap_seg(I + 1) + r, 8 * kg, kK), pack16(kh));
      if (I < 2) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = kh[e] * t2[e];
        st16(sKc + tc::kmajor_offset(ap_seg(I + 2) + r, 8 * kg, kK), pack16(y));
      }
      if (I < 1) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = kh[e] * t3[e];
        st16(sKc + tc::kmajor_offset(ap_seg(3) + r, 8 * kg, kK), pack16(y));
      }
      st16(sKV + tc::mnmajor_offset(8 * kg, r, NKV), pack16(kgm));
      st16(blk + kOffE + tc::kmajor_offset(r, 8 * kg, kK), pack16(qgm));  // Q.Gamma, E later
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) btp[ip >> 1][e] = pack_bf16x2(bt[e][0], bt[e][1]);
  }
  // B^T rows are 16 bytes of 8 consecutive tokens for one channel.  Lanes 2m and 2m+1 hold
  // tokens 8m .. 8m+3 and 8m+4 .. 8m+7 of the same 8 channels: they swap half their channels,
  // so that each ends with 4 channels x 8 tokens, i.e. four whole 16-byte rows.
  const bool odd = rsub & 1;
  uint4 btr[4];  // rows of channels 8 kg + 4 odd + c, tokens 8 (rsub / 2) .. +7
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t got[2];
#pragma unroll
    for (int q = 0; q < 2; ++q)
      got[q] = __shfl_xor_sync(0xffffffffu, odd ? btp[q][c] : btp[q][4 + c], 1);
    btr[c] = odd ? make_uint4(got[0], got[1], btp[0][4 + c], btp[1][4 + c])
                 : make_uint4(btp[0][c], btp[1][c], got[0], got[1]);
  }

  // ---- 4. A and P: [K.f; Q.f] (128 x K) times the 160 columns -> 128 x 160
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = s_taddr;
  if (tid == 0) {
#pragma unroll
    for (int ks = 0; ks < kK / 16; ++ks)
      tc::mma_bf16(taddr, tc::kmajor_desc(sX, kK, ks), tc::kmajor_desc(sKc, kK, ks),
                   tc::idesc_bf16<128, kApN>(), ks > 0);
    tc::mma_commit(&s_bar);
  }
  const int q4 = warp & 3, half = warp >> 2;
  bool ok = __syncthreads_and(staged && mbar_wait(&s_bar, 0));
  tc::fence_after_sync();
  if (ok) {
    // B^T over the spent column operand: 16-byte rows, the channel order rotated by lane pair
    // so that the 8 lanes of a quarter warp write 8 different 16-byte bank groups
    {
      const int m = rsub >> 1;
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2) {
        const int c = (c2 + m) & 3;
        const uint4 v = c == 0 ? btr[0] : c == 1 ? btr[1] : c == 2 ? btr[2] : btr[3];
        st16(sBT + tc::kmajor_offset(8 * kg + 4 * odd + c, 8 * m, kC), v);
      }
    }
    // Lane quadrant q4 is row block q4: lanes 0-15 its key rows (A), lanes 16-31 its query rows
    // (P).  Row rr's entry j (j < 16 q4 + 16) is column ap_seg(q4) + j; the quadrant's two
    // warps take alternate 16-column chunks.  P is zero beyond the block (an operand); A is
    // read only below its diagonal blocks.
    ApRow w;
    w.rb = q4;
    w.rr = 16 * q4 + (lane & 15);
    w.isP = lane >= 16;
    w.rwide = (wide_blocks >> q4) & 1;
    w.live = w.rr < Lc;
    w.br = s_beta[w.rr];
#pragma unroll 1
    for (int cidx = half; cidx < 4; cidx += 2) {
      const bool have = cidx <= q4;  // warp-uniform
      float d[16];
      if (have) {
        tc::tmem_ld16(tc::tmem_addr(taddr, 32 * q4, ap_seg(q4) + 16 * cidx), d);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) d[e] = 0.f;
      }
      if (have || w.isP) {
        // the exact diagonal values only in a block beyond kDiagSpread (warp-uniform), so the
        // common path never touches them
        if (w.rwide) ap_emit<16, true>(d, 16 * cidx, w, fb, sA, sPP);
        else ap_emit<16, false>(d, 16 * cidx, w, fb, sA, sPP);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();

  // ---- 5. T = (I + A)^-1 by 16x16 blocks.  Diagonal blocks: thread (I, c) < 64 solves
  // column c of block I by forward substitution; the others zero T Diag(beta) above them.
  float x[16];
  if (ok) {
    if (tid < 64) {
      const int I = tid >> 4, c = tid & 15;
      const float *ab = sA + 16 * I * kAS + 16 * I;
      // right-looking: once x[m] is known, every later row takes its term at once, so
      // the dependent chain is one FMA per row
      float acc[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) acc[r] = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        x[m] = m == c ? 1.f : (m > c ? -acc[m] : 0.f);
#pragma unroll
        for (int r = m + 1; r < 16; ++r) acc[r] = fmaf(ab[r * kAS + m], x[m], acc[r]);
      }
    } else {
      // the 6 blocks (I, J > I) x 4 core matrices x 8 rows, in both parts
      for (int idx = tid - 64; idx < 2 * 6 * 32; idx += 192) {
        const int mat = idx / 192, rem = idx % 192, b6 = rem / 32, w = rem % 32;
        const int I = b6 < 3 ? 0 : b6 < 5 ? 1 : 2;
        const int J = b6 < 3 ? b6 + 1 : b6 < 5 ? b6 - 1 : 3;
        const uint32_t off = ((2 * I + (w >> 4)) * 8 + 2 * J + ((w >> 3) & 1)) * 128 + (w & 7) * 16;
        st16((mat ? sTL : sTH) + off, make_uint4(0, 0, 0, 0));
      }
    }
  }
  __syncthreads();
  if (ok && tid < 64) {
    const int I = tid >> 4, c = tid & 15;
    const float bc = s_beta[16 * I + c];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      sA[(16 * I + r) * kAS + 16 * I + c] = x[r];
      const float v = x[r] * bc;
      const float hi = __bfloat162float(__float2bfloat16_rn(v));
      const uint32_t off = tc::kmajor_offset(16 * I + r, 16 * I + c, kC);
      st_bf16(sTH + off, hi);
      st_bf16(sTL + off, v - hi);
    }
  }
  __syncthreads();
  if (ok) {
    inverse_stage<1>(sA, sSt, sTH, sTL, s_beta, tid);
    inverse_stage<2>(sA, sSt, sTH, sTL, s_beta, tid);
    inverse_stage<3>(sA, sSt, sTH, sTL, s_beta, tid);
  }

  // ---- 6. [W | U'] = T Diag(beta) [K.Gamma | V]   (M = 64: row r in lane r % 16 of
  // quadrant r / 16)
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (ok && tid == 0) {
#pragma unroll
    for (int ks = 0; ks < kC / 16; ++ks)
      tc::mma_bf16(taddr, tc::kmajor_desc(sTH, kC, ks), tc::mnmajor_desc(sKV, NKV, ks),
                   tc::idesc_bf16_bmn<64, NKV>(), ks > 0);
#pragma unroll
    for (int ks = 0; ks < kC / 16; ++ks)
      tc::mma_bf16(taddr, tc::kmajor_desc(sTL, kC, ks), tc::mnmajor_desc(sKV, NKV, ks),
                   tc::idesc_bf16_bmn<64, NKV>(), true);
    tc::mma_commit(&s_bar);
  }
  if (ok) ok = __syncthreads_and(mbar_wait(&s_bar, 1));
  tc::fence_after_sync();
  if (ok) {
    const int r = 16 * q4 + lane;      // lanes 0..15 hold rows
    const int c0 = half ? kK : 0, ncol = half ? V : kK;
    for (int cc = 0; cc < ncol; cc += 32) {
      float d[32];
      tc::tmem_ld32(tc::tmem_addr(taddr, 32 * q4, c0 + cc), d);
      if (lane < 16) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float a[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) a[e] = d[8 * q + e];
          st16(sWU + tc::mnmajor_offset(c0 + cc + 8 * q, r, NKV), pack16(a));
        }
      }
    }
  }

  // ---- 7. [Z | N^T] = B^T [W | U']   (M = 128: row k in lane k)
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // Q.Gamma (parked in the block's E slot by step 3) back into shared memory over the
  // spent [K.Gamma | V] operand, for step 8
  if (ok) {
#pragma unroll
    for (int i = 0; i < kC * kK * 2 / 16 / 256; ++i) {
      const int o = (tid + 256 * i) * 16;
      cp_async16(sQG + o, blk + kOffE + o);
    }
    cp_async_commit();
  }
  if (ok && tid == 0) {
#pragma unroll
    for (int ks = 0; ks < kC / 16; ++ks)
      tc::mma_bf16(taddr, tc::kmajor_desc(sBT, kC, ks), tc::mnmajor_desc(sWU, NKV, ks),
                   tc::idesc_bf16_bmn<128, NKV>(), ks > 0);
    tc::mma_commit(&s_bar);
  }
  if (ok) ok = __syncthreads_and(mbar_wait(&s_bar, 0));
  tc::fence_after_sync();
  if (ok) {
    const int k = 32 * q4 + lane;
    if (half == 0) {
      for (int cc = 0; cc < kK; cc += 32) {
        float d[32];
        tc::tmem_ld32(tc::tmem_addr(taddr, 32 * q4, cc), d);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float a[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) a[e] = d[8 * q + e];
          st16(blk + kOffZ + tc::kmajor_offset(k, cc + 8 * q, kK), pack16(a));
        }
      }
    } else {
      for (int cc = 0; cc < V; cc += 32) {
        float d[32];
        tc::tmem_ld32(tc::tmem_addr(taddr, 32 * q4, kK + cc), d);
        char *p = blk + kOffN + ((size_t)((cc / kVT) * kK + k) * kVT) * 2;  // one 32-column tile row
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float a[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) a[e] = d[8 * q + e];
          st16(p + 16 * q, pack16(a));
        }
      }
    }
  }
  cp_async_wait_all();  // this thread's part of Q.Gamma; the barrier below publishes it

  // ---- 8. [P W | F] = P [W | U'];  E = Q.Gamma - P W   (M = 64)
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (ok && tid == 0) {
#pragma unroll
    for (int ks = 0; ks < kC / 16; ++ks)
      tc::mma_bf16(taddr, tc::kmajor_desc(sPP, kC, ks), tc::mnmajor_desc(sWU, NKV, ks),
                   tc::idesc_bf16_bmn<64, NKV>(), ks > 0);
    tc::mma_commit(&s_bar);
  }
  const int r = 16 * q4 + lane;
  if (ok) ok = __syncthreads_and(mbar_wait(&s_bar, 1));
  tc::fence_after_sync();
  if (ok) {
    if (half == 0) {
      for (int cc = 0; cc < kK; cc += 32) {
        float d[32];
        tc::tmem_ld32(tc::tmem_addr(taddr, 32 * q4, cc), d);
        if (lane < 16) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t off = tc::kmajor_offset(r, cc + 8 * q, kK);
            float a[8];
            unpack16(ld16(sQG + off), a);
#pragma unroll
            for (int e = 0; e < 8; ++e) a[e] -= d[8 * q + e];
            st16(blk + kOffE + off, pack16(a));
          }
        }
      }
    } else {
      for (int cc = 0; cc < V; cc += 32) {
        float d[32];
        tc::tmem_ld32(tc::tmem_addr(taddr, 32 * q4, kK + cc), d);
        if (lane < 16) {
          char *p = blk + kOffF + ((size_t)((cc / kVT) * kC + r) * kVT) * 2;  // one 32-column tile row
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float a[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) a[e] = d[8 * q + e];
            st16(p + 16 * q, pack16(a));
          }
        }
      }
    }
  } else if (tid == 0) {
    flag_error(pv.err, RSC_DEVERR_TIMEOUT);
    if (!staged) mbar_wait(&s_sbar, 0);  // the staged rows land before shared memory is released
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(taddr, 256);
}

// Sequential state pass of one (32-row tile, head, sequence): per chunk S1^T = Gamma_c S0^T
// - Z S0^T + N^T, one 128x32x128 product on the path; S0 of every chunk also goes to the
// chunk's block for the output kernel.  Z is the product's A operand in tensor memory (two
// buffers): while chunk c's product runs, the threads move chunk c+1's Z from its operand
// buffer into the other one (thread k: row k), so the product itself reads only the 8 KB
// S0 operand from shared memory.  Warps 0-3 own the state (thread k: column k); warp 4
// only issues the products and the operand copies, so neither waits behind the other.
constexpr int kStateThreads = kK + 32;
template <typename IO, int V>
__global__ void __launch_bounds__(kStateThreads)
prefill_tc_state_kernel(PoolView pv, int layer, const int32_t *__restrict__ slots,
                        const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_base,
                        int T, const uint8_t *__restrict__ has_init, char *__restrict__ blocks,
                        const IO *__restrict__ qkv) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ uint32_t s_taddr;
  __shared__ __align__(8) uint64_t s_lbar[kNBuf];  // a buffer's operand block landed
  __shared__ __align__(8) uint64_t s_barz;         // Z S0^T of a chunk done
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
  auto block = [&](int c) { return blocks + ((size_t)(chunk_base[n] + c) * H + h) * kBlockBytes; };

  // The slot's window after the sequence: the last three raw inputs (rows before the
  // sequence's start come from the old window, or zero for a fresh sequence).  The chunk
  // kernel, which read the old window, has completed; this tile writes CHT of the head's
  // window channels (thread t: channel vt * CHT + t), the new rows requested now and stored
  // at the end.
  constexpr int CH = 2 * kK + V, CHT = CH / (V / kVT);
  static_assert(CHT <= kStateThreads, "a window channel per thread");
  IO *Wn = reinterpret_cast<IO *>(pv.conv) + prow * 3 * (size_t)pv.D;
  IO wnew[3];
  int wcol = -1;
  if (tid < CHT) {
    const int c = vt * CHT + tid;
    wcol = c < kK ? h * kK + c : c < 2 * kK ? H * kK + h * kK + (c - kK) : 2 * H * kK + h * V + (c - 2 * kK);
    const int len = end - start;
    IO old[3];
#pragma unroll
    for (int m = 0; m < 3; ++m) old[m] = init ? Wn[(size_t)m * pv.D + wcol] : from_f32<IO>(0.f);
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      const int pp = len - 3 + m;
      wnew[m] = pp >= 0 ? qkv[(size_t)(start + pp) * pv.D + wcol] : old[3 + pp];
    }
  }

  const bool owner = tid < kK;      // warps 0-3: thread k holds column k of the state tile
  const bool issuer = tid == kK;    // warp 4, lane 0: products and operand copies
  // state tile in registers, transposed: thread k holds S[v][k] for the tile's 32 rows v
  float S[kVT];
#pragma unroll
  for (int v = 0; v < kVT; ++v) S[v] = init && owner ? __bfloat162float(Sg[(size_t)v * kK + tid]) : 0.f;

  if (tid == 0) {
    for (int b = 0; b < kNBuf; ++b) mbar_init(&s_lbar[b], 1);
    mbar_init(&s_barz, 1);
    s_fail = 0;
  }
  if (warp == 0) { tc::tmem_alloc(&s_taddr, 256); tc::tmem_relinquish(); }
  // S0 of chunk c (bf16): into S buffer c & 1 as the MN-major B operand (element (v, k = tid))
  // and into chunk c's block, rows 32 vt .. +31 of the N = V operand there
  auto write_s0 = [&](int c) {
    unsigned char *sS = smem + kStS + (c & 1) * kSBytes;
    char *g = block(c) + kOffS0;
#pragma unroll
    for (int q = 0; q < kVT / 8; ++q) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = S[8 * q + e];
      const uint4 u = pack16(x);
      st16(sS + tc::mnmajor_offset(8 * q, tid, kVT), u);
      st16(g + tc::mnmajor_offset(kVT * vt + 8 * q, tid, V), u);
    }
  };
  if (nch > 0 && owner) write_s0(0);
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tDZ = s_taddr;  // Z S0^T: columns 0..31; Z of chunk c: columns 64 + 64 (c & 1) ..
  auto tA = [&](int c) { return tDZ + 64 + 64 * (uint32_t)(c & 1); };

  auto issue_load = [&](int c) {
    const int b = c % kNBuf;
    const char *blk = block(c);
    unsigned char *dst = smem + b * kSBuf;
    mbar_arrive_expect_tx(&s_lbar[b], kLoadBytes);
    bulk_g2s(dst + kSbZ, blk + kOffZ, kK * kK * 2, &s_lbar[b]);
    bulk_g2s(dst + kSbN, blk + kOffN + (size_t)vt * kK * kVT * 2, kK * kVT * 2, &s_lbar[b]);
    bulk_g2s(dst + kSbGC, blk + kOffGC, kK * 4, &s_lbar[b]);
  };
  // Z of chunk c (operand buffer c % 4, K-major rows) into tensor-memory buffer c & 1: row k
  // (thread k) as 64 columns of bf16 pairs, four 16-byte reads per 16 columns.
  auto stage_z = [&](int c) {
    if (!mbar_wait(&s_lbar[c % kNBuf], (c / kNBuf) & 1)) { s_fail = 1; return; }
    const unsigned char *zb = smem + (c % kNBuf) * kSBuf + kSbZ;
#pragma unroll
    for (int j0 = 0; j0 < kK / 8; j0 += 4) {
      uint32_t r[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = ld16(zb + tc::kmajor_offset(tid, 8 * (j0 + q), kK));
        r[4 * q] = v.x; r[4 * q + 1] = v.y; r[4 * q + 2] = v.z; r[4 * q + 3] = v.w;
      }
      tc::tmem_st16(tc::tmem_addr(tA(c), 32 * warp, 4 * j0), r);
    }
    tc::tmem_wait_st();
  };
  // Shared-memory descriptor of S buffer 0; the loop moves it by fixed offsets.
  const uint64_t dS0 = tc::mnmajor_desc(smem + kStS, kVT, 0);
  constexpr uint32_t kIdZ = tc::idesc_bf16_bmn<128, kVT>();

  // Chunk c (operand buffer c % 4, S0 in S buffer c & 1):
  //   the issuer starts Z S0^T and commits it, then fetches chunk c+3 into the buffer chunk
  //   c-1 used (its last readers finished before the last barrier); meanwhile warps 0-3
  //   stage chunk c+1's Z, read N^T and Gamma_c of their column, wait for Z S0^T, update
  //   the state and write S1 into the other S buffer (its last reader, chunk c-1's product,
  //   is done) and into chunk c+1's block -> barrier.  Waits on mbarriers are per thread and
  //   bounded; a failed one sets s_fail, which every thread reads after the next barrier, so
  //   all leave the loop together.
  int issued = 0;  // chunks whose operand copies were requested (every thread keeps it)
  bool ok = true;
  if (nch > 0) {
    if (issuer)
      for (int k = 0; k < nch && k < kNBuf - 1; ++k) issue_load(k);
    issued = nch < kNBuf - 1 ? nch : kNBuf - 1;
    if (owner) stage_z(0);
    tc::fence_before_sync();
    __syncthreads();
    if (s_fail) ok = false;
    tc::fence_after_sync();
  }
  int c = 0;
  for (; ok && c < nch; ++c) {
    const int b = c % kNBuf;
    const unsigned char *buf = smem + b * kSBuf;
    if (issuer) {
      // chunk c's Z is in tensor memory (staged and fenced before the last barrier)
      const uint64_t ds = tc::desc_add(dS0, (c & 1) * kSBytes);
#pragma unroll
      for (int ks = 0; ks < kK / 16; ++ks)
        tc::mma_bf16_ta(tDZ, tA(c) + 8 * ks, tc::desc_add(ds, ks * 2 * kVT * 16), kIdZ, ks > 0);
      tc::mma_commit(&s_barz);
      if (c + kNBuf - 1 < nch) issue_load(c + kNBuf - 1);
    }
    if (c + kNBuf - 1 < nch) issued = c + kNBuf;
    if (owner) {
      // the next chunk's Z into the other tensor-memory buffer (its last reader, chunk c-1's
      // product, is done) while this chunk's product runs
      if (c + 1 < nch) stage_z(c + 1);
      float nt[kVT];  // operand buffer b is visible: this thread waited for it when staging
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float f[8];
        unpack16(ld16(buf + kSbN + tid * kVT * 2 + 16 * q), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) nt[8 * q + e] = f[e];
      }
      const float gc = reinterpret_cast<const float *>(buf + kSbGC)[tid];
      if (!mbar_wait(&s_barz, c & 1)) s_fail = 1;
      tc::fence_after_sync();
      {
        // S_c^T[k][:] = Gamma_c[k] S0^T[k][:] - (Z S0^T)[k][:] + N^T[k][:] for this thread's k
        float d[kVT];
        tc::tmem_ld32(tc::tmem_addr(tDZ, 32 * warp, 0), d);
#pragma unroll
        for (int i = 0; i < kVT; ++i) S[i] = fmaf(gc, S[i], nt[i] - d[i]);
      }
      if (c + 1 < nch) {
        write_s0(c + 1);
        tc::fence_smem_to_async();
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (s_fail) { ok = false; break; }
    tc::fence_after_sync();
  }
  if (!ok) {
    if (issuer) {
      flag_error(pv.err, RSC_DEVERR_TIMEOUT);
      // let every requested bulk copy land before the shared memory is released
      for (int k = c; k < issued; ++k) mbar_wait(&s_lbar[k % kNBuf], (k / kNBuf) & 1);
    }
  } else if (owner) {
#pragma unroll
    for (int v = 0; v < kVT; ++v) Sg[(size_t)v * kK + tid] = __float2bfloat16_rn(S[v]);
  }
  if (wcol >= 0) {
#pragma unroll
    for (int m = 0; m < 3; ++m) Wn[(size_t)m * pv.D + wcol] = wnew[m];
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tDZ, 256);
}

// Outputs of one (chunk, head): O = E S0^T + F, one 64 x V x 128 product from the block
// (E, F from the chunk kernel, S0 from the state pass).  128 threads; token r of the
// chunk is lane r % 16 of warp r / 16.
template <typename IO, int V>
__global__ void __launch_bounds__(128)
prefill_tc_out_kernel(PoolView pv, const int32_t *__restrict__ slots,
                      const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_base,
                      int N, const char *__restrict__ blocks, IO *__restrict__ out) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ uint32_t s_taddr;
  __shared__ __align__(8) uint64_t s_lbar, s_bar;
  const int cid = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int H = pv.H;
  if (cid >= chunk_base[N]) return;
  const int n = last_le(chunk_base, N, cid);
  if (slots[n] < 0 || slots[n] > pv.P) return;  // flagged by the state pass
  const int t0 = cu[n] + kC * (cid - chunk_base[n]);
  const int Lc = min(kC, cu[n + 1] - t0);
  const char *blk = blocks + ((size_t)cid * H + h) * kBlockBytes;
  if (tid == 0) {
    mbar_init(&s_lbar, 1);
    mbar_init(&s_bar, 1);
    mbar_arrive_expect_tx(&s_lbar, kC * kK * 2 + V * kK * 2 + kC * V * 2);
    bulk_g2s(smem + kOuE, blk + kOffE, kC * kK * 2, &s_lbar);
    bulk_g2s(smem + kOuS, blk + kOffS0, V * kK * 2, &s_lbar);
    bulk_g2s(smem + kOuF, blk + kOffF, kC * V * 2, &s_lbar);
  }
  if (warp == 0) { tc::tmem_alloc(&s_taddr, V); tc::tmem_relinquish(); }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = s_taddr;
  bool ok = mbar_wait(&s_lbar, 0);  // the operands are visible to this thread
  if (tid == 0 && ok) {
#pragma unroll
    for (int ks = 0; ks < kK / 16; ++ks)
      tc::mma_bf16(taddr, tc::kmajor_desc(smem + kOuE, kK, ks), tc::mnmajor_desc(smem + kOuS, V, ks),
                   tc::idesc_bf16_bmn<64, V>(), ks > 0);
    tc::mma_commit(&s_bar);
  }
  ok = __syncthreads_and(ok && mbar_wait(&s_bar, 0));
  tc::fence_after_sync();
  if (ok) {
    const int r = 16 * warp + lane;
#pragma unroll
    for (int cc = 0; cc < V; cc += 32) {
      float d[32];
      tc::tmem_ld32(tc::tmem_addr(taddr, 32 * warp, cc), d);
      if (lane < 16 && r < Lc) {
        const unsigned char *fr = smem + kOuF + ((size_t)((cc / kVT) * kC + r) * kVT) * 2;
        float o[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float f[8];
          unpack16(ld16(fr + 16 * q), f);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[8 * q + e] = d[8 * q + e] + f[e];
        }
        IO *op = out + ((size_t)(t0 + r) * H + h) * V + cc;
        constexpr int EPV = 16 / sizeof(IO);
#pragma unroll
        for (int q = 0; q < 32 / EPV; ++q) {
          float y[EPV];
#pragma unroll
          for (int e = 0; e < EPV; ++e) y[e] = o[EPV * q + e];
          st16(op + EPV * q, pack16(y));
        }
      }
    }
  } else if (tid == 0) {
    flag_error(pv.err, RSC_DEVERR_TIMEOUT);
    mbar_wait(&s_lbar, 0);  // let the copies land before the shared memory is released
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(taddr, V);
}

// ---------------------------------------------------------------------------- launch

template <typename IO, int V, int GATE>
static int launch_tc_v(const LayerArgs &a, const int32_t *slots, const int32_t *cu, int N, int T,
                       const uint8_t *has_init, const void *qkv, const float *conv_w,
                       const float *g, const float *beta, void *out, int32_t *chunk_base,
                       char *blocks, cudaStream_t s) {
  auto chunk_kernel = prefill_tc_chunk_kernel<IO, V, GATE>;
  auto state_kernel = prefill_tc_state_kernel<IO, V>;
  auto out_kernel = prefill_tc_out_kernel<IO, V>;
  static PerDeviceFlag attr;  // per instantiation and device
  const int rc = once_per_device(attr, [&] {
    return cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kChSmem) == cudaSuccess &&
                   cudaFuncSetAttribute(state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kStateSmem) == cudaSuccess &&
                   cudaFuncSetAttribute(out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kOutSmem) == cudaSuccess
               ? RSC_OK
               : RSC_ECUDA;
  });
  if (rc != RSC_OK) return rc;
  const unsigned cap = (unsigned)prefill_tc_chunk_capacity(N, T);
  if (cap > 0 && T > 0) {
    chunk_kernel<<<dim3(cap, a.pv.H), 256, kChSmem, s>>>(a.pv, a.layer, slots, cu, chunk_base, N,
                                                          has_init, static_cast<const IO *>(qkv),
                                                          conv_w, g, beta, blocks);
    if (launch_status() != RSC_OK) return RSC_ECUDA;
  }
  state_kernel<<<dim3(V / kVT, a.pv.H, N), kStateThreads, kStateSmem, s>>>(
      a.pv, a.layer, slots, cu, chunk_base, T, has_init, blocks, static_cast<const IO *>(qkv));
  if (launch_status() != RSC_OK) return RSC_ECUDA;
  if (cap > 0 && T > 0)
    out_kernel<<<dim3(cap, a.pv.H), 128, kOutSmem, s>>>(a.pv, slots, cu, chunk_base, N, blocks,
                                                         static_cast<IO *>(out));
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

/*
 * rsc_oracle.c -- plain, slow, fp64 CPU oracle of the slot-indexed recurrent-state
 * layer step (short conv + L2 norm + gated delta rule over a slot pool).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *  [p1] "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理" (xxmr.cn/news/181459),
 *       sections "Conv state", "KDA 的 recurrent update" / ReplaySSM replay steps,
 *       "Speculative decoding的Conv State部分", mamba track copy.
 *  [p2] "SGLang之KV Cache内存池机制" (yuyanqi.com), §8.2 KDA 层的状态结构 and
 *       §8.5 KDA 运行时的缓存使用 (decode pseudo-code: decay, delta, beta, rank-1, output).
 *  [p3] hotelren.com/news/5417338, §2.1 Temporal/SSM state 与 Conv state 两部分.
 *  [p4] "sglang-mamba-kv-cache-kimi-k3" (treerouter.ai blog), §3.2 KDA Linear Layer
 *       Fixed State Memory Calculation.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - L2 norm: x / sqrt(sum x^2 + eps) with eps = 1e-6 ([p1] replay step prints eps, no value).
 *  - q is not scaled: the output is o = S q.
 *  - conv: no bias, no activation; taps w[c][0..2] act on the window rows (oldest first),
 *    w[c][3] on the current input.
 *  - channel split of the conv output: [q: H*K | k: H*K | v: H*V], head-major in each block.
 *  - the output is read from the updated state ([p2] §8.5 computes o after h += k (x) v).
 *  - storage rounding (fp32 or bf16, round-to-nearest-even) happens only where the API
 *    stores: end of a decode call, end of a prefill call, each spec-cache entry.
 *
 * Everything is fp64; storage values are widened on load and rounded on store.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_GATE_KDA = 0, ORC_GATE_GDN = 1 };

#define ORC_EPS 1e-6

/* Pool description as the oracle sees it: host arrays laid out exactly as the pages'
 * pool ([p1] "Conv state" shapes; [p2] §8.2): ssm [layers][P+1][H][V][K] and
 * conv [layers][P+1][3][D], D = H*(2K+V); row 0 of each layer is the padding slot. */
typedef struct {
  int32_t num_layers, num_slots, H, K, V;
  int32_t state_dtype, conv_dtype, gate;
  void *ssm;
  void *conv;
} orc_pool;

/* ---------------------------------------------------------------- storage types */

double orc_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, fp32 exponent range), ties to
 * even, by scaling to an integer count of ulps and rounding that with nearbyint (the
 * default rounding mode is round-half-even). */
uint16_t orc_bf16_round(double x) {
  if (isnan(x)) return 0x7fc0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double ax = fabs(x);
  if (ax == 0.0) return sign;
  if (isinf(ax)) return sign | 0x7f80;
  int e;
  frexp(ax, &e);            /* ax = m * 2^e with m in [0.5, 1) */
  int E = e - 1;            /* ax in [2^E, 2^(E+1)) */
  if (E < -126) E = -126;   /* subnormal bf16: fixed spacing 2^-133 */
  double ulp = ldexp(1.0, E - 7);
  double r = nearbyint(ax / ulp) * ulp;
  if (r >= ldexp(1.0, 128)) return sign | 0x7f80; /* overflow to infinity */
  float f = (float)r;       /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)(u >> 16);
}

static double ld(const void *base, size_t i, int dt) {
  if (dt == ORC_F32) return (double)((const float *)base)[i];
  return orc_bf16_to_double(((const uint16_t *)base)[i]);
}

static void st(void *base, size_t i, int dt, double x) {
  if (dt == ORC_F32) ((float *)base)[i] = (float)x;
  else ((uint16_t *)base)[i] = orc_bf16_round(x);
}

static size_t dsize(int dt) { return dt == ORC_F32 ? 4 : 2; }

/* ---------------------------------------------------------------- short conv */

/* One token of the depthwise causal conv with kernel 4 ([p1] "Conv state": the current
 * token mixes with the previous kernel_size-1 = 3 tokens, so the window keeps the last 3
 * projected q/k/v vectors, q included).  win is [3][D], row 0 oldest. */
void orc_conv_token(int D, double *win, const double *x, const float *w, double *y) {
  for (int c = 0; c < D; ++c) {
    y[c] = (double)w[4 * c + 0] * win[c] + (double)w[4 * c + 1] * win[D + c] +
           (double)w[4 * c + 2] * win[2 * D + c] + (double)w[4 * c + 3] * x[c];
  }
  for (int c = 0; c < D; ++c) {
    win[c] = win[D + c];
    win[D + c] = win[2 * D + c];
    win[2 * D + c] = x[c];
  }
}

/* T tokens of the conv from a given window (window updated in place). */
void orc_conv_sequence(int D, int T, double *win, const double *x, const float *w, double *y) {
  for (int t = 0; t < T; ++t) orc_conv_token(D, win, x + (size_t)t * D, w, y + (size_t)t * D);
}

/* ---------------------------------------------------------------- delta rule */

/* One token of the gated delta rule for one head, in the order of [p2] §8.5:
 *   decay   S <- S Diag(alpha)
 *   delta   u = S k ;  d = beta (v - u)
 *   write   S <- S + d k^T
 *   read    o = S q          (from the updated state)
 * S is V x K row-major (S[v][k]); alpha is a K-vector (KDA; a GDN head scalar is
 * broadcast by the caller).  d (length V) receives the delta vector. */
static void head_token(int K, int V, double *S, const double *q, const double *k,
                       const double *v, const double *alpha, double beta, double *o,
                       double *d) {
  for (int r = 0; r < V; ++r)
    for (int c = 0; c < K; ++c) S[(size_t)r * K + c] *= alpha[c];
  for (int r = 0; r < V; ++r) {
    double u = 0.0;
    for (int c = 0; c < K; ++c) u += S[(size_t)r * K + c] * k[c];
    d[r] = beta * (v[r] - u);
  }
  for (int r = 0; r < V; ++r)
    for (int c = 0; c < K; ++c) S[(size_t)r * K + c] += d[r] * k[c];
  for (int r = 0; r < V; ++r) {
    double acc = 0.0;
    for (int c = 0; c < K; ++c) acc += S[(size_t)r * K + c] * q[c];
    o[r] = acc;
  }
}

/* The recurrence of one head over T tokens with q, k, v, log-gate g ([T][K]) and beta
 * ([T]) given as they enter the delta rule (no conv, no normalisation).  S ([V][K]) is
 * updated in place; o is [T][V]; d_out ([T][V], may be NULL) receives every delta. */
void orc_recurrent_head(int T, int K, int V, const double *q, const double *k,
                        const double *v, const double *g, const double *beta, double *S,
                        double *o, double *d_out) {
  double *alpha = malloc(sizeof(double) * (size_t)K);
  double *d = malloc(sizeof(double) * (size_t)V);
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < K; ++c) alpha[c] = exp(g[(size_t)t * K + c]);
    head_token(K, V, S, q + (size_t)t * K, k + (size_t)t * K, v + (size_t)t * V, alpha,
               beta[t], o + (size_t)t * V, d);
    if (d_out) memcpy(d_out + (size_t)t * V, d, sizeof(double) * (size_t)V);
  }
  free(alpha);
  free(d);
}

/* ---------------------------------------------------------------- chunkwise form */

/* Chunkwise (WY / UT) form of the same recurrence, used only to check that it equals the
 * token-by-token result.  Derived from the unrolled closed form printed in [p1] (ReplaySSM
 * section: S_m = S_0 Diag(prod alpha) + sum_j d_j (k_j . prod_{i>j} alpha_i)^T) together
 * with d_j = beta_j (v_j - S_{j-1} Diag(alpha_j) k_j).  For a chunk of c tokens starting
 * from S0, with G_r = sum_{i<=r} g_i and Gamma_r = exp(G_r) per key channel:
 *   A[r][j] = beta_r sum_c k_r[c] k_j[c] exp(G_r[c] - G_j[c])          (j < r)
 *   Tm      = (I + A)^-1 Diag(beta)                                    (forward substitution)
 *   W       = Tm (K . Gamma) ;  U' = Tm V ;  Dm = U' - W S0^T           (rows of Dm are d_r)
 *   P[r][j] = sum_c q_r[c] k_j[c] exp(G_r[c] - G_j[c])                  (j <= r)
 *   O       = (Q . Gamma) S0^T + P Dm
 *   S_c     = S0 Diag(Gamma_c) + Dm^T (K . Gamma_c / Gamma)
 * Shapes as orc_recurrent_head; C is the chunk length (the last chunk may be shorter). */
int orc_chunkwise_head(int T, int K, int V, int C, const double *q, const double *k,
                       const double *v, const double *g, const double *beta, double *S,
                       double *o) {
  if (C <= 0 || K <= 0 || V <= 0 || T < 0) return -1;
  double *G = malloc(sizeof(double) * (size_t)C * K);
  double *A = malloc(sizeof(double) * (size_t)C * C);
  double *Tm = malloc(sizeof(double) * (size_t)C * C);
  double *W = malloc(sizeof(double) * (size_t)C * K);
  double *Up = malloc(sizeof(double) * (size_t)C * V);
  double *Dm = malloc(sizeof(double) * (size_t)C * V);
  double *Sn = malloc(sizeof(double) * (size_t)V * K);
  for (int t0 = 0; t0 < T; t0 += C) {
    int c = T - t0 < C ? T - t0 : C;
    const double *qc = q + (size_t)t0 * K, *kc = k + (size_t)t0 * K;
    const double *vc = v + (size_t)t0 * V, *gc = g + (size_t)t0 * K, *bc = beta + t0;
    double *oc = o + (size_t)t0 * V;
    /* cumulative log gates */
    for (int i = 0; i < K; ++i) {
      double acc = 0.0;
      for (int r = 0; r < c; ++r) {
        acc += gc[(size_t)r * K + i];
        G[(size_t)r * K + i] = acc;
      }
    }
    /* A, strictly lower */
    for (int r = 0; r < c; ++r)
      for (int j = 0; j < c; ++j) {
        double a = 0.0;
        if (j < r)
          for (int i = 0; i < K; ++i)
            a += kc[(size_t)r * K + i] * kc[(size_t)j * K + i] *
                 exp(G[(size_t)r * K + i] - G[(size_t)j * K + i]);
        A[(size_t)r * c + j] = bc[r] * a;
      }
    /* Tm = (I + A)^-1 Diag(beta): row r of Tm = beta_r e_r - sum_{j<r} A[r][j] Tm[j] */
    for (int r = 0; r < c; ++r)
      for (int j = 0; j < c; ++j) {
        double x = (j == r) ? bc[r] : 0.0;
        for (int m = 0; m < r; ++m) x -= A[(size_t)r * c + m] * Tm[(size_t)m * c + j];
        Tm[(size_t)r * c + j] = x;
      }
    /* W = Tm (K . Gamma), U' = Tm V */
    for (int r = 0; r < c; ++r) {
      for (int i = 0; i < K; ++i) {
        double x = 0.0;
        for (int j = 0; j < c; ++j)
          x += Tm[(size_t)r * c + j] * kc[(size_t)j * K + i] * exp(G[(size_t)j * K + i]);
        W[(size_t)r * K + i] = x;
      }
      for (int e = 0; e < V; ++e) {
        double x = 0.0;
        for (int j = 0; j < c; ++j) x += Tm[(size_t)r * c + j] * vc[(size_t)j * V + e];
        Up[(size_t)r * V + e] = x;
      }
    }
    /* Dm = U' - W S0^T */
    for (int r = 0; r < c; ++r)
      for (int e = 0; e < V; ++e) {
        double x = Up[(size_t)r * V + e];
        for (int i = 0; i < K; ++i) x -= W[(size_t)r * K + i] * S[(size_t)e * K + i];
        Dm[(size_t)r * V + e] = x;
      }
    /* O = (Q . Gamma) S0^T + (P masked) Dm */
    for (int r = 0; r < c; ++r)
      for (int e = 0; e < V; ++e) {
        double x = 0.0;
        for (int i = 0; i < K; ++i)
          x += qc[(size_t)r * K + i] * exp(G[(size_t)r * K + i]) * S[(size_t)e * K + i];
        for (int j = 0; j <= r; ++j) {
          double p = 0.0;
          for (int i = 0; i < K; ++i)
            p += qc[(size_t)r * K + i] * kc[(size_t)j * K + i] *
                 exp(G[(size_t)r * K + i] - G[(size_t)j * K + i]);
          x += p * Dm[(size_t)j * V + e];
        }
        oc[(size_t)r * V + e] = x;
      }
    /* S_c = S0 Diag(Gamma_c) + Dm^T (K . Gamma_c / Gamma) */
    for (int e = 0; e < V; ++e)
      for (int i = 0; i < K; ++i) {
        double gl = G[(size_t)(c - 1) * K + i];
        double x = S[(size_t)e * K + i] * exp(gl);
        for (int j = 0; j < c; ++j)
          x += Dm[(size_t)j * V + e] * kc[(size_t)j * K + i] * exp(gl - G[(size_t)j * K + i]);
        Sn[(size_t)e * K + i] = x;
      }
    memcpy(S, Sn, sizeof(double) * (size_t)V * K);
  }
  free(G); free(A); free(Tm); free(W); free(Up); free(Dm); free(Sn);
  return 0;
}

/* ---------------------------------------------------------------- layer step */

typedef struct {
  int H, K, V, D, gate;
  double *y, *qn, *kn, *alpha, *d;
} layer_ws;

static int ws_init(layer_ws *w, const orc_pool *p) {
  w->H = p->H; w->K = p->K; w->V = p->V; w->gate = p->gate;
  w->D = p->H * (2 * p->K + p->V);
  w->y = malloc(sizeof(double) * (size_t)w->D);
  w->qn = malloc(sizeof(double) * (size_t)w->K);
  w->kn = malloc(sizeof(double) * (size_t)w->K);
  w->alpha = malloc(sizeof(double) * (size_t)w->K);
  w->d = malloc(sizeof(double) * (size_t)w->V);
  return (w->y && w->qn && w->kn && w->alpha && w->d) ? 0 : -1;
}

static void ws_free(layer_ws *w) { free(w->y); free(w->qn); free(w->kn); free(w->alpha); free(w->d); }

static void l2norm(int n, const double *x, double *out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double s = 1.0 / sqrt(ss + ORC_EPS);
  for (int i = 0; i < n; ++i) out[i] = x[i] * s;
}

/* One token of one request over all heads: conv (window rolls), split, normalise q and
 * k, gate, delta rule.  win [3][D], S [H][V][K], x [D]; g_tok is [H][K] (KDA) or [H]
 * (GDN); beta_tok [H]; o [H][V]. */
static void layer_token(layer_ws *w, double *win, double *S, const double *x,
                        const float *conv_w, const float *g_tok, const float *beta_tok,
                        double *o) {
  const int H = w->H, K = w->K, V = w->V, D = w->D;
  orc_conv_token(D, win, x, conv_w, w->y);
  for (int h = 0; h < H; ++h) {
    const double *q = w->y + (size_t)h * K;
    const double *k = w->y + (size_t)H * K + (size_t)h * K;
    const double *v = w->y + (size_t)2 * H * K + (size_t)h * V;
    l2norm(K, q, w->qn);
    l2norm(K, k, w->kn);
    for (int c = 0; c < K; ++c)
      w->alpha[c] = exp(w->gate == ORC_GATE_KDA ? (double)g_tok[(size_t)h * K + c]
                                                : (double)g_tok[h]);
    head_token(K, V, S + (size_t)h * V * K, w->qn, w->kn, v, w->alpha, (double)beta_tok[h],
               o + (size_t)h * V, w->d);
  }
}

static size_t ssm_row_elems(const orc_pool *p) { return (size_t)p->H * p->V * p->K; }
static size_t conv_row_elems(const orc_pool *p) {
  return (size_t)3 * p->H * (2 * p->K + p->V);
}
static size_t ssm_row(const orc_pool *p, int layer, int slot) {
  return ((size_t)layer * (p->num_slots + 1) + slot) * ssm_row_elems(p);
}
static size_t conv_row(const orc_pool *p, int layer, int slot) {
  return ((size_t)layer * (p->num_slots + 1) + slot) * conv_row_elems(p);
}
static size_t gate_elems(const orc_pool *p) {
  return p->gate == ORC_GATE_KDA ? (size_t)p->H * p->K : (size_t)p->H;
}

static int check_slot(const orc_pool *p, int s) { return s >= 0 && s <= p->num_slots; }

/* Pool byte accounting of [p1]/[p4]: per layer and row, ssm H*V*K and conv 3*D elements;
 * rows = usable slots + 1 (the allocation logs of [p1] show one row more than the
 * reported slot count; row 0 is padding). */
void orc_pool_bytes(const orc_pool *p, uint64_t *ssm_bytes, uint64_t *conv_bytes) {
  uint64_t rows = (uint64_t)p->num_layers * (uint64_t)(p->num_slots + 1);
  *ssm_bytes = rows * ssm_row_elems(p) * dsize(p->state_dtype);
  *conv_bytes = rows * conv_row_elems(p) * dsize(p->conv_dtype);
}

/* Decode: one token per request; slot state read, updated, written back in place
 * ([p2] §8.5 forward_decode; cache_indices index the pool directly). */
int orc_decode_step(const orc_pool *p, int layer, const int32_t *slots, int B,
                    const void *qkv, const float *conv_w, const float *g,
                    const float *beta, void *out) {
  if (layer < 0 || layer >= p->num_layers) return -1;
  for (int b = 0; b < B; ++b)
    if (!check_slot(p, slots[b])) return -1;
  layer_ws w;
  if (ws_init(&w, p)) return -2;
  const int D = w.D, H = p->H, V = p->V;
  const size_t nS = ssm_row_elems(p), nW = conv_row_elems(p);
  double *S = malloc(sizeof(double) * nS), *win = malloc(sizeof(double) * nW);
  double *x = malloc(sizeof(double) * (size_t)D), *o = malloc(sizeof(double) * (size_t)H * V);
  for (int b = 0; b < B; ++b) {
    size_t sr = ssm_row(p, layer, slots[b]), cr = conv_row(p, layer, slots[b]);
    for (size_t i = 0; i < nS; ++i) S[i] = ld(p->ssm, sr + i, p->state_dtype);
    for (size_t i = 0; i < nW; ++i) win[i] = ld(p->conv, cr + i, p->conv_dtype);
    for (int c = 0; c < D; ++c) x[c] = ld(qkv, (size_t)b * D + c, p->conv_dtype);
    layer_token(&w, win, S, x, conv_w, g + (size_t)b * gate_elems(p), beta + (size_t)b * H, o);
    for (size_t i = 0; i < nS; ++i) st(p->ssm, sr + i, p->state_dtype, S[i]);
    for (size_t i = 0; i < nW; ++i) st(p->conv, cr + i, p->conv_dtype, win[i]);
    for (int i = 0; i < H * V; ++i) st(out, (size_t)b * H * V + i, p->conv_dtype, o[i]);
  }
  free(S); free(win); free(x); free(o);
  ws_free(&w);
  return 0;
}

/* Decode with the track copy ([p1] mamba_track_interval / track_mamba_states_if_needed: after
 * the forward step, if mask[b] then conv[track] = conv[active] and ssm[track] = ssm[active]):
 * the decode step, then the masked copy of this layer's rows. */
int orc_slot_copy(const orc_pool *p, int layer, const int32_t *src, const int32_t *dst,
                  const uint8_t *mask, int n);

int orc_decode_step_track(const orc_pool *p, int layer, const int32_t *slots, int B,
                          const void *qkv, const float *conv_w, const float *g, const float *beta,
                          void *out, const uint8_t *mask, const int32_t *track_slots) {
  int rc = orc_decode_step(p, layer, slots, B, qkv, conv_w, g, beta, out);
  if (rc) return rc;
  return orc_slot_copy(p, layer, slots, track_slots, mask, B);
}

/* Gates from the raw projections ([p2] §8.5 forward_decode takes the raw a, b of the layer;
 * "SGLang之KV Cache内存池机制" §10 names the fused sigmoid-gating decode kernel).  The pages
 * give no formula; the reading taken here (the usual KDA / GDN gating):
 *   beta = sigmoid(b) = 1 / (1 + e^-b)
 *   g    = -exp(A_log[h]) * softplus(a + dt_bias),  softplus(x) = log(1 + e^x)
 * with a and dt_bias per key channel (KDA: a [H][K], dt_bias [H][K]) or per head (GDN: a [H],
 * dt_bias [H]); A_log [H].  Written in forms that neither overflow nor lose small values:
 * softplus(x) = max(x, 0) + log1p(e^-|x|), sigmoid(x) = 1/(1 + e^-x) for x >= 0 and
 * e^x / (1 + e^x) otherwise. */
double orc_softplus(double x) { return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x))); }
double orc_sigmoid(double x) {
  if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
  double e = exp(x);
  return e / (1.0 + e);
}

/* Gates of one token batch: a [B][H][K] (KDA) or [B][H] (GDN), b [B][H] -> g (same shape as
 * a), beta [B][H], as fp32 (the type the layer step takes them in). */
void orc_gates_from_raw(int B, int H, int K, int gate, const float *a, const float *b,
                        const float *A_log, const float *dt_bias, float *g, float *beta) {
  const int n = gate == ORC_GATE_KDA ? K : 1;
  for (int i = 0; i < B; ++i)
    for (int h = 0; h < H; ++h) {
      const double scale = exp((double)A_log[h]);
      for (int c = 0; c < n; ++c) {
        const size_t e = ((size_t)i * H + h) * n + c;
        g[e] = (float)(-scale * orc_softplus((double)a[e] + (double)dt_bias[(size_t)h * n + c]));
      }
      beta[(size_t)i * H + h] = (float)orc_sigmoid((double)b[(size_t)i * H + h]);
    }
}

/* Decode with fused gating: the gates of the batch from the raw projections, then the
 * decode step. */
int orc_decode_step_gated(const orc_pool *p, int layer, const int32_t *slots, int B,
                          const void *qkv, const float *conv_w, const float *a, const float *b,
                          const float *A_log, const float *dt_bias, void *out) {
  const size_t ng = gate_elems(p);
  float *g = malloc(sizeof(float) * ng * (size_t)(B > 0 ? B : 1));
  float *beta = malloc(sizeof(float) * (size_t)p->H * (size_t)(B > 0 ? B : 1));
  orc_gates_from_raw(B, p->H, p->K, p->gate, a, b, A_log, dt_bias, g, beta);
  int rc = orc_decode_step(p, layer, slots, B, qkv, conv_w, g, beta, out);
  free(g); free(beta);
  return rc;
}

/* Prefill of N sequences packed along tokens (cu_seqlens [N+1]); sequence n starts from
 * its slot's state (or from zero when has_init is given and has_init[n] == 0), runs the
 * recurrence token by token and writes the final state back to the slot ([p2] §8.5
 * forward_extend: initial state from the pool, final state written back in place). */
int orc_prefill(const orc_pool *p, int layer, const int32_t *slots, const int32_t *cu_seqlens,
                int N, const uint8_t *has_init, const void *qkv, const float *conv_w,
                const float *g, const float *beta, void *out) {
  if (layer < 0 || layer >= p->num_layers) return -1;
  for (int n = 0; n < N; ++n)
    if (!check_slot(p, slots[n]) || cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  layer_ws w;
  if (ws_init(&w, p)) return -2;
  const int D = w.D, H = p->H, V = p->V;
  const size_t nS = ssm_row_elems(p), nW = conv_row_elems(p), ng = gate_elems(p);
  double *S = malloc(sizeof(double) * nS), *win = malloc(sizeof(double) * nW);
  double *x = malloc(sizeof(double) * (size_t)D), *o = malloc(sizeof(double) * (size_t)H * V);
  for (int n = 0; n < N; ++n) {
    size_t sr = ssm_row(p, layer, slots[n]), cr = conv_row(p, layer, slots[n]);
    int fresh = has_init && !has_init[n];
    for (size_t i = 0; i < nS; ++i) S[i] = fresh ? 0.0 : ld(p->ssm, sr + i, p->state_dtype);
    for (size_t i = 0; i < nW; ++i) win[i] = fresh ? 0.0 : ld(p->conv, cr + i, p->conv_dtype);
    for (int t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
      for (int c = 0; c < D; ++c) x[c] = ld(qkv, (size_t)t * D + c, p->conv_dtype);
      layer_token(&w, win, S, x, conv_w, g + (size_t)t * ng, beta + (size_t)t * H, o);
      for (int i = 0; i < H * V; ++i) st(out, (size_t)t * H * V + i, p->conv_dtype, o[i]);
    }
    for (size_t i = 0; i < nS; ++i) st(p->ssm, sr + i, p->state_dtype, S[i]);
    for (size_t i = 0; i < nW; ++i) st(p->conv, cr + i, p->conv_dtype, win[i]);
  }
  free(S); free(win); free(x); free(o);
  ws_free(&w);
  return 0;
}

/* Slot copy ([p1] mamba track copy: if mask[i], conv[dst] = conv[src] and ssm[dst] =
 * ssm[src]).  layer < 0 copies every layer.  Bytes are copied unchanged. */
int orc_slot_copy(const orc_pool *p, int layer, const int32_t *src, const int32_t *dst,
                  const uint8_t *mask, int n) {
  if (layer >= p->num_layers) return -1;
  for (int i = 0; i < n; ++i)
    if (!check_slot(p, src[i]) || !check_slot(p, dst[i])) return -1;
  int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? p->num_layers : layer + 1;
  size_t sb = ssm_row_elems(p) * dsize(p->state_dtype);
  size_t cb = conv_row_elems(p) * dsize(p->conv_dtype);
  for (int l = l0; l < l1; ++l)
    for (int i = 0; i < n; ++i) {
      if (mask && !mask[i]) continue;
      memcpy((char *)p->ssm + ssm_row(p, l, dst[i]) * dsize(p->state_dtype),
             (const char *)p->ssm + ssm_row(p, l, src[i]) * dsize(p->state_dtype), sb);
      memcpy((char *)p->conv + conv_row(p, l, dst[i]) * dsize(p->conv_dtype),
             (const char *)p->conv + conv_row(p, l, src[i]) * dsize(p->conv_dtype), cb);
    }
  return 0;
}

/* Speculative verify ([p1] "Speculative decoding的Conv State部分": the verify pass saves
 * the window after consuming each token into intermediate_conv_window[step]; the SSM
 * intermediate cache plays the same role for S).  For each request, run T tokens from the
 * slot state; after token t store S_t (rounded to the state dtype) into spec_ssm[b][t] and
 * the window into spec_conv[b][t].  The slot itself is not modified.  The running state
 * stays in fp64 across the T tokens.
 * spec_ssm [B][Lc][H][V][K], spec_conv [B][Lc][3][D], qkv [B][T][D], g [B][T][H][K] or
 * [B][T][H], beta [B][T][H], out [B][T][H][V]. */
int orc_spec_verify(const orc_pool *p, int layer, const int32_t *slots, int B, int T, int Lc,
                    void *spec_ssm, void *spec_conv, const void *qkv, const float *conv_w,
                    const float *g, const float *beta, void *out) {
  if (layer < 0 || layer >= p->num_layers || T < 1 || T > Lc) return -1;
  for (int b = 0; b < B; ++b)
    if (!check_slot(p, slots[b])) return -1;
  layer_ws w;
  if (ws_init(&w, p)) return -2;
  const int D = w.D, H = p->H, V = p->V;
  const size_t nS = ssm_row_elems(p), nW = conv_row_elems(p), ng = gate_elems(p);
  double *S = malloc(sizeof(double) * nS), *win = malloc(sizeof(double) * nW);
  double *x = malloc(sizeof(double) * (size_t)D), *o = malloc(sizeof(double) * (size_t)H * V);
  for (int b = 0; b < B; ++b) {
    size_t sr = ssm_row(p, layer, slots[b]), cr = conv_row(p, layer, slots[b]);
    for (size_t i = 0; i < nS; ++i) S[i] = ld(p->ssm, sr + i, p->state_dtype);
    for (size_t i = 0; i < nW; ++i) win[i] = ld(p->conv, cr + i, p->conv_dtype);
    for (int t = 0; t < T; ++t) {
      size_t bt = (size_t)b * T + t;
      for (int c = 0; c < D; ++c) x[c] = ld(qkv, bt * D + c, p->conv_dtype);
      layer_token(&w, win, S, x, conv_w, g + bt * ng, beta + bt * H, o);
      size_t e = (size_t)b * Lc + t;
      for (size_t i = 0; i < nS; ++i) st(spec_ssm, e * nS + i, p->state_dtype, S[i]);
      for (size_t i = 0; i < nW; ++i) st(spec_conv, e * nW + i, p->conv_dtype, win[i]);
      for (int i = 0; i < H * V; ++i) st(out, bt * H * V + i, p->conv_dtype, o[i]);
    }
  }
  free(S); free(win); free(x); free(o);
  ws_free(&w);
  return 0;
}

/* Speculative commit ([p1] fused_conv_window_scatter_with_mask: the snapshot of the last
 * accepted step is written back into the persistent state).  accept[b] = number of
 * accepted draft tokens a in [0, T-1]; the state after tokens 0..a is cache entry a. */
int orc_spec_commit(const orc_pool *p, int layer, const int32_t *slots, int B, int T, int Lc,
                    const void *spec_ssm, const void *spec_conv, const int32_t *accept) {
  if (layer < 0 || layer >= p->num_layers || T < 1 || T > Lc) return -1;
  for (int b = 0; b < B; ++b)
    if (!check_slot(p, slots[b]) || accept[b] < 0 || accept[b] >= T) return -1;
  size_t sb = ssm_row_elems(p) * dsize(p->state_dtype);
  size_t cb = conv_row_elems(p) * dsize(p->conv_dtype);
  for (int b = 0; b < B; ++b) {
    size_t e = (size_t)b * Lc + accept[b];
    memcpy((char *)p->ssm + ssm_row(p, layer, slots[b]) * dsize(p->state_dtype),
           (const char *)spec_ssm + e * sb, sb);
    memcpy((char *)p->conv + conv_row(p, layer, slots[b]) * dsize(p->conv_dtype),
           (const char *)spec_conv + e * cb, cb);
  }
  return 0;
}

/* ---------------------------------------------------------------- ReplaySSM */

/* ReplaySSM rings ("SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理", ReplaySSM
 * section; "Kimi K3 ... KV cache", §4 replay buffers): per pool row (slot) and head, `depth`
 * entries, each the records of one token:
 *   d     the delta beta (v - S k) the token wrote (length V)
 *   k     its L2-normalised key (K)
 *   g     its log-decay (K for KDA, one value for GDN)
 *   rawv  the value entering the delta rule, before v - S k (V)
 *   rawk  the key before its L2 norm (K)
 *   beta  its beta.
 * d, k, rawv, rawk are stored in the pool's state dtype (bf16 in the pages' deployment), g
 * and beta in fp32.  Layout [layers][P+1][H][depth][n].  Token t of a verify call for a
 * request whose ring position is pos goes to entry (pos + t) mod depth. */
typedef struct {
  int32_t depth;
  void *d, *k, *rawv, *rawk;
  float *g, *beta;
} orc_rings;

static size_t ring_at(const orc_pool *p, const orc_rings *R, int layer, int slot, int h, int e,
                      size_t n) {
  return ((((size_t)layer * (p->num_slots + 1) + slot) * p->H + h) * (size_t)R->depth + e) * n;
}

static int replay_args_ok(const orc_pool *p, const orc_rings *R, int layer, const int32_t *slots,
                          const int32_t *pos, int B, int T, int Lc) {
  if (layer < 0 || layer >= p->num_layers || T < 1 || T > Lc) return 0;
  if (R->depth < 1 || (R->depth & (R->depth - 1)) != 0 || 2 * T > R->depth) return 0;
  for (int b = 0; b < B; ++b)
    if (!check_slot(p, slots[b]) || pos[b] < 0 || pos[b] >= R->depth) return 0;
  return 1;
}

/* ReplaySSM verify: for each request run T tokens from the slot state (which is not
 * modified), as the snapshot verify does, but instead of storing S_t record the token's
 * (d, k, g, rawv, rawk, beta) in the rings at entry (pos[b] + t) mod depth.  The window
 * after token t goes to spec_conv[b][t] and the outputs to out, as in orc_spec_verify. */
int orc_replay_verify(const orc_pool *p, const orc_rings *R, int layer, const int32_t *slots,
                      const int32_t *pos, int B, int T, int Lc, void *spec_conv, const void *qkv,
                      const float *conv_w, const float *g, const float *beta, void *out) {
  if (!replay_args_ok(p, R, layer, slots, pos, B, T, Lc)) return -1;
  layer_ws w;
  if (ws_init(&w, p)) return -2;
  const int D = w.D, H = p->H, K = p->K, V = p->V, st_dt = p->state_dtype;
  const size_t nS = ssm_row_elems(p), nW = conv_row_elems(p), ng = gate_elems(p);
  const size_t gn = p->gate == ORC_GATE_KDA ? (size_t)K : 1;
  double *S = malloc(sizeof(double) * nS), *win = malloc(sizeof(double) * nW);
  double *x = malloc(sizeof(double) * (size_t)D), *o = malloc(sizeof(double) * (size_t)H * V);
  for (int b = 0; b < B; ++b) {
    size_t sr = ssm_row(p, layer, slots[b]), cr = conv_row(p, layer, slots[b]);
    for (size_t i = 0; i < nS; ++i) S[i] = ld(p->ssm, sr + i, st_dt);
    for (size_t i = 0; i < nW; ++i) win[i] = ld(p->conv, cr + i, p->conv_dtype);
    for (int t = 0; t < T; ++t) {
      const size_t bt = (size_t)b * T + t;
      const int e = (pos[b] + t) & (R->depth - 1);
      for (int c = 0; c < D; ++c) x[c] = ld(qkv, bt * D + c, p->conv_dtype);
      orc_conv_token(D, win, x, conv_w, w.y);
      for (int h = 0; h < H; ++h) {
        const double *q = w.y + (size_t)h * K;
        const double *k = w.y + (size_t)H * K + (size_t)h * K;
        const double *v = w.y + (size_t)2 * H * K + (size_t)h * V;
        const float *gt = g + bt * ng + (p->gate == ORC_GATE_KDA ? (size_t)h * K : (size_t)h);
        const float bh = beta[bt * H + h];
        l2norm(K, q, w.qn);
        l2norm(K, k, w.kn);
        for (int c = 0; c < K; ++c) w.alpha[c] = exp((double)gt[p->gate == ORC_GATE_KDA ? c : 0]);
        head_token(K, V, S + (size_t)h * V * K, w.qn, w.kn, v, w.alpha, (double)bh,
                   o + (size_t)h * V, w.d);
        const size_t rk = ring_at(p, R, layer, slots[b], h, e, (size_t)K);
        const size_t rv = ring_at(p, R, layer, slots[b], h, e, (size_t)V);
        for (int c = 0; c < K; ++c) {
          st(R->k, rk + c, st_dt, w.kn[c]);
          st(R->rawk, rk + c, st_dt, k[c]);
        }
        for (int r = 0; r < V; ++r) {
          st(R->d, rv + r, st_dt, w.d[r]);
          st(R->rawv, rv + r, st_dt, v[r]);
        }
        memcpy(R->g + ring_at(p, R, layer, slots[b], h, e, gn), gt, sizeof(float) * gn);
        R->beta[ring_at(p, R, layer, slots[b], h, e, 1)] = bh;
      }
      for (size_t i = 0; i < nW; ++i) st(spec_conv, ((size_t)b * Lc + t) * nW + i, p->conv_dtype, win[i]);
      for (int i = 0; i < H * V; ++i) st(out, bt * H * V + i, p->conv_dtype, o[i]);
    }
  }
  free(S); free(win); free(x); free(o);
  ws_free(&w);
  return 0;
}

/* ReplaySSM commit ([p3] exact commit of accepted tokens): from the slot state replay tokens
 * 0..accept[b] in order from the rings,
 *   k = rawk / sqrt(|rawk|^2 + eps),  alpha = exp(g),  S <- S Diag(alpha),
 *   d = beta (rawv - S k),  S <- S + d k^T,
 * in fp64, then store S (rounded to the state dtype) into the slot; the window becomes the
 * snapshot spec_conv[b][accept[b]]. */
int orc_replay_commit(const orc_pool *p, const orc_rings *R, int layer, const int32_t *slots,
                      const int32_t *pos, int B, int T, int Lc, const void *spec_conv,
                      const int32_t *accept) {
  if (!replay_args_ok(p, R, layer, slots, pos, B, T, Lc)) return -1;
  for (int b = 0; b < B; ++b)
    if (accept[b] < 0 || accept[b] >= T) return -1;
  const int H = p->H, K = p->K, V = p->V, st_dt = p->state_dtype;
  const size_t nS = ssm_row_elems(p), nW = conv_row_elems(p);
  const size_t gn = p->gate == ORC_GATE_KDA ? (size_t)K : 1;
  double *S = malloc(sizeof(double) * nS), *raw = malloc(sizeof(double) * (size_t)K);
  double *kn = malloc(sizeof(double) * (size_t)K);
  for (int b = 0; b < B; ++b) {
    const size_t sr = ssm_row(p, layer, slots[b]);
    for (size_t i = 0; i < nS; ++i) S[i] = ld(p->ssm, sr + i, st_dt);
    for (int t = 0; t <= accept[b]; ++t) {
      const int e = (pos[b] + t) & (R->depth - 1);
      for (int h = 0; h < H; ++h) {
        const size_t rk = ring_at(p, R, layer, slots[b], h, e, (size_t)K);
        const size_t rv = ring_at(p, R, layer, slots[b], h, e, (size_t)V);
        const float *gt = R->g + ring_at(p, R, layer, slots[b], h, e, gn);
        const double bh = R->beta[ring_at(p, R, layer, slots[b], h, e, 1)];
        for (int c = 0; c < K; ++c) raw[c] = ld(R->rawk, rk + c, st_dt);
        l2norm(K, raw, kn);
        double *Sh = S + (size_t)h * V * K;
        for (int r = 0; r < V; ++r) {
          double u = 0.0;
          for (int c = 0; c < K; ++c) {
            Sh[(size_t)r * K + c] *= exp((double)gt[gn == 1 ? 0 : c]);
            u += Sh[(size_t)r * K + c] * kn[c];
          }
          const double d = bh * (ld(R->rawv, rv + r, st_dt) - u);
          for (int c = 0; c < K; ++c) Sh[(size_t)r * K + c] += d * kn[c];
        }
      }
    }
    for (size_t i = 0; i < nS; ++i) st(p->ssm, sr + i, st_dt, S[i]);
    memcpy((char *)p->conv + conv_row(p, layer, slots[b]) * dsize(p->conv_dtype),
           (const char *)spec_conv + ((size_t)b * Lc + accept[b]) * nW * dsize(p->conv_dtype),
           nW * dsize(p->conv_dtype));
  }
  free(S); free(raw); free(kn);
  return 0;
}

/* Array helper for the Python wrapper: round n doubles to bf16 bit patterns. */
void orc_bf16_round_array(const double *x, uint16_t *out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = orc_bf16_round(x[i]);
}

/*
 * rsc.h -- C ABI of the GB300 slot-indexed recurrent-state cache (librsc.so).
 *
 * The library runs one layer step of a KDA / GDN linear-attention layer over a pool of
 * per-request recurrent states, entirely in hand-written sm_103a CUDA kernels:
 *   short conv (kernel 4, depthwise, causal) over the projected q/k/v with the slot's
 *   window of the last three raw inputs, L2 normalisation of q and k, and the gated
 *   delta rule on the slot's state S[H][V][K]:
 *       S <- S Diag(alpha);  d = beta (v - S k);  S <- S + d k^T;  o = S q
 *   with alpha = exp(g) per key channel (KDA) or per head (GDN).
 * Sources (web pages; cited by title and section):
 *   [p1] "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理" (xxmr.cn/news/181459):
 *        "Conv state" (window of the last 3 q/k/v vectors), the KDA recurrent update and
 *        its ReplaySSM replay steps (normalised key, alpha = exp(g), decay, delta, rank-1),
 *        the speculative conv-window snapshots and their scatter commit, and the masked
 *        track copy of conv and ssm state between slots.
 *   [p2] "SGLang之KV Cache内存池机制" (yuyanqi.com) §8.2 (pool shapes, row 0 padding)
 *        and §8.5 (forward_decode / forward_extend: state looked up by cache_indices,
 *        updated in place; chunked extend with chunk 64 and cu_seqlens).
 *   [p4] "sglang-mamba-kv-cache-kimi-k3" (treerouter.ai) §3.2 (conv and SSM state shapes).
 *
 * Conventions for every call
 *   - Every pointer argument documented "device" is CUDA device memory owned by the
 *     caller; the library never allocates, frees or retains device memory, except where
 *     a call says otherwise.  Pointers documented "host" are read before the call returns.
 *   - Device arrays read or written with 16-byte vector accesses must be 16-byte
 *     aligned: pool bases, qkv, out, conv_w, g, spec caches, workspace.  Other
 *     arrays need their element alignment.  Otherwise RSC_EALIGN.
 *   - Launches are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Host-side validation failures return a negative status before anything
 *     is launched.  A CUDA launch failure returns RSC_ECUDA.
 *   - Every call that launches runs on the current device, which must be the device that
 *     holds the pool's memory; otherwise it returns RSC_EDEVICE and launches nothing (the
 *     device of the pool is looked up on its first launching call and remembered).
 *   - Values the host cannot see (slot ids, accept counts, sequence offsets: all device
 *     arrays) are checked on the device.  A bad row is skipped (nothing of that row is
 *     written) and a bit is OR-ed into the pool's device error word; read it with
 *     rsc_get_device_error.  No kernel traps or asserts.
 *   - Slot ids within one call must be distinct (states are updated in place); slot 0
 *     is the padding row and is a legal target for padded batch entries.
 *   - Calls that touch the same slots must be ordered on one stream by the caller.
 */
#ifndef RSC_H
#define RSC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status codes */
#define RSC_OK        0
#define RSC_EINVAL   -1 /* null pointer, bad count, bad mode                        */
#define RSC_ERANGE   -2 /* layer, batch, length or cache depth out of range         */
#define RSC_EDTYPE   -3 /* unsupported dtype, gate, head dims or conv kernel        */
#define RSC_EALIGN   -4 /* a vector-accessed pointer is not 16-byte aligned         */
#define RSC_ECUDA    -5 /* a CUDA runtime call or launch failed                      */
#define RSC_ENOSPACE -6 /* caller-provided workspace too small                       */
#define RSC_EDEVICE  -7 /* the pool's memory is not device memory of the current device */

/* Bits of the device error word. */
#define RSC_DEVERR_SLOT   1 /* a slot id outside [0, num_slots]                      */
#define RSC_DEVERR_ACCEPT 2 /* an accept count outside [0, T-1]                      */
#define RSC_DEVERR_SEQ    4 /* cu_seqlens not non-decreasing within [0, total]       */
#define RSC_DEVERR_TIMEOUT 8 /* a bounded on-chip wait ran out; that tile was skipped  */
#define RSC_DEVERR_GATE   16 /* prefill: a growing gate (g > 0) raised a cumulative log
                                gate beyond what the blocked forms represent -- on the
                                tensor-core path by more than 60 above one of a chunk's
                                16-token reference points, on the other pools' blocked
                                path by more than 80 within an 8-token block; that block's
                                result is not reliable.  Never set for a decaying gate
                                (g <= 0), however strong.                             */
#define RSC_DEVERR_RING   32 /* a ReplaySSM ring position outside [0, depth)            */

typedef enum { RSC_F32 = 0, RSC_BF16 = 1 } rsc_dtype;
typedef enum { RSC_GATE_KDA = 0, RSC_GATE_GDN = 1 } rsc_gate;
typedef enum { RSC_SPEC_VERIFY = 0, RSC_SPEC_COMMIT = 1 } rsc_spec_mode;

/* Pool layout ([p2] §8.2; [p1] "Conv state"; [p4] §3.2), D = H*(2K+V):
 *   ssm  [num_layers][num_slots+1][H][V][K]  state_dtype, K contiguous
 *   conv [num_layers][num_slots+1][3][D]     conv_dtype, row 0 the oldest input;
 *        channels [q: H*K | k: H*K | v: H*V], head-major inside each block
 * Row 0 of each layer is padding.  conv_dtype is also the dtype of the projected
 * inputs (qkv) and of the outputs of every call.
 * Supported: head_k in {64, 128}, head_v in {64, 128}, conv_kernel == 4,
 * state_dtype and conv_dtype each RSC_F32 or RSC_BF16, gate KDA or GDN. */
typedef struct rsc_pool_desc {
  int32_t num_layers;
  int32_t num_slots;    /* usable slots P; the arrays hold P+1 rows per layer       */
  int32_t num_heads;    /* H (heads of this GPU's shard)                           */
  int32_t head_k;       /* K                                                       */
  int32_t head_v;       /* V                                                       */
  int32_t conv_kernel;  /* must be 4                                               */
  int32_t state_dtype;  /* rsc_dtype of ssm                                        */
  int32_t conv_dtype;   /* rsc_dtype of conv, qkv and outputs                      */
  int32_t gate;         /* rsc_gate                                                */
  void *ssm_base;       /* device, 16-byte aligned, caller-owned                    */
  void *conv_base;      /* device, 16-byte aligned, caller-owned                    */
  int32_t *dev_error;   /* device, one int32 zeroed by the caller, caller-owned      */
} rsc_pool_desc;

typedef struct rsc_pool rsc_pool; /* opaque host handle */

/* Validate a pool description and record its layout in a host handle (*out).  Owns no
 * device memory; performs no CUDA call.  Errors: RSC_EINVAL (null), RSC_ERANGE (counts),
 * RSC_EDTYPE (dims, dtypes, gate, conv kernel), RSC_EALIGN (bases). */
int ssm_pool_create(const rsc_pool_desc *desc, rsc_pool **out);

/* Free the host handle (NULL is a no-op).  Device memory stays the caller's. */
int ssm_pool_destroy(rsc_pool *pool);

/* Bytes the caller must allocate for ssm_base and conv_base of a description (only
 * the counts, dims and dtypes of desc are read).  Host only. */
int ssm_pool_bytes(const rsc_pool_desc *desc, uint64_t *ssm_bytes, uint64_t *conv_bytes);

/* Decode: one token per request ([p2] §8.5 forward_decode).
 *   slot_ids [batch]      device int32, distinct, each in [0, num_slots]
 *   qkv      [batch][D]   device, conv_dtype: projected inputs before the conv
 *   conv_w   [D][4]       device fp32: taps 0..2 act on window rows 0..2, tap 3 on qkv
 *   g        [batch][H][K] (KDA) or [batch][H] (GDN)  device fp32 log-decay, alpha=exp(g)
 *   beta     [batch][H]   device fp32
 *   out      [batch][H][V] device, conv_dtype: o = S q from the updated state
 * Each slot's window rolls (rows 1,2 move to 0,1; qkv lands in row 2) and its state is
 * updated in place; both are rounded once to their storage dtype.  batch == 0 is a
 * no-op.  Errors: RSC_EINVAL, RSC_ERANGE (layer), RSC_EALIGN, RSC_ECUDA. */
int kda_decode_step(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                    const void *qkv, const float *conv_w, const float *g,
                    const float *beta, void *out, void *stream);

/* Options of kda_decode_step_ex; zero-initialise and set what is wanted. */
#define RSC_DECODE_OVERLAP 1 /* launch as kda_decode_step_overlap does (same precondition) */
typedef struct rsc_decode_opts {
  const float *A_log;          /* fused gating (see kda_decode_step_gated) when non-NULL:  */
  const float *dt_bias;        /*   g and beta then carry the raw projections a and b     */
  const uint8_t *track_mask;   /* fused track copy (see kda_decode_step_track) when       */
  const int32_t *track_slots;  /*   non-NULL                                               */
  int flags;                   /* RSC_DECODE_OVERLAP or 0                                  */
} rsc_decode_opts;

/* The general decode call: kda_decode_step with any combination of fused gating, the fused
 * track copy and the overlapped launch; opts NULL is kda_decode_step.  Each option keeps the
 * layouts, alignment and preconditions of the entry point that has it alone; with gating and
 * tracking together the track slot receives the state updated with the formed gates.
 * Errors: as kda_decode_step; RSC_EINVAL also for an unknown flag, or for A_log without
 * dt_bias or track_mask without track_slots (or the reverse). */
int kda_decode_step_ex(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                       const void *qkv, const float *conv_w, const float *g, const float *beta,
                       void *out, const rsc_decode_opts *opts, void *stream);

/* kda_decode_step as a programmatic dependent launch of the previous kernel on `stream`, so
 * that this layer's state reads overlap the tail of the work before it.  The kernel may
 * start while the kernel just before it on the stream still runs; BEFORE waiting for it, it
 * reads slot_ids and layer `layer`'s state tiles and conv windows of those slots; qkv,
 * conv_w, g and beta are read, and every write is made, after the wait.  The kernel
 * releases its own dependents only after that wait, so when an overlapped call starts,
 * every kernel before its immediate predecessor has completed: its early reads can overlap
 * that one kernel alone.
 * Caller precondition: the kernel immediately before this call on `stream` does not write
 * slot_ids or those state and window rows (a caller's own programmatic-dependent kernel
 * placed there must also release its dependents only after its own griddepcontrol.wait).
 * Overlapped calls on different layers, one after another in any number and across steps
 * (a model step's graph replayed back to back), meet it; two consecutive calls on the same
 * layer and slots do not -- use kda_decode_step for the second.  Results are bit-identical
 * to kda_decode_step.
 * Errors: as kda_decode_step. */
int kda_decode_step_overlap(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                            const void *qkv, const float *conv_w, const float *g,
                            const float *beta, void *out, void *stream);

/* Decode with the track copy fused in ([p1] mamba_track_interval: when a request's length
 * reaches the tracking interval its mamba_track_mask is set and, after the forward step,
 * conv and ssm state of its active slot are copied into its tracking slot).  Exactly
 * kda_decode_step, and for every b with track_mask[b] != 0 the updated state and window of
 * slot_ids[b] are also written, byte for byte, into slot track_slots[b] (from the kernel's
 * registers: nothing is read back).
 *   track_mask  [batch] device uint8;  track_slots [batch] device int32 in [0, num_slots],
 *               distinct from every slot id of the call and from each other where the mask is
 *               set (caller precondition); out of range: RSC_DEVERR_SLOT and no track write.
 * Errors: RSC_EINVAL, RSC_ERANGE, RSC_EALIGN, RSC_ECUDA. */
int kda_decode_step_track(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                          const void *qkv, const float *conv_w, const float *g, const float *beta,
                          void *out, const uint8_t *track_mask, const int32_t *track_slots,
                          void *stream);

/* Decode with fused gating ([p2] §8.5: forward_decode(layer, mixed_qkv, a, b) hands the
 * layer's raw gate projections to the fused sigmoid-gating decode kernel named in §10).  The
 * pages give no gating formula; the reading implemented (the usual KDA / GDN gating):
 *   beta = sigmoid(b),   g = -exp(A_log[h]) * softplus(a + dt_bias),   alpha = exp(g)
 *   a        [batch][H][K] (KDA) or [batch][H] (GDN)  device fp32: raw decay projection
 *   b        [batch][H]   device fp32: raw beta projection
 *   A_log    [H]          device fp32
 *   dt_bias  [H][K] (KDA) or [H] (GDN)  device fp32
 * Otherwise exactly kda_decode_step.  a and dt_bias must be 16-byte aligned.
 * Errors: RSC_EINVAL, RSC_ERANGE, RSC_EALIGN, RSC_ECUDA. */
int kda_decode_step_gated(rsc_pool *pool, int layer, const int32_t *slot_ids, int batch,
                          const void *qkv, const float *conv_w, const float *a, const float *b,
                          const float *A_log, const float *dt_bias, void *out, void *stream);

/* Workspace bytes kda_prefill_chunk needs for num_seqs sequences of total_tokens
 * tokens (host only). */
int kda_prefill_workspace_size(const rsc_pool *pool, int num_seqs, int total_tokens,
                               size_t *bytes);

/* Chunked prefill ([p2] §8.5 forward_extend: initial state from the pool, final state
 * written back in place; sequences packed along tokens by cu_seqlens).  The result is
 * the token-by-token recurrence over each sequence; state and window are rounded once,
 * at the end of the call.
 *   slot_ids          [num_seqs]    device int32, distinct
 *   cu_seqlens        [num_seqs+1]  device int32, cu[0] = 0, non-decreasing, cu[N] = total
 *   has_initial_state [num_seqs]    device uint8 or NULL (= all 1); 0 starts that
 *                                   sequence from a zero state and a zero window
 *   qkv [total][D], g [total][H][K] or [total][H], beta [total][H], out [total][H][V]
 *   workspace         device, >= kda_prefill_workspace_size bytes, 16-byte aligned
 * bf16-state pools with head_k == 128 run the chunkwise form (chunk 64, every
 * contraction on the tcgen05 tensor cores with bf16 operands and fp32 accumulation);
 * any decaying gate (g <= 0, as the models' gates are) is exact to that precision,
 * however strong; a growing gate beyond the range above flags RSC_DEVERR_GATE.
 * Every other pool (fp32 state, or head_k == 64) runs the recurrence eight tokens at a
 * time in a closed form (exact algebra, fp32 on the CUDA cores, the state rounded once at
 * the end of the call; the same gate rule, with its own range).
 * Errors: RSC_EINVAL, RSC_ERANGE, RSC_EALIGN, RSC_ENOSPACE, RSC_ECUDA. */
int kda_prefill_chunk(rsc_pool *pool, int layer, const int32_t *slot_ids,
                      const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                      const uint8_t *has_initial_state, const void *qkv,
                      const float *conv_w, const float *g, const float *beta, void *out,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of the device scratch array behind kda_prefill_chunk_noalloc. */
#define RSC_PREFILL_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/* kda_prefill_chunk without a caller workspace.  The pages have no counterpart of this
 * call: it exists for callers that cannot allocate device memory when they prefill --
 * for example a serving engine that hands all of HBM to its own state and KV pools at
 * start-up (a later cudaMalloc fails or fragments its pools), or a latency-bound host
 * path that cannot afford cudaMalloc's implicit device synchronisation.
 * Arguments and results are those of kda_prefill_chunk minus the workspace.  The
 * scratch is a file-scope device array of RSC_PREFILL_STATIC_SCRATCH_BYTES (32 MiB)
 * that every GPU loading the library holds until the process exits.
 *   - The first call on a device looks up that device's address of the array
 *     (cudaGetSymbolAddress, with the device current); make that first call before
 *     any stream capture.
 *   - A call whose workspace need (kda_prefill_workspace_size) exceeds the array
 *     returns RSC_ENOSPACE before launching anything.
 *   - All calls share the one array and it keeps the last call's contents; nothing in
 *     it needs clearing (every byte a call reads was written earlier in that call).
 *     Calls that may overlap on the GPU (different streams, different host threads)
 *     race on the array: order them on one stream.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
int kda_prefill_chunk_noalloc(rsc_pool *pool, int layer, const int32_t *slot_ids,
                              const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                              const uint8_t *has_initial_state, const void *qkv,
                              const float *conv_w, const float *g, const float *beta,
                              void *out, void *stream);

/* Slot copy ([p1] masked track copy: conv[dst] = conv[src], ssm[dst] = ssm[src]).
 *   layer  >= 0 copies that layer, -1 copies every layer
 *   src, dst [n] device int32; dst distinct and disjoint from src
 *   mask     [n] device uint8 or NULL (= copy all); rows with mask 0 are skipped
 * Bytes are copied unchanged.  Errors: RSC_EINVAL, RSC_ERANGE, RSC_ECUDA. */
int ssm_slot_copy(rsc_pool *pool, int layer, const int32_t *src, const int32_t *dst,
                  const uint8_t *mask, int n, void *stream);

/* Speculative verify / commit ([p1] speculative decoding conv-state section: per-step
 * window snapshots, scatter of the last accepted step; the SSM intermediate cache works
 * the same way).
 *   VERIFY: for each request b run T tokens (anchor + drafts) from its slot state and
 *     store, after token t, S_t into spec_ssm[b][t] and the window into spec_conv[b][t]
 *     (rounded to their storage dtypes); out[b][t] = o_t.  The slot is not modified;
 *     the running state stays fp32 across the T tokens.  accept is ignored.
 *   COMMIT: slot_ids[b] <- entry accept[b] of request b (S and window), bytes unchanged.
 *     accept[b] = accepted drafts in [0, T-1].  qkv, conv_w, g, beta, out are ignored.
 *   spec_ssm  [batch][L][H][V][K] device, state_dtype;  spec_conv [batch][L][3][D]
 *   qkv [batch][T][D], g [batch][T][H][K] or [batch][T][H], beta [batch][T][H],
 *   out [batch][T][H][V];  1 <= T <= L, L a power of two.
 * Errors: RSC_EINVAL, RSC_ERANGE, RSC_EALIGN, RSC_ECUDA. */
int kda_spec_verify_commit(rsc_pool *pool, int layer, int mode, const int32_t *slot_ids,
                           int batch, int T, int L, void *spec_ssm, void *spec_conv,
                           const void *qkv, const float *conv_w, const float *g,
                           const float *beta, void *out, const int32_t *accept,
                           void *stream);

/* ReplaySSM rings of a pool ([p1] ReplaySSM section: the (d, k, g) records rebuild the
 * state from a checkpoint by the unrolled closed form, the (rawv, rawk, g, beta) records
 * replay accepted tokens exactly; [p4] §4 replay buffer table: six ring buffers per KDA
 * layer, depth L a power of two, L >= 2 x the tokens of one verify).  All device, owned by
 * the caller, indexed like the pool by [layer][slot (P+1 rows)][head][entry 0..depth-1]:
 *   d     [..][V]  state dtype   the delta beta (v - S k) the token wrote
 *   k     [..][K]  state dtype   its L2-normalised key
 *   rawv  [..][V]  state dtype   the value entering the delta rule (conv'd, before v - S k)
 *   rawk  [..][K]  state dtype   the conv'd key before its L2 norm
 *   g     [..][K] (KDA) or [..] (GDN)  fp32   its log-decay as given to the call
 *   beta  [..]     fp32          its beta
 * d, k, rawv, rawk, g must be 16-byte aligned, beta 4-byte aligned. */
typedef struct {
  int depth;
  void *d, *k, *rawv, *rawk;
  float *g, *beta;
} rsc_replay_rings;

/* ReplaySSM speculative verify / commit: the same contract as kda_spec_verify_commit, but
 * verify keeps no per-token states.
 *   VERIFY: for each request b run T tokens from its slot state (not modified); the records
 *     of token t go to entry (ring_pos[b] + t) mod depth of the slot's rings; the window
 *     after token t goes to spec_conv[b][t]; out[b][t] = o_t.  accept is ignored.
 *   COMMIT: from the slot state replay tokens 0..accept[b] out of the rings in fp32
 *     (k = rawk / sqrt(|rawk|^2 + eps), S <- S Diag(exp(g)), d = beta (rawv - S k),
 *     S <- S + d k^T), store the state into the slot and the window snapshot
 *     spec_conv[b][accept[b]].  qkv, conv_w, g, beta, out are ignored.
 *   ring_pos  [batch] device int32 in [0, depth), the entry of each request's token 0;
 *             advancing it between rounds is the caller's (RSC_DEVERR_RING if outside)
 *   spec_conv [batch][depth][3][D] device, conv dtype;  other arrays as in
 *   kda_spec_verify_commit;  1 <= T, 2 T <= depth, depth a power of two <= 4096.
 * Errors: RSC_EINVAL, RSC_ERANGE, RSC_EALIGN, RSC_ECUDA. */
int kda_replay_verify_commit(rsc_pool *pool, const rsc_replay_rings *rings, int layer, int mode,
                             const int32_t *slot_ids, const int32_t *ring_pos, int batch, int T,
                             void *spec_conv, const void *qkv, const float *conv_w,
                             const float *g, const float *beta, void *out,
                             const int32_t *accept, void *stream);

/* ------------------------------------------------------------------ host slot management
 * ([p2] §8.3 MambaPool.alloc: a state slot per request from the pool's free list; [p1] the
 * concurrency cap of the mamba state pool and the mamba_track_interval ping-pong track
 * slots).  Host only: no CUDA call, callable without a GPU. */
typedef struct rsc_slot_alloc rsc_slot_alloc;

/* An allocator over slots 1..num_slots (row 0, the padding row, is never handed out); slot 1
 * is handed out first.  Thread-safe.  Errors: RSC_EINVAL, RSC_ERANGE, RSC_ENOSPACE. */
int rsc_slot_alloc_create(int num_slots, rsc_slot_alloc **out);
int rsc_slot_alloc_destroy(rsc_slot_alloc *alloc);
int rsc_slot_alloc_free_count(rsc_slot_alloc *alloc, int *count);
/* n distinct free slots into slots[0..n) (host), or RSC_ENOSPACE and nothing taken. */
int rsc_slot_alloc_acquire(rsc_slot_alloc *alloc, int n, int32_t *slots);
/* Give n held slots back; a slot out of range (RSC_ERANGE), not held or repeated (RSC_EINVAL)
 * rejects the whole call and frees nothing. */
int rsc_slot_alloc_release(rsc_slot_alloc *alloc, int n, const int32_t *slots);

/* Requests a pool of num_slots can run at once: each reserves 3 slots, 2 more with the
 * overlap scheduler (its ping-pong track slots), 1 fewer with the decode-lock skip; the pages'
 * example: 80 slots at 5 per request cap the running requests at 16.  Host only. */
int rsc_max_running_requests(int num_slots, int overlap, int skip_decode_lock, int *out);

/* Track plan of one decode step (host arrays): request b is tracked when seq_lens[b] is a
 * positive multiple of interval; then mask[b] = 1, track_slots[b] =
 * track_pairs[b][next_idx[b]] and next_idx[b] moves to the other of its ntrack (1 or 2) track
 * slots (ping-pong); otherwise mask[b] = 0 and track_slots[b] = 0.  The outputs feed
 * kda_decode_step_track.  Errors: RSC_EINVAL, RSC_ERANGE. */
int rsc_track_plan(int batch, const int32_t *seq_lens, int interval, const int32_t *track_pairs,
                   int ntrack, int32_t *next_idx, uint8_t *mask, int32_t *track_slots);

/* Read the pool's device error word into *code and clear it.  Synchronises `stream`.
 * Errors: RSC_EINVAL, RSC_ECUDA. */
int rsc_get_device_error(rsc_pool *pool, int32_t *code, void *stream);

/* Static text for a status code (host only). */
const char *rsc_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* RSC_H */

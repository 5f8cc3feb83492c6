/*
 * kvs.h -- C ABI of the GB300 (sm_103a) KV-cache importance scoring and pruning library.
 *
 * The library computes, on one GPU, the data-parallel path shared by the KV-cache
 * eviction methods described in:
 *   [KVzap]  "KVzap: Fast, Adaptive, and Faithful KV Cache Pruning" (review):
 *            3.1 KVzip score (Eq. 1), 3.2 KVzip+ score (Eq. 2, Eq. 3), 3.3 KVzap
 *            surrogate, thresholding with a sliding window, Algorithm 1 (compress).
 *   [KVpop]  "[Paper review] KVpop -- Key-Value Cache Compression with Predictive
 *            Online Pruning": 1. Key Terms (future-attention target, transposed-
 *            attention pass reusing the attention kernel's LSE), 3. Method (per-head
 *            top-k).
 *   [KVzip]  KVzip review: Methods (teacher-forced repeat), technical details
 *            (chunked reconstruction).
 *
 * Conventions shared by every entry point
 *   - Tensor arguments are DEVICE pointers owned by the caller.  The library never
 *     allocates, frees or retains them.  Scratch memory, where an entry point needs
 *     it, is passed in by the caller (ws, ws_bytes) and sized by the matching
 *     kvs_*_workspace_size() function.
 *   - bf16 tensors are passed as raw 16-bit patterns (kvs_bf16).  All tensors are
 *     dense row-major with the innermost dimension last, as documented per call.
 *     Every pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls only enqueue work on it and return; none synchronises the host.
 *   - Return value: KVS_OK, or an error code with a message available from
 *     kvs_last_error() (thread-local, valid until the next call on that thread).
 *     Arguments are validated before anything is enqueued; on an error nothing is
 *     enqueued and no output is touched.
 *   - Query head hq reads KV head hq / g with g = H_q / H_kv (contiguous groups).
 *   - Logarithms are natural; the logit of query j and key i is q_j . k_i / sqrt(d),
 *     computed in fp32 from the bf16 inputs.
 */
#ifndef KVS_H_
#define KVS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvs_bf16; /* raw bfloat16 bit pattern */

typedef enum kvs_status {
  KVS_OK = 0,
  KVS_ERR_ARG = 1,         /* null pointer where one is required, negative size, bad mode */
  KVS_ERR_SHAPE = 2,       /* inconsistent sizes (H_q % H_kv != 0, n_q > keys, ...) */
  KVS_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  KVS_ERR_UNSUPPORTED = 4, /* a size the kernels do not handle (d not 64/128, ...) */
  KVS_ERR_CAPACITY = 5,    /* a caller-provided buffer (workspace) is too small */
  KVS_ERR_CUDA = 6,        /* the CUDA runtime reported an error at launch */
  KVS_ERR_DEVICE = 7       /* a kernel recorded a device-side error (see kvs_device_error) */
} kvs_status;

/* Model shape of one call.  L is the number of layers the call covers (each
 * tensor's leading dimension). */
typedef struct kvs_dims {
  int32_t L;    /* layers, >= 1 */
  int32_t H_q;  /* query heads, multiple of H_kv */
  int32_t H_kv; /* key/value heads, >= 1 */
  int32_t d;    /* head dimension: 64 or 128 */
  int32_t D_h;  /* hidden size (kvs_vnorm, kvs_score_max with h, kvs_surrogate*); else ignored */
} kvs_dims;

enum { KVS_THRESHOLD = 0, KVS_TOPK = 1 };

const char* kvs_version(void);
const char* kvs_last_error(void);

/* Number of kernels this library has enqueued since it was loaded (all threads, all
 * devices).  A diagnostic for counting launches around a region of interest. */
uint64_t kvs_launch_count(void);

/* Device-side error word shared by all kernels of the library on the current device
 * (0 = none; 1 = a bounded wait of a tensor-core kernel ran out, 3 = shared-memory
 * window misaligned, 4/5 = kvs_decode_step out of pages, 6 = kvs_value_refit met a
 * non-positive pivot).  Reading synchronises
 * `stream`; `clear` != 0 resets it to 0. */
kvs_status kvs_device_error(int32_t* code_out, int32_t clear, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_lse -- pass 1: per-query log-sum-exp normaliser [KVpop 1. Key Terms: the
 * transposed pass reuses the LSE normaliser of the attention kernel].
 *
 *   lse[l][hq][j] = ln sum_{i <= off + j} exp(q[l][hq][j] . key_i / sqrt(d))
 *
 * Keys are the concatenation [k_ctx | k_tail] of KV head hq / g: n_k = T + n_tail.
 * Causality is bottom-right aligned: the n_q queries are the last n_q positions of
 * the n_k-token sequence, off = n_k - n_q (the repeated block after context and
 * repeat prompt [KVzap 3.1; KVzip Methods], or self-attention when n_q == n_k).
 *
 *   q      [L][H_q][n_q][d]      bf16
 *   k_ctx  [L][H_kv][T][d]       bf16
 *   k_tail [L][H_kv][n_tail][d]  bf16   (may be NULL when n_tail == 0)
 *   lse    [L][H_q][n_q]         fp32   output
 * Requires 0 <= n_q <= T + n_tail.
 * ------------------------------------------------------------------------------- */
kvs_status kvs_lse(const kvs_dims* dims, const kvs_bf16* q, int32_t n_q,
                   const kvs_bf16* k_ctx, int32_t T, const kvs_bf16* k_tail, int32_t n_tail,
                   float* lse, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_attn_fwd -- attention forward that also returns its LSE normaliser, so that a
 * caller running attention anyway gets pass 1 for free [KVpop 1. Key Terms: the
 * transposed pass reuses the LSE the attention kernel returns; KVzap 3.2, Eq. 2: the
 * output of head hq at query j is sum_i a_ji v_i].
 *
 *   o[l][hq][j]   = sum_{i <= off + j} a_ji v_i,  a_ji = exp(q_j . key_i / sqrt(d) - lse_j)
 *   lse[l][hq][j] = exactly as kvs_lse
 *
 * Keys and values are [k_ctx | k_tail] and [v_ctx | v_tail] of KV head hq / g, with the
 * bottom-right causal alignment of kvs_lse.  The softmax weights are rounded to bf16
 * before they multiply V on the tensor cores; o is fp32-accumulated and stored as bf16.
 *
 *   q              [L][H_q][n_q][d]      bf16
 *   k_ctx, v_ctx   [L][H_kv][T][d]       bf16   (may be NULL when T == 0)
 *   k_tail, v_tail [L][H_kv][n_tail][d]  bf16   (may be NULL when n_tail == 0)
 *   o              [L][H_q][n_q][d]      bf16   output
 *   lse            [L][H_q][n_q]         fp32   output
 * Requires n_q <= T + n_tail.
 * ------------------------------------------------------------------------------- */
kvs_status kvs_attn_fwd(const kvs_dims* dims, const kvs_bf16* q, int32_t n_q,
                        const kvs_bf16* k_ctx, const kvs_bf16* v_ctx, int32_t T,
                        const kvs_bf16* k_tail, const kvs_bf16* v_tail, int32_t n_tail,
                        kvs_bf16* o, float* lse, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_score_max -- pass 2, KVzip / KVzip+ reduction [KVzap 3.1 Eq. 1, 3.2 Eq. 3].
 * Recomputes a_ji = exp(q_j . k_i / sqrt(d) - lse_j) tile by tile (the dense matrix
 * is never formed) and reduces each context key over the scoring queries and over
 * the query heads of its GQA group, in the log domain:
 *
 *   log_score[l][hk][i] = max_{hq in group(hk)} [ ln vnorm[l][hq][i]
 *                           + max_j ( q_j . k_i / sqrt(d) - lse[l][hq][j] - ln ||h[l][j]|| ) ]
 *                       = ln max_{hq, j} a_ji ||W_O^{(hq)} v_i|| / ||h_j||
 *
 * vnorm == NULL drops the value factor, h == NULL drops the hidden-state factor
 * (both NULL: the KVzip score ln s_i of Eq. 1).  All context keys are visible to all
 * scoring queries (the queries follow the context).
 *
 *   q         [L][H_q][n_q][d]  bf16   scoring queries (same as passed to kvs_lse)
 *   k_ctx     [L][H_kv][T][d]   bf16   context keys to score
 *   lse       [L][H_q][n_q]     fp32   from kvs_lse over the same queries
 *   vnorm     [L][H_q][T]       fp32   ||W_O^{(hq)} v_i|| from kvs_vnorm, or NULL
 *   h         [L][n_q][D_h]     bf16   residual-stream input at the queries, or NULL
 *   log_score [L][H_kv][T]      fp32   output; with accumulate != 0 the result is
 *                                      max(previous contents, new score) (chunked
 *                                      reconstruction [KVzip technical details])
 *   ws        scratch of kvs_score_max_workspace_size(dims, n_q, h != NULL) bytes: the
 *             per-query constants -(lse_j + ln||h_j||) sqrt(d) as three bf16 parts,
 *             which one extra K = 16 MMA step adds to every accumulator column (the
 *             size does not depend on h)
 * ------------------------------------------------------------------------------- */
size_t kvs_score_max_workspace_size(const kvs_dims* dims, int32_t n_q, int32_t with_h);
kvs_status kvs_score_max(const kvs_dims* dims, const kvs_bf16* q, int32_t n_q,
                         const kvs_bf16* k_ctx, int32_t T, const float* lse,
                         const float* vnorm, const kvs_bf16* h, int32_t accumulate,
                         float* log_score, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_score_future_sum -- pass 2, KVpop future-attention target [KVpop 1. Key Terms]:
 * the attention mass key i receives after it leaves the protected window of w tokens,
 * summed over the query heads of its group, for causal self-attention over T tokens:
 *
 *   score[l][hk][i] = sum_{hq in group(hk)} sum_{j = i + w}^{T - 1}
 *                       exp(q[l][hq][j] . k[l][hk][i] / sqrt(d) - lse[l][hq][j])
 *
 *   q     [L][H_q][T][d]  bf16,  k [L][H_kv][T][d] bf16
 *   lse   [L][H_q][T]     fp32   from kvs_lse(q, n_q = T, k_ctx = k, T, n_tail = 0)
 *   score [L][H_kv][T]    fp32   output (linear mass, not a log); keys i > T-1-w get 0
 *   ws    scratch of kvs_score_future_sum_workspace_size() bytes: the per-query
 *         constants -lse_j sqrt(d) as three bf16 parts, added to every accumulator
 *         column by one extra K = 16 MMA step
 * Requires w >= 0.
 * ------------------------------------------------------------------------------- */
size_t kvs_score_future_sum_workspace_size(const kvs_dims* dims, int32_t T);
kvs_status kvs_score_future_sum(const kvs_dims* dims, const kvs_bf16* q, const kvs_bf16* k,
                                int32_t T, const float* lse, int32_t w, float* score, void* ws,
                                size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_vnorm -- value factor of KVzip+ [KVzap 3.2, Eq. 2 and Eq. 3]:
 *
 *   vnorm[l][hq][i] = || W_O^{(hq)} v[l][hq/g][i] ||_2
 *
 * W_O^{(hq)} is the d-column slice hq*d .. hq*d+d-1 of the output projection
 * o_proj.weight [D_h][H_q*d].  Computed through the Gram matrix
 * G_hq = W_O^{(hq)T} W_O^{(hq)} (d x d, kept in the workspace as a pair of bf16
 * matrices whose sum carries G to ~2^-17 relative) as sqrt(v^T G v).
 *
 *   v     [L][H_kv][T][d]   bf16
 *   w_o   [L][D_h][H_q*d]   bf16
 *   vnorm [L][H_q][T]       fp32 output
 *   ws    scratch of kvs_vnorm_workspace_size() bytes (4*L*H_q*d*d)
 * Requires H_q / H_kv <= 16.
 * ------------------------------------------------------------------------------- */
size_t kvs_vnorm_workspace_size(const kvs_dims* dims);
kvs_status kvs_vnorm(const kvs_dims* dims, const kvs_bf16* v, int32_t T, const kvs_bf16* w_o,
                     float* vnorm, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_vnorm_noalloc -- kvs_vnorm without a caller-provided workspace.  The pages have
 * no counterpart: this entry point exists for callers that cannot allocate device
 * memory, e.g. a plugin inside a host framework that owns every device allocation, or
 * a serving loop that forbids allocation (and its implicit synchronisation) after
 * warm-up.  It computes the same vnorm as kvs_vnorm (same kernels, same results) and
 * allocates nothing: the Gram scratch is a device array built into the library, of
 * 8 MiB, which every GPU that loads the library keeps until the process exits.  Layers
 * are processed one after another on `stream`, so the limit is per layer:
 * H_q * d * d * 4 bytes <= 8 MiB (H_q <= 128 at d = 128); larger shapes return
 * KVS_ERR_CAPACITY.  The first call in each CUDA context looks up the array's device
 * address and caches it with the context's id: once per device, and once more after
 * the device's context is re-created (cudaDeviceReset), since the old address belongs
 * to the destroyed context.  Make each such first call before capturing a stream into
 * a graph.  All calls share the one array: calls that overlap on the GPU (other streams,
 * other host threads) race on it and must be serialised by the caller.  Nothing in it
 * needs to start at zero: every byte a call reads is written earlier by that call.
 *   v [L][H_kv][T][d] bf16,  w_o [L][D_h][H_q*d] bf16,  vnorm [L][H_q][T] fp32 output.
 * ------------------------------------------------------------------------------- */
kvs_status kvs_vnorm_noalloc(const kvs_dims* dims, const kvs_bf16* v, int32_t T,
                             const kvs_bf16* w_o, float* vnorm, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_surrogate -- KVzap-Linear score [KVzap 3.3; Algorithm 1, step 1]: at each
 * position t the hidden state h_t (D_h) maps to one predicted log-score per KV head,
 *
 *   score[l][hk][t] = sum_c h[l][t][c] * W[l][c][hk] + b[l][hk]
 *
 * Optionally fused with the threshold rule [KVzap, thresholding with a sliding
 * window]: when mask != NULL, mask[l][hk][t] = (score >= tau || t >= T - w) and
 * keep[l][hk] = number of kept tokens.
 *
 *   h     [L][T][D_h]   bf16,  W [L][D_h][H_kv] bf16,  b [L][H_kv] fp32
 *   score [L][H_kv][T]  fp32 output
 *   mask  [L][H_kv][T]  uint8 output or NULL;  keep [L][H_kv] int32 (required with mask)
 * Requires H_kv <= 16 and D_h a positive multiple of 128 with D_h * ceil(H_kv/8) <= 12800.
 * ------------------------------------------------------------------------------- */
kvs_status kvs_surrogate(const kvs_dims* dims, const kvs_bf16* h, int32_t T,
                         const kvs_bf16* W, const float* b, float* score,
                         float tau, int32_t w, uint8_t* mask, int32_t* keep, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_surrogate_mlp -- KVzap-MLP score [KVzap 3.3; training setup table: a two-layer
 * MLP per layer, D_h -> D_mid = D_h/8 -> H_kv; Appendix B: cost (D_h/4)(D_h + H)]:
 *
 *   u[c]             = sum_k h[l][t][k] * W1[l][c][k] + b1[l][c]        (c < D_mid)
 *   score[l][hk][t]  = sum_c GELU(u[c]) * W2[l][hk][c] + b2[l][hk]
 *
 * GELU(x) = x * Phi(x) (exact, erf form): the pages do not name the activation.
 * The first layer runs on the tensor cores (bf16 x bf16 -> fp32); GELU and the second
 * layer are fp32.  score is zeroed and accumulated in place (fp32 atomic adds of the
 * partial sums of D_mid split into parts of at most 256 columns, each a multiple of
 * 32).  With at most two parts (D_mid <= 256, or D_mid <= 512 with D_mid / 2 a
 * multiple of 32, as at D_h = 4096) the result is deterministic.  Optionally fused
 * with the threshold rule exactly as kvs_surrogate (mask != NULL).
 *
 *   h     [L][T][D_h]       bf16
 *   W1    [L][D_mid][D_h]   bf16 (out, in: a linear layer's weight),  b1 [L][D_mid] fp32
 *   W2    [L][H_kv][D_mid]  bf16 (out, in),                           b2 [L][H_kv]  fp32
 *   score [L][H_kv][T]      fp32 output
 *   mask  [L][H_kv][T]      uint8 output or NULL;  keep [L][H_kv] int32 (required with mask)
 * Requires D_h a positive multiple of 64, D_mid a positive multiple of 32, and
 * H_kv in {1, 2, 4, 8, 16}.
 * ------------------------------------------------------------------------------- */
kvs_status kvs_surrogate_mlp(const kvs_dims* dims, const kvs_bf16* h, int32_t T, int32_t D_mid,
                             const kvs_bf16* W1, const float* b1, const kvs_bf16* W2,
                             const float* b2, float* score, float tau, int32_t w,
                             uint8_t* mask, int32_t* keep, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_prune_mask -- keep mask per (layer, KV head) row of T scores.
 *   KVS_THRESHOLD [KVzap thresholding; Algorithm 1]: keep t  <=>  score >= tau or
 *                 t >= T - w.  A NaN score is dropped unless inside the window.
 *   KVS_TOPK      [KVpop 3. Method; KVzap 3.1 fixed-ratio KVzip]: keep the last w
 *                 tokens plus the k highest-scoring of the other T - w tokens (all of
 *                 them if k >= T - w).  Ranking: score descending, ties to the
 *                 earlier position, NaN below every number.
 *   score [L][H_kv][T] fp32;  mask [L][H_kv][T] uint8 output;  keep [L][H_kv] int32 output.
 * ------------------------------------------------------------------------------- */
kvs_status kvs_prune_mask(const kvs_dims* dims, const float* score, int32_t T, int32_t mode,
                          float tau, int32_t k, int32_t w, uint8_t* mask, int32_t* keep,
                          void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_prune_quantile -- threshold pruning with a per-layer threshold set at a quantile
 * of the layer's own scores [KVzip Methods: tau chosen so that a ratio of the scores
 * falls below it; KVzap thresholding with a sliding window; Algorithm 1].  Per layer l:
 *   tau[l] = the lower nearest-rank quantile q of the N = H_kv (T - w) non-window
 *            scores of all KV heads of layer l: the element of rank floor(q (N - 1))
 *            (0-based, ascending, computed in double from the fp32 q), NaN ranked
 *            below every number; +inf when N = 0
 *   keep t of head h  <=>  score[l][h][t] >= tau[l]  or  t >= T - w
 *   score [L][H_kv][T] fp32;  tau [L] fp32 output (device);  mask [L][H_kv][T] uint8
 *   output;  keep [L][H_kv] int32 output.  0 <= q <= 1, else KVS_ERR_ARG.
 * Every byte of mask and keep is written; until the masks are, the call keeps its
 * selection state in them (layers of at least 65536 non-window scores, with rows of at
 * least 4096, select over many blocks per layer), so neither may alias score or tau.
 * ------------------------------------------------------------------------------- */
kvs_status kvs_prune_quantile(const kvs_dims* dims, const float* score, int32_t T, float q,
                              int32_t w, float* tau, uint8_t* mask, int32_t* keep, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_prune_topk_multi -- the KVS_TOPK rule of kvs_prune_mask for several budgets over
 * the same scores in one launch [KVpop 3. Method: per-head top-k within a fixed
 * budget; KVzap 3.1: KVzip at fixed keep ratios].  For budget b the result equals
 * kvs_prune_mask(..., KVS_TOPK, k = k[b], w, ...) written at mask + b L H_kv T and
 * keep + b L H_kv.
 *   score [L][H_kv][T] fp32;  k [n_budgets] int32 in HOST memory, each >= 0;
 *   masks [n_budgets][L][H_kv][T] uint8 output;  keeps [n_budgets][L][H_kv] int32 output.
 * 1 <= n_budgets <= 8 (else KVS_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------------- */
kvs_status kvs_prune_topk_multi(const kvs_dims* dims, const float* score, int32_t T,
                                int32_t n_budgets, const int32_t* k, int32_t w, uint8_t* masks,
                                int32_t* keeps, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_value_refit -- closed-form value refit on the kept keys [KVSculpt summary,
 * 2. Method: with the keys fixed, the attention weights they induce are fixed and the
 * values follow by ridge least squares; Select+Fit = attention-score selection plus
 * this value fit].  Per (layer, KV head), with the g query heads' n_q scoring queries
 * stacked as n = g * n_q training rows, each seeing every context key:
 *
 *   O   = softmax(q K_ctx^T / sqrt d) V_ctx                  (full-context output, n x d)
 *   A_S = softmax(q K_kept^T / sqrt d) over the k kept keys  (n x k)
 *   v_fit = argmin ||A_S V - O||^2 + lam ||V||^2 = (A_S^T A_S + lam I)^-1 A_S^T O
 *   lam = lambda_rel * mean of the diagonal of A_S^T A_S
 *
 * O comes from the attention forward and A_S from the tensor cores, both kept in fp16
 * (weights in [0, 1] and attention outputs: 2^-12 relative each), so that the Gram
 * matrix and the right-hand side, accumulated in fp32 on the tensor cores, carry
 * ~2^-11 relative error; the ridge system is solved by an fp32 Cholesky factorisation.
 *
 *   q      [L][H_q][n_q][d]    bf16    k_ctx, v_ctx [L][H_kv][T][d] bf16
 *   k_kept [L][H_kv][k][d]     bf16    the kept keys in position order (for instance
 *                                      kvs_compact_paged with page_size = k)
 *   v_fit  [L][H_kv][k][d]     fp32    output
 *   ws     scratch of kvs_value_refit_workspace_size() bytes
 * Requires k <= T and k <= 8192.
 * ------------------------------------------------------------------------------- */
size_t kvs_value_refit_workspace_size(const kvs_dims* dims, int32_t n_q, int32_t k);
kvs_status kvs_value_refit(const kvs_dims* dims, const kvs_bf16* q, int32_t n_q,
                           const kvs_bf16* k_ctx, const kvs_bf16* v_ctx, int32_t T,
                           const kvs_bf16* k_kept, int32_t k, float lambda_rel, float* v_fit,
                           void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_decode_step -- decode-time pruning at the window boundary [KVzap: the threshold
 * criterion is phase-agnostic and prunes while decoding; KVpop 1. Key Terms: a token is
 * decided when it leaves the protected window].  One call = one decode step of B
 * sequences, for every (layer, KV head, sequence) row r = (l * H_kv + hk) * B + b:
 *
 *   the token arriving now (position pos[b]) enters the row's ring of the last w
 *   tokens at slot pos[b] % w; the token it displaces (position pos[b] - w, present
 *   once pos[b] >= w) is appended to the row's paged cache iff its score >= tau
 *   (NaN never passes).  With w == 0 the arriving token itself is decided.
 *
 * Over a whole sequence this keeps exactly the tokens that the prefill threshold rule
 * (kvs_prune_mask, KVS_THRESHOLD) keeps: the appended ones plus the final ring.
 * Pages: a row appends in position order into its own pages; when a row needs a new
 * page it takes next_page[0] (an atomic add on a device counter shared by all rows, so
 * page ids depend on the order rows run in; a row's contents do not), records it in
 * block_table[r][seq_lens[r] / page_size] and zero-fills it.  If the pool
 * (capacity_pages) or the row's block table (max_pages) is full the token is not
 * appended and the device error word is set (kvs_device_error: 4 = pool full,
 * 5 = block table full).  With advance_pos != 0, pos[b] += 1 after the step.
 *
 *   pos          [B]                     int32 (device; read, advanced if asked)
 *   new_score    [L][H_kv][B]            fp32  score of the arriving token
 *   new_k, new_v [L][H_kv][B][d]         bf16
 *   ring_score   [L][H_kv][B][w]         fp32  state (NULL when w == 0)
 *   ring_k, ring_v [L][H_kv][B][w][d]    bf16  state (NULL when w == 0)
 *   k_pages, v_pages [capacity_pages][page_size][d] bf16 state
 *   next_page    [1] int32 state;  block_table [L][H_kv][B][max_pages] int32 state
 *   seq_lens     [L][H_kv][B] int32 state (tokens appended so far)
 * Start a stream with pos = 0, seq_lens = 0, next_page = 0 and block_table = -1.
 * ------------------------------------------------------------------------------- */
kvs_status kvs_decode_step(const kvs_dims* dims, int32_t B, int32_t w, int32_t* pos,
                           const float* new_score, const kvs_bf16* new_k, const kvs_bf16* new_v,
                           float* ring_score, kvs_bf16* ring_k, kvs_bf16* ring_v, float tau,
                           int32_t page_size, kvs_bf16* k_pages, kvs_bf16* v_pages,
                           int32_t capacity_pages, int32_t* next_page, int32_t* block_table,
                           int32_t max_pages, int32_t* seq_lens, int32_t advance_pos,
                           void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_compact_paged -- gather of the kept K/V rows [KVzap Algorithm 1: keys[indices],
 * values[indices]] into a per-head variable-length paged cache (non-uniform head
 * lengths need PagedAttention-like storage [KVzap, limitation 3]).
 *
 * Layout: each (layer, head) row gets ceil(kept / page_size) consecutive pages,
 * allocated layer-major then head from page 0; kept tokens are stored in ascending
 * position; unused rows of a row's last page are zero-filled.
 *   block_table[l][hk][p] = absolute page id of the row's p-th page, -1 past the end
 *   seq_lens[l][hk]       = kept tokens;   needed_pages[0] = total pages (device int32)
 * If the total exceeds capacity_pages, no page is written and every block_table
 * entry is -1; needed_pages and seq_lens are still written, so the caller can read
 * needed_pages, grow the pool and call again.
 *
 *   k, v          [L][H_kv][T][d]                 bf16
 *   mask          [L][H_kv][T]                    uint8 (non-zero = keep)
 *   k_pages, v_pages [capacity_pages][page_size][d] bf16 outputs
 *   block_table   [L][H_kv][max_pages] int32, max_pages >= ceil(T / page_size)
 *   seq_lens      [L][H_kv] int32;  needed_pages [1] int32
 *   ws            scratch of kvs_compact_workspace_size() bytes
 * ------------------------------------------------------------------------------- */
size_t kvs_compact_workspace_size(const kvs_dims* dims, int32_t T);
kvs_status kvs_compact_paged(const kvs_dims* dims, const kvs_bf16* k, const kvs_bf16* v,
                             int32_t T, const uint8_t* mask, int32_t page_size,
                             kvs_bf16* k_pages, kvs_bf16* v_pages, int32_t capacity_pages,
                             int32_t* block_table, int32_t max_pages, int32_t* seq_lens,
                             int32_t* needed_pages, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * kvs_compact_paged_multi -- kvs_compact_paged for n_masks masks over the same K/V
 * (for instance one per top-k budget) in one set of launches, into one shared page
 * pool.  The result is that of kvs_compact_paged over n_masks L "layers" whose K/V
 * rows repeat every L layers: rows are taken mask-major, then layer, then head, so the
 * pages of mask b follow all pages of masks 0 .. b-1.
 *   masks        [n_masks][L][H_kv][T] uint8
 *   block_table  [n_masks][L][H_kv][max_pages] int32;  seq_lens [n_masks][L][H_kv] int32
 *   needed_pages [1] int32: total pages of all masks
 *   ws           scratch of kvs_compact_multi_workspace_size(dims, T, n_masks) bytes
 * Other arguments, the capacity rule and the errors as kvs_compact_paged; n_masks >= 1.
 * ------------------------------------------------------------------------------- */
size_t kvs_compact_multi_workspace_size(const kvs_dims* dims, int32_t T, int32_t n_masks);
kvs_status kvs_compact_paged_multi(const kvs_dims* dims, const kvs_bf16* k, const kvs_bf16* v,
                                   int32_t T, int32_t n_masks, const uint8_t* masks,
                                   int32_t page_size, kvs_bf16* k_pages, kvs_bf16* v_pages,
                                   int32_t capacity_pages, int32_t* block_table, int32_t max_pages,
                                   int32_t* seq_lens, int32_t* needed_pages, void* ws,
                                   size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVS_H_ */

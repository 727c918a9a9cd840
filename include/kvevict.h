/*
 * kvevict — C-ABI of the GB300 (sm_103a) KV-cache eviction library.
 *
 * Two eviction modes:
 *   LORE-KV  (project page "LORE-KV: Monte Carlo Estimation for KV-Cache Eviction"): score every
 *            cached token of every KV head by its projected deletion score under the window and
 *            lookahead queries, then keep the protected sink/window plus the top-B tokens in
 *            chunks of 4 and gather them into a dense compressed cache.
 *   H2O      (paper summary "H2O: Heavy-Hitter Oracle for Efficient Generative Inference of Large
 *            Language Models"): per-step decode eviction by accumulated attention, with half of
 *            the budget reserved for the most recent tokens.
 *
 * Conventions, for every call below:
 *   - Tensor arguments are DEVICE pointers (unless a comment says otherwise), row-major, densely
 *     packed, and owned by the caller. The library never frees them and keeps no reference after
 *     the call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Calls enqueue
 *     kernels on that stream and return without synchronising, except where stated.
 *   - Every call returns a status (KVE_OK = 0). On failure nothing is enqueued, unless the status
 *     is KVE_ECUDA (a CUDA launch failed); kve_last_error() then gives a message for the calling
 *     thread. No exception crosses this interface and nothing falls back to the CPU.
 *   - The scoring and selection calls allocate no device memory: their scratch lives in a
 *     caller-provided workspace of at least the size the matching *_workspace_size() call returns.
 *   - Kernels that wait on an on-chip barrier give up after a bounded number of polls and record
 *     the failure in a device error word; kve_check_device(stream) synchronises the stream and
 *     turns a recorded failure into KVE_ETIMEOUT.
 *
 * Notation follows the pages: K, V cached keys/values; Q_W the w window queries (last prompt
 * tokens); Q_look the M x T lookahead queries; W_O the attention output projection; logits and
 * sampled ids of the lookahead tokens; B the budget; chunk the adjacent-token group size.
 */
#ifndef KVEVICT_H
#define KVEVICT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------------- */
#define KVE_OK 0
#define KVE_EINVAL 1     /* a size, shape rule or pointer is invalid                             */
#define KVE_EDTYPE 2     /* dtype not supported by this call                                      */
#define KVE_EWORKSPACE 3 /* workspace missing or smaller than *_workspace_size()                  */
#define KVE_ENOTPD 4     /* W_O^h^T W_O^h is not positive definite (Cholesky pivot <= 0)         */
#define KVE_ECUDA 5      /* a CUDA runtime call failed                                            */
#define KVE_ETIMEOUT 6   /* a bounded on-device wait gave up (see kve_check_device)               */

/* ---- element types ------------------------------------------------------------------------ */
#define KVE_F32 0
#define KVE_BF16 1
#define KVE_F16 2

/* Problem shape of one LORE-KV pass. A "unit" is one (sequence, layer, KV head); there are
 * n_seq * n_layers * n_kv_heads units. Query head h belongs to KV head h / (n_q_heads/n_kv_heads)
 * (grouped-query attention). dtype is the element type of K, V, Q_W, Q_look and W_O. */
typedef struct {
    int n_seq, n_layers, n_q_heads, n_kv_heads, d_head, d_model, n_tokens, vocab;
    int dtype;
} KveShape;

/* Method parameters (LORE-KV page, "Hyperparameters" table; defaults w=32, M=4, T=8,
 * lambda_L=1, (beta, gamma, lambda_D) = (1, 1.3, 0) for /E or (1, 1, 0.3) for /D, eps=1e-6,
 * chunk=4). sink = number of leading tokens always kept (attention sink). budget_B = number of
 * non-protected tokens kept per KV head (a multiple of chunk). window_causal = 1: window query r
 * (0-based, at position n-w+r) attends only to tokens i <= n-w+r; lookahead queries see all n. */
typedef struct {
    int w, M, T, chunk, sink, budget_B, window_causal;
    float lambda_L, beta, gamma, lambda_D, eps;
} KveLorekvParams;

/* ---- LORE-KV -------------------------------------------------------------------------------- */

/* Per-model preparation of e = ||W_O^h x|| (LORE-KV page, Method, Eqs. 5-7): for every layer l
 * and query head h, G = W_O^h^T W_O^h and its Cholesky factor L (G = L L^T, L lower triangular),
 * so that ||W_O^h x|| = ||L^T x||. W_O^h is columns h*d .. h*d+d-1 of the o_proj weight.
 *   W_O   [n_layers][d_model][n_q_heads*d_head]   shape->dtype
 *   L_out [n_layers][n_q_heads][d_head][d_head]   fp32 (upper triangle written as 0)
 *   G_out [n_layers][n_q_heads][d_head][d_head]   fp32
 * Synchronises `stream` before returning (it must read the positive-definiteness flag).
 * Accuracy: G and L to about 1e-8 of their largest entry. bf16 weights with d_head 128 and
 * d_model a multiple of 128 form G on the tensor cores (exact bf16 products, 32-row slices
 * accumulated in fp32 and added in compensated fp32); other shapes accumulate in double. The
 * Cholesky factorisation runs in double. Allocates its double-precision scratch on `stream`.
 * Returns KVE_ENOTPD if any G is not positive definite. */
int lorekv_prepare_wo(const KveShape *shape, const void *W_O, float *L_out, float *G_out,
                      void *stream);

/* Bytes of workspace lorekv_score() needs for this shape and parameters. 0 on invalid input.
 * Size limits of every LORE-KV call (KVE_EINVAL beyond them): units = n_seq * n_layers *
 * n_kv_heads at most 65535; units * n_tokens and units * (n_q_heads / n_kv_heads) * (w + M*T)
 * below 2^31. */
size_t lorekv_workspace_size(const KveShape *shape, const KveLorekvParams *params);

/* Scores every cached token (LORE-KV page, Method, Eqs. 2-7).
 *   K, V      [n_seq][n_layers][n_kv_heads][n_tokens][d_head]   shape->dtype
 *   Q_W       [n_seq][n_layers][n_q_heads][w][d_head]           shape->dtype
 *   Q_look    [n_seq][n_layers][n_q_heads][M*T][d_head]         shape->dtype, row m*T+t
 *   L, G      from lorekv_prepare_wo                            fp32
 *   logits    [n_seq][M*T][vocab] fp32, row m*T+t is the next-token logits at lookahead token t
 *             of trajectory m; sampled [n_seq][M*T] int32 is the token drawn there.
 *   scores_out [n_seq][n_layers][n_kv_heads][n_tokens] fp32: S_i = mean_W e + lambda_L *
 *             sum_m omega_m mean_m e, with e = a/(1-a+eps) ||L_h^T (v_i - o_q)|| and the means over
 *             all g query heads of the KV head; 0 for protected tokens (i < sink or i >= n-w).
 *   omega_out [n_seq][M] fp32: omega = softmax(beta*cbar - gamma*Hbar - lambda_D*Dhat) (Eq. 10).
 * Requirements: n_tokens >= sink + w; n_q_heads % n_kv_heads == 0; dtype KVE_F32 or KVE_BF16;
 * d_head a multiple of 32 (KVE_F32) or 128 (KVE_BF16); sampled ids in [0, vocab). */
int lorekv_score(const KveShape *shape, const KveLorekvParams *params, const void *K,
                 const void *V, const void *Q_W, const void *Q_look, const float *L,
                 const float *G, const float *logits, const int32_t *sampled, float *scores_out,
                 float *omega_out, void *workspace, size_t ws_bytes, void *stream);

/* lorekv_score without a caller-provided workspace, for callers that cannot allocate device
 * memory (for example code that runs inside a memory budget owned by someone else, or where no
 * device allocator is reachable). There is no counterpart on the pages: it is the same pass as
 * lorekv_score with identical arguments and results, only the scratch memory differs.
 *   - Scratch comes from one fixed array of 64 MiB in the library's device image. Shapes whose
 *     lorekv_workspace_size() exceeds 64 MiB are rejected with KVE_EWORKSPACE (nothing launched);
 *     use lorekv_score with a workspace for them.
 *   - The call allocates nothing (no cudaMalloc/cudaFree, no library allocator).
 *   - The first call in each CUDA context (a device's primary context, a context made current
 *     through the driver API, a context created again after cudaDeviceReset) looks up the
 *     array's device address in that context (cudaGetSymbolAddress) and caches it by the
 *     driver's context id; make that first call before any stream capture.
 *   - The array is shared by every call on the device and keeps the last call's contents; nothing
 *     in it needs to start at zero (each call writes every scratch region before reading it).
 *     Calls that overlap on the GPU (different streams, or threads without ordering) race on it:
 *     serialise them.
 *   - Each GPU on which the array is loaded keeps it until the process exits. */
int lorekv_score_noalloc(const KveShape *shape, const KveLorekvParams *params, const void *K,
                         const void *V, const void *Q_W, const void *Q_look, const float *L,
                         const float *G, const float *logits, const int32_t *sampled,
                         float *scores_out, float *omega_out, void *stream);

/* Attention-output fidelity of a compressed cache (LORE-KV page, analyses, "Attention-output
 * fidelity"; reading: per query, the cosine similarity between its attention output over the
 * compressed cache and over the full cache). Typical use: lorekv_attention_stats for the same
 * held-out queries over the full K/V and over the compacted K_out/V_out (a cache of kept_capacity
 * tokens), then this call.
 *   o_full, o_comp [rows][d_head] fp32 device (row-major, 16-byte aligned for the vector path);
 *   cos_out [rows] fp32 device: o_full.o_comp / (|o_full| |o_comp|), 0 when either norm is 0;
 *   mean_out [1] fp32 device or NULL: the mean of cos_out, summed in a fixed order.
 * Returns KVE_EINVAL for null inputs, rows < 1 or d_head < 1. Asynchronous on `stream`. */
int lorekv_output_fidelity(const float *o_full, const float *o_comp, int rows, int d_head,
                           float *cos_out, float *mean_out, void *stream);

/* Attention statistics only (the first half of lorekv_score, exposed for testing): for each unit
 * and each of its g*(w+M*T) queries (query head major, then window rows, then lookahead rows):
 *   lse_out [units][g*(w+M*T)] fp32 natural-log log-sum-exp of q.k/sqrt(d) over visible tokens,
 *   o_out   [units][g*(w+M*T)][d_head] fp32 attention output o_q.
 * Uses the same workspace as lorekv_score. */
int lorekv_attention_stats(const KveShape *shape, const KveLorekvParams *params, const void *K,
                           const void *V, const void *Q_W, const void *Q_look, float *lse_out,
                           float *o_out, void *workspace, size_t ws_bytes, void *stream);

/* Kept-row capacity per unit: n_tokens if n - sink - w <= budget_B, else sink + budget_B + w. */
int lorekv_kept_capacity(const KveShape *shape, const KveLorekvParams *params);

/* Chunked top-B selection and gather-compaction (LORE-KV page, "Evict and decode", Eq. 8;
 * "Hyperparameters": adjacent-token chunks of `chunk`).
 *   scores   [units][n_tokens] fp32 from lorekv_score
 *   K, V     as in lorekv_score
 *   kept_idx [units][cap] int32, cap = lorekv_kept_capacity(): kept positions, ascending
 *   kept_len [units] int32
 *   K_out, V_out [units][cap][d_head] shape->dtype: K_out[u][j] = K[u][kept_idx[u][j]]
 * Chunk c covers tokens [sink + c*chunk, sink + (c+1)*chunk); its score is the mean of S over
 * the chunk; the budget_B/chunk chunks with the highest score are kept (equal scores: lower c).
 * (n_tokens - sink - w) and budget_B must be multiples of chunk. Needs no workspace: pass NULL, 0
 * (a non-NULL workspace is accepted and ignored). */
int lorekv_select_compact(const KveShape *shape, const KveLorekvParams *params,
                          const float *scores, const void *K, const void *V, int32_t *kept_idx,
                          int32_t *kept_len, void *K_out, void *V_out, void *workspace,
                          size_t ws_bytes, void *stream);

/* ---- H2O ------------------------------------------------------------------------------------ */

/* Opaque decode state. It owns preallocated device slots for K, V, accumulated scores and
 * positions of every (batch, layer, head) unit (H2O summary, Appendix A: preallocated memory,
 * evicted slots are overwritten in place). */
typedef struct KveH2O KveH2O;

/* Allocates the state for batch x n_layers x n_heads units of head size d_head, for sequences of
 * up to max_len tokens (prompt + decode steps), budget_frac in (0, 1]. Slot capacity per unit is
 * floor(budget_frac*max_len) + 1. dtype KVE_F16 or KVE_BF16. *out receives the handle. The state
 * also holds the prefill's scratch (two fp32 partial column sums per unit and prompt token, sized
 * for a prompt of max_len), so h2o_prefill and h2o_decode_step allocate nothing. KVE_EINVAL for
 * d_head other than 64 or 128, a slot capacity above 4096, or batch * n_layers * n_heads * max_len
 * of 2^31 or more (checked before anything is allocated). */
int h2o_state_create(KveH2O **out, int batch, int n_layers, int n_heads, int d_head, int max_len,
                     float budget_frac, int dtype);

/* Prefill (H2O summary, Section 4.1; prompt handled as one block): accumulated scores of the
 * prompt tokens are the causal-attention column sums acc_j = sum_{i>=j} softmax_i(q_i.K_{<=i}/
 * sqrt d)_j; then the cache is compressed to k_t = floor(budget_frac*t) tokens (t = prompt_len):
 * the r_t = floor(k_t/2) most recent are kept, and among the rest the highest accumulated scores
 * (equal scores: the newer token stays).
 *   K, V, Q [batch][n_layers][n_heads][prompt_len][d_head] state dtype. */
int h2o_prefill(KveH2O *st, const void *K, const void *V, const void *Q, int prompt_len,
                void *stream);

/* One decode step for every unit (H2O summary, Section 4.1, Algorithm 1 with linear h; Section
 * 2.1 and Definition 2.2 for attention over the retained set; Definition 2.1: at most one
 * eviction per step): append (k_new, v_new) into a free slot; attend with q over the retained
 * tokens including the new one; add the softmax row to the accumulated scores; with t the new
 * length, k_t = floor(budget_frac*t) and r_t = floor(k_t/2), while more than k_t tokens are held
 * evict the lowest accumulated score among positions < t - r_t (equal scores: the oldest).
 *   q, k_new, v_new, attn_out [batch][n_layers][n_heads][d_head] state dtype;
 *   attn_out = softmax(q.K/sqrt d) V over the retained tokens. */
int h2o_decode_step(KveH2O *st, const void *q, const void *k_new, const void *v_new,
                    void *attn_out, void *stream);

/* Copies the state out (device pointers, any may be NULL):
 *   K, V [units][cap][d_head] state dtype; pos [units][cap] int32 (-1 for an empty slot);
 *   acc [units][cap] fp32; count [units] int32 (retained tokens). */
int h2o_export(const KveH2O *st, void *K, void *V, int32_t *pos, float *acc, int32_t *count,
               void *stream);

/* Slot capacity per unit and the current sequence length t (tokens seen so far). */
int h2o_capacity(const KveH2O *st);
int h2o_length(const KveH2O *st);

void h2o_state_destroy(KveH2O *st);

/* ---- counter-causal surprise refresh --------------------------------------------------------- */

/* Problem shape of one counter-causal refresh (review of "Back from the Future: KV Cache Management
 * by Counter-Causal Surprise", Section 3.3: the fast variant that runs only the last layer).
 * n_seq independent sequences of n_tokens cached tokens; query head h reads KV head
 * h / (n_q_heads/n_kv_heads); sink = leading system-prompt slots that are never scored or evicted
 * (design choice 4); keep_J = tokens kept per sequence (Algorithm 3, J). dtype is the element type
 * of K, V, Q_fresh, H_last, W_O and W_U: KVE_F32 or KVE_BF16. d_head is 32, 64 or 128;
 * 0 <= sink <= n_tokens; 1 <= keep_J <= n_tokens; n_seq and n_q_heads at most 65535, d_model at
 * most 2^22, n_seq * n_q_heads * n_tokens below 2^31 (KVE_EINVAL otherwise). */
typedef struct {
    int n_seq, n_q_heads, n_kv_heads, d_head, d_model, n_tokens, vocab, dtype, sink, keep_J;
} KveCcShape;

/* Bytes of workspace cc_surprise() needs: the heads' attention outputs (fp32, n_seq * n_tokens *
 * n_q_heads * d_head floats) and per-column-tile partial logits. 0 on invalid input. */
size_t cc_workspace_size(const KveCcShape *shape);

/* Counter-causal surprise of every cached token (same review, Section 3.2 steps 1-5, Eq. 1).
 *   K, V     [n_seq][n_kv_heads][n_tokens][d_head]  the last layer's cached keys and values
 *   Q_fresh  [n_seq][n_q_heads][n_tokens][d_head]   fresh queries at the tokens' own positions
 *   H_last   [n_seq][n_tokens][d_model]             the last layer's stored input activations
 *   W_O      [d_model][n_q_heads*d_head]            the last layer's output projection (o_proj)
 *   W_U      [vocab][d_model]                       the unembedding
 *   tokens   [n_seq][n_tokens] int32                the cached token ids x_i, in [0, vocab)
 *   surprise_out [n_seq][n_tokens] fp32: -logit_i with logit_i = W_U[x_i] . (h_i + W_O o_i),
 *            o_i the heads' outputs concatenated, o_i^h = sum_{j>i} softmax_j(q_i^h.k_j/sqrt d) v_j
 *            (strictly later tokens only; the last token's o is 0); +inf for the sink slots and
 *            the last token.
 * Token ids are checked on the device: an id outside [0, vocab) is read as 0 and recorded in the
 * device error word, which kve_check_device(stream) reports as KVE_EINVAL. */
int cc_surprise(const KveCcShape *shape, const void *K, const void *V, const void *Q_fresh,
                const void *H_last, const void *W_O, const void *W_U, const int32_t *tokens,
                float *surprise_out, void *workspace, size_t ws_bytes, void *stream);

/* Memory refresh (same review, Algorithm 3): per sequence keep the keep_J tokens of highest
 * surprise (equal surprise: the lower position), in ascending position order, and gather them.
 *   surprise [n_seq][n_tokens] fp32 (from cc_surprise); K, V, tokens as in cc_surprise
 *   kept_idx [n_seq][keep_J] int32 kept positions, ascending
 *   K_out, V_out [n_seq][n_kv_heads][keep_J][d_head] shape->dtype: K_out[s][h][j] =
 *            K[s][h][kept_idx[s][j]]; tokens_out [n_seq][keep_J] int32.
 * No workspace. Outputs must not overlap the inputs. */
int cc_select_compact(const KveCcShape *shape, const float *surprise, const void *K,
                      const void *V, const int32_t *tokens, int32_t *kept_idx, void *K_out,
                      void *V_out, int32_t *tokens_out, void *stream);

/* Refresh-cycle cache (same review, Algorithms 1 and 3; Section 5, design choice 3: refresh every
 * h tokens). Per sequence it holds the memory M = (K', V') of at most keep_J tokens followed by the
 * recent chunk of up to h = n_tokens - keep_J tokens, with each token's fresh queries, stored
 * last-layer input activation, id and original position (a token's fresh query depends only on
 * its own activation and position, so it is stored with it). A refresh scores the mem + recent
 * candidates with cc_surprise's arithmetic and keeps the keep_J most surprising (cc_select_compact's
 * rule), in ascending position order; with keep_J or fewer candidates it keeps them all and
 * launches nothing. The cache owns its device memory: two buffers of n_tokens rows per sequence
 * and head (a refresh gathers into the other buffer and swaps) plus the scoring workspace.
 * Requirements: those of cc_surprise, keep_J < n_tokens, keep_J >= sink + 1, d_model rows a
 * multiple of 16 bytes. */
typedef struct KveCcCache KveCcCache;

/* Allocates a cache for shape (n_tokens = keep_J + h, the candidates of a full refresh).
 * Synchronises the device once. *out receives the handle. */
int cc_cache_create(KveCcCache **out, const KveCcShape *shape);

/* Appends `count` tokens to the recent chunk (Algorithm 2, lines 3-5), 1 <= count <= h minus the
 * tokens already in the chunk. Device pointers:
 *   K_new, V_new [n_seq][n_kv_heads][count][d_head]; Q_new [n_seq][n_q_heads][count][d_head];
 *   H_new [n_seq][count][d_model] (all shape->dtype); tokens_new [n_seq][count] int32.
 * Their original positions are the number of tokens appended before them. */
int cc_cache_append(KveCcCache *c, const void *K_new, const void *V_new, const void *Q_new,
                    const void *H_new, const int32_t *tokens_new, int count, void *stream);

/* Memory refresh (Algorithm 3) over the current candidates, then the chunk is empty. W_O
 * [d_model][n_q_heads*d_head] and W_U [vocab][d_model] as in cc_surprise. Token ids outside
 * [0, vocab) are reported by kve_check_device. */
int cc_cache_refresh(KveCcCache *c, const void *W_O, const void *W_U, void *stream);

/* One step of Algorithm 1's loop without the model: cc_cache_append, then cc_cache_refresh if the
 * chunk now holds h tokens. *refreshed (host, may be NULL) tells whether the refresh ran. */
int cc_cache_step(KveCcCache *c, const void *K_new, const void *V_new, const void *Q_new,
                  const void *H_new, const int32_t *tokens_new, int count, const void *W_O,
                  const void *W_U, int *refreshed, void *stream);

/* Copies the held tokens out, memory then chunk (len = cc_cache_length rows, ascending original
 * positions): K, V [n_seq][n_kv_heads][len][d_head]; Q [n_seq][n_q_heads][len][d_head];
 * H [n_seq][len][d_model]; tokens, pos [n_seq][len] int32. Any pointer may be NULL. */
int cc_cache_export(const KveCcCache *c, void *K, void *V, void *Q, void *H, int32_t *tokens,
                    int32_t *pos, void *stream);

/* Tokens held (memory + chunk) and tokens appended so far. */
int cc_cache_length(const KveCcCache *c);
int cc_cache_seen(const KveCcCache *c);

void cc_cache_destroy(KveCcCache *c);

/* ---- diagnostics ---------------------------------------------------------------------------- */

/* Message of the last failing call on this thread ("" if none). Valid until the next call. */
const char *kve_last_error(void);

/* Synchronises `stream`, then reads and clears the device error word that bounded on-device
 * waits and device-side index checks set. Returns KVE_OK, KVE_ETIMEOUT (a wait gave up),
 * KVE_EINVAL (cc_surprise met a token id outside [0, vocab)) or KVE_ECUDA. */
int kve_check_device(void *stream);

/* Self-test of the bounded on-device waits: launches one CTA whose thread waits, through the same
 * routine the tensor-core kernels use, on an on-chip barrier that nothing signals, with a limit of
 * limit_ms milliseconds (1..10000). The wait gives up, records the timeout in the device error word
 * and the kernel returns normally; kve_check_device(stream) then reports KVE_ETIMEOUT and clears
 * the word. Asynchronous on `stream`. */
int kve_selftest_wait_timeout(int limit_ms, void *stream);

/* Host-side fault injection for tests: the next `count` calls of the API (excluding the
 * diagnostics) fail with `status` before touching the GPU. count = 0 clears it. */
int kve_inject_failure(int status, int count);

/* Kernel timing for measurement: while enabled, every launch group of the library (one
 * pipeline stage, e.g. "scores" or "select_compact") is bracketed by CUDA events recorded on the
 * stream it runs on. Disabled by default; enabling costs two event records per stage. */
int kve_profile_enable(int on);

/* Synchronises on the recorded events and writes one line per stage into buf (host memory,
 * NUL-terminated, truncated to len): "<stage> <launch groups> <kernels> <total ms>\n". Clears the
 * record. Returns the number of stages, or -KVE_EINVAL if buf is NULL. */
int kve_profile_report(char *buf, size_t len);

/* Library version (major*10000 + minor*100 + patch). */
int kve_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVEVICT_H */

// Internal declarations shared by the library's translation units (not part of the C-ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>
#include <vector>

#include "../../include/kvevict.h"

namespace kve {

// ---- element conversion ------------------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

inline size_t dtype_size(int dt) { return dt == KVE_F32 ? 4 : 2; }

// ---- device error word -------------------------------------------------------------------------
// Bit 0: a bounded wait on an mbarrier gave up. The host reads and clears it in kve_check_device.
// Bit 1: a token id outside [0, vocab) reached the counter-causal logit kernel.
enum : unsigned { KVE_DEVERR_TIMEOUT = 1u, KVE_DEVERR_BADINDEX = 2u };
unsigned *device_error_word();  // device address of the word in the current context

// Device address of a __device__ variable (its host-side stand-in `symbol`) in the calling
// thread's current context, looked up with cudaGetSymbolAddress once per context and cached by
// the driver's context id. nullptr if the lookup fails.
struct SymbolCache {
    std::mutex mu;
    std::vector<std::pair<unsigned long long, void *>> entries;
};
void *context_symbol_address(const void *symbol, SymbolCache &cache);

// Records a message for kve_last_error() on the calling thread and returns `code`.
int report_error(int code, const char *fmt, ...);

// ---- warp helpers ------------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---- LORE-KV launch description ----------------------------------------------------------------
struct LorekvDims {
    int S, L, Hq, Hkv, g, d, d_model, n, vocab, dtype;
    int w, M, T, MT, nq;       // nq = w + M*T queries per query head
    int Qu;                    // g * nq queries per unit
    int units;                 // S * L * Hkv
    int chunk, sink, B, window_causal;
    float lambda_L, beta, gamma, lambda_D, eps;
    int nsplit;                // token splits of the attention-statistics pass
    int split_len;             // tokens per split (multiple of 128)
    int at_qt;                 // 128-query tiles per attention CTA on the tensor cores (1 or 2)
    int rel_splits;            // CTAs per logits row in the reliability pass
};

// Workspace carve-up of lorekv_score (byte offsets, 256-aligned).
struct LorekvWorkspace {
    size_t part_ml, part_o;    // split partials: [units][nsplit][Qu] float2 (m2, l), [..][d] f32
    size_t lse2, o;            // combined: [units][Qu] f32 (log2 domain), [units][Qu][d] f32
    size_t u32, cq, wq;        // u = G o [units][Qu][d] f32; c = o^T G o, weight [units][Qu]
    size_t u16, lt16;          // bf16 operands: U [units][Qu][d]; L^T packed [L][Hq][d][d]
    size_t q16;                // bf16 queries packed [units][Qu][d]
    size_t part_s;             // per-query-head partial scores [units][g][n] f32
    size_t qconst;             // per-query {-lse2, c, weight, 0} [units][Qu] float4
    size_t rel_part;           // reliability partials [S][MT][rel_splits] float4
    size_t cosm;               // cosine sums [S][L*Hq][M][M] f32
    // peaked pairs (a > kPeakTau): per-split maximum logit over non-protected tokens [units]
    // [nsplit][Qu] (log2 domain), the largest non-protected probability a_max [units][Qu], and
    // per query the count, tokens and weighted exact scores of the pairs the scoring kernels
    // left out [units][Qu] / [units][Qu][kPeakSlots]
    size_t part_mx, amax, pk_cnt, pk_tok, pk_e;
    size_t total;
};

// Peaked pairs. Where a_{q,i} is close to 1, o_q is close to v_i and the expanded quadratic form
// ||L^T v||^2 - 2 v.(G o) + o^T G o cancels, 1 - a cancels, and the bf16 rounding of the
// attention weights in o no longer averages out against the small ||L^T (v_i - o_q)||. Pairs
// with a > kPeakTau are therefore left out by the scoring kernels, recorded (at most
// kPeakSlots per query: more than three tokens cannot exceed 1/4) and evaluated exactly by
// peak_fix_kernel in difference form. The tensor-core scoring kernel only checks pairs in CTAs
// whose queries have a_max > kPeakFlag (a margin below kPeakTau), so unpeaked workloads pay
// nothing for it.
constexpr float kPeakTau = 0.25f;
constexpr float kPeakFlag = 0.125f;
constexpr int kPeakSlots = 4;

bool lorekv_dims(const KveShape *sh, const KveLorekvParams *p, LorekvDims *D, const char **why);
bool tc_supported(const LorekvDims &D);  // tensor-core kernels cover this shape
void tc_plan(LorekvDims *D);             // token splits of the tensor-core attention pass
LorekvWorkspace lorekv_ws_layout(const LorekvDims &D);

// ---- launchers (each returns cudaGetLastError() of its launches) -------------------------------
cudaError_t launch_reliability(const LorekvDims &D, const void *Q_look, const float *logits,
                               const int32_t *sampled, float *omega_out, void *ws,
                               const LorekvWorkspace &W, cudaStream_t st);
cudaError_t launch_prepare_wo(int L, int Hq, int d, int d_model, int dtype, const void *W_O,
                              float *L_out, float *G_out, int *notpd_flag, cudaStream_t st);
cudaError_t launch_attention_simt(const LorekvDims &D, const void *K, const void *V,
                                  const void *QW, const void *QL, void *ws,
                                  const LorekvWorkspace &W, cudaStream_t st);
cudaError_t launch_combine(const LorekvDims &D, void *ws, const LorekvWorkspace &W,
                           float *lse_out, float *o_out, cudaStream_t st);
cudaError_t launch_prep_u(const LorekvDims &D, const float *G, const float *omega, void *ws,
                          const LorekvWorkspace &W, cudaStream_t st);
cudaError_t launch_scores_simt(const LorekvDims &D, const void *K, const void *V,
                               const void *QW, const void *QL, const float *Lf, void *ws,
                               const LorekvWorkspace &W, float *scores, cudaStream_t st);
// exact scores of the recorded peaked pairs, then added into scores [units][n] in a fixed order
cudaError_t launch_peak_fix(const LorekvDims &D, const void *K, const void *V, const void *QW,
                            const void *QL, const float *Lf, void *ws, const LorekvWorkspace &W,
                            float *scores, cudaStream_t st);
cudaError_t launch_select_compact(const LorekvDims &D, const float *scores, const void *K,
                                  const void *V, int32_t *kept_idx, int32_t *kept_len,
                                  void *K_out, void *V_out, int cap, cudaStream_t st);

// H2O
struct H2OState {
    int batch, L, H, d, max_len, cap, dtype;
    float frac;
    int units;
    int t;             // tokens seen so far
    int prefilled;
    void *K, *V;       // [units][cap][d]
    float *acc;        // [units][cap]
    int32_t *pos;      // [units][cap], -1 = empty
    int32_t *nslots;   // [units] slots in use (including a hole)
    int32_t *hole;     // [units] free slot left by the last eviction, -1 if none
    float *prefill_part;  // [units][kColsumTcParts][max_len] partial prefill scores (scratch)
};
cudaError_t launch_h2o_prefill(H2OState &s, const void *K, const void *V, const void *Q, int P,
                               cudaStream_t st);
bool h2o_prefill_fits(int d, int P, int dtype);
size_t h2o_prefill_smem(int d, int P, int dtype);  // CUDA-core column-sum kernel
cudaError_t launch_output_fidelity(const float *o_full, const float *o_comp, int rows, int d,
                                   float *cos_out, float *mean_out, cudaStream_t st);
// tensor-core prefill column sums (h2o_tc.cu): writes kColsumTcParts partial sums per token,
// acc_out [units][kColsumTcParts][P]
constexpr int kColsumTcParts = 2;
bool h2o_colsum_tc_supported(int d, int P, int dtype);
cudaError_t launch_h2o_colsum_tc(int units, int P, const void *K, const void *Q, int dtype,
                                 float *acc_out, cudaStream_t st);
cudaError_t launch_h2o_step(H2OState &s, const void *q, const void *k, const void *v, void *out,
                            cudaStream_t st);
cudaError_t launch_h2o_export(const H2OState &s, void *K, void *V, int32_t *pos, float *acc,
                              int32_t *count, cudaStream_t st);

// Counter-causal surprise refresh, fast single-layer variant (counter_causal.cu)
// n tokens scored per sequence; ld = row stride of the token dimension (>= n) of K, V, Q, H,
// the token ids and the surprise (n for the stateless calls, the buffer capacity for the
// refresh-cycle cache)
struct CcDims {
    int batch, hq, hkv, d, dm, n, vocab, dtype, sink, J, ld;
};
size_t cc_o_bytes(const CcDims &D);
size_t cc_workspace_bytes(const CcDims &D);
// attention outputs O [batch][n][hq*d] fp32 at the start of the workspace
cudaError_t launch_cc_attention(const CcDims &D, const void *K, const void *V, const void *Q,
                                void *ws, unsigned *err, cudaStream_t st);
// tensor-core attention (cc_tc.cu): bf16, d_head 128, at least 128 K/V rows in all; writes O as
// fp32 into O, or as bf16 into Ob when Ob is not null
bool cc_attention_tc_supported(const CcDims &D);
cudaError_t launch_cc_attention_tc(const CcDims &D, const void *K, const void *V, const void *Q,
                                   float *O, __nv_bfloat16 *Ob, unsigned *err, cudaStream_t st);
// tensor-core projection + logit (cc_tc.cu): also needs d_model % 8 == 0; partial logits
// [batch][ceil(d_model/256) * ksplit * 2][n], ksplit from cc_logits_tc_split (<= kCcMaxKSplit)
constexpr int kCcMaxKSplit = 4;
bool cc_logits_tc_supported(const CcDims &D);
int cc_logits_tc_split(const CcDims &D);
cudaError_t launch_cc_logits_tc(const CcDims &D, const __nv_bfloat16 *Ob, const void *H,
                                const void *W_O, const void *W_U, const int32_t *X, float *part,
                                int ksplit, unsigned *err, cudaStream_t st);
// surprise from O, h, W_O, W_U[x] (partial logits after O in the workspace)
cudaError_t launch_cc_logits(const CcDims &D, const void *H, const void *W_O, const void *W_U,
                             const int32_t *X, float *surprise, void *ws, unsigned *err,
                             cudaStream_t st);
cudaError_t launch_cc_select(const CcDims &D, const float *surprise, const void *K, const void *V,
                             const int32_t *X, int32_t *kept, void *K_out, void *V_out,
                             int32_t *X_out, cudaStream_t st);
// selection only: kept [batch][J]; X_out and pos_out (optional) [batch][ldo]
cudaError_t launch_cc_select_idx(const CcDims &D, const float *surprise, const int32_t *X,
                                 const int32_t *pos, int32_t *kept, int32_t *X_out,
                                 int32_t *pos_out, int ldo, cudaStream_t st);
// gather of kept rows from up to four tensors [batch][heads][ld][row bytes], one launch
struct CcGatherSet {
    const uint4 *src[4];
    uint4 *dst[4];
    int heads[4], vpr[4];
    long start[5];  // word offsets of each tensor in the launch's index space
    int count;
};
void cc_gather_add(CcGatherSet *G, const void *src, void *dst, int batch, int heads,
                   size_t row_bytes, int J);
cudaError_t launch_cc_gather(const CcGatherSet &G, const int32_t *kept, int J, int ld_in,
                             int ld_out, cudaStream_t st);
// append: count new rows of each table tensor (sources [batch][heads][count][row], entered with
// cc_gather_add(..., J = count)) at row `at` of the [batch][heads][ld][row] destinations, plus
// ids x_new [batch][count] and positions first + r, in one launch
cudaError_t launch_cc_append(const CcGatherSet &G, int count, int at, int ld,
                             const int32_t *x_new, int32_t *X, int32_t *pos, int batch, int first,
                             cudaStream_t st);

}  // namespace kve

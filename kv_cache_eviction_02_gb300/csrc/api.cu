// C-ABI entry points of libkvevict (declared in include/kvevict.h): argument validation,
// workspace layout, error reporting and kernel dispatch. No computation happens here.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "kve_internal.cuh"

namespace kve {

cudaError_t launch_prep_u(const LorekvDims &D, const float *G, const float *omega, void *ws,
                          const LorekvWorkspace &W, cudaStream_t st, const void *QW,
                          const void *QL, bool want_bf16);
cudaError_t launch_scores_tc(const LorekvDims &D, const void *K, const void *V, const float *Lf,
                             void *ws, const LorekvWorkspace &W, float *scores,
                             unsigned *err_word, cudaStream_t st);
cudaError_t launch_attention_tc(const LorekvDims &D, const void *K, const void *V, void *ws,
                                const LorekvWorkspace &W, unsigned *err_word, cudaStream_t st);
cudaError_t launch_pack_queries(const LorekvDims &D, const void *QW, const void *QL, void *ws,
                                const LorekvWorkspace &W, cudaStream_t st);
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, unsigned *err, cudaStream_t st);

namespace {

thread_local std::string g_err;
std::atomic<int> g_inject_status{0};
std::atomic<int> g_inject_count{0};

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *where) {
    return fail(KVE_ECUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Returns a non-zero status if a test asked the next call to fail.
int injected() {
    int c = g_inject_count.load();
    while (c > 0) {
        if (g_inject_count.compare_exchange_weak(c, c - 1))
            return fail(g_inject_status.load(), "injected failure (test hook)");
    }
    return KVE_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---- stage profiler (kve_profile_enable / kve_profile_report) ----------------------------------
struct ProfRec {
    const char *name;
    int kernels;
    cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::atomic<int> g_prof_on{0};
std::vector<ProfRec> g_prof;

// Brackets one launch group with events on `st` while profiling is enabled.
struct ProfScope {
    ProfRec rec{nullptr, 0, nullptr, nullptr};
    cudaStream_t st;
    bool on;
    ProfScope(const char *name, int kernels, cudaStream_t s) : st(s), on(g_prof_on.load() != 0) {
        if (!on) return;
        rec.name = name;
        rec.kernels = kernels;
        if (cudaEventCreate(&rec.a) != cudaSuccess || cudaEventCreate(&rec.b) != cudaSuccess) {
            on = false;
            return;
        }
        cudaEventRecord(rec.a, st);
    }
    ~ProfScope() {
        if (!on) return;
        cudaEventRecord(rec.b, st);
        std::lock_guard<std::mutex> lk(g_prof_mu);
        g_prof.push_back(rec);
    }
};

}  // namespace

int report_error(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

// ---- device addresses of the library's __device__ variables ------------------------------------
namespace {
using PFN_ctxGetCurrent = int (*)(void **);
using PFN_ctxGetId = int (*)(void *, unsigned long long *);

// The driver's unique id of the calling thread's current context (ids are never reused, so a
// context created after cudaDeviceReset, or a non-primary context, has an id of its own).
bool current_context_id(unsigned long long *id) {
    static PFN_ctxGetCurrent get_cur = nullptr;
    static PFN_ctxGetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_ctxGetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_ctxGetId>(p);
    });
    if (!get_cur || !get_id) return false;
    void *ctx = nullptr;
    if (get_cur(&ctx) != 0 || !ctx) return false;
    return get_id(ctx, id) == 0;
}
}  // namespace

void *context_symbol_address(const void *symbol, SymbolCache &cache) {
    unsigned long long id = 0;
    std::lock_guard<std::mutex> lk(cache.mu);
    const bool have_id = current_context_id(&id);
    if (have_id)
        for (auto &e : cache.entries)
            if (e.first == id) return e.second;
    void *p = nullptr;  // also makes the runtime's context current if none was yet
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return nullptr;
    if (have_id || current_context_id(&id)) cache.entries.emplace_back(id, p);
    return p;
}

// ---- device error word ---------------------------------------------------------------------------
__device__ unsigned g_kve_error_word;

unsigned *device_error_word() {
    static SymbolCache cache;
    return static_cast<unsigned *>(
        context_symbol_address(reinterpret_cast<const void *>(&g_kve_error_word), cache));
}

// ---- LORE-KV shape rules -------------------------------------------------------------------------
bool lorekv_dims(const KveShape *sh, const KveLorekvParams *p, LorekvDims *D, const char **why) {
    *why = nullptr;
    if (!sh || !p) return (*why = "null shape or params"), false;
    if (sh->n_seq < 1 || sh->n_layers < 1 || sh->n_q_heads < 1 || sh->n_kv_heads < 1 ||
        sh->d_head < 1 || sh->d_model < 1 || sh->n_tokens < 1 || sh->vocab < 1)
        return (*why = "shape sizes must be positive"), false;
    if (sh->n_q_heads % sh->n_kv_heads != 0)
        return (*why = "n_q_heads must be a multiple of n_kv_heads"), false;
    if (sh->d_head != 32 && sh->d_head != 64 && sh->d_head != 128)
        return (*why = "d_head must be 32, 64 or 128"), false;
    if (p->w < 1 || p->M < 1 || p->T < 1 || p->M > 32 || p->M * p->T > 64)
        return (*why = "need w >= 1, 1 <= M <= 32, T >= 1, M*T <= 64"), false;
    if (p->chunk < 1 || p->sink < 0 || p->budget_B < 0 || p->budget_B % p->chunk != 0)
        return (*why = "need chunk >= 1, sink >= 0, budget_B >= 0 and a multiple of chunk"), false;
    if (sh->n_tokens < p->sink + p->w) return (*why = "n_tokens < sink + w"), false;
    if ((sh->n_tokens - p->sink - p->w) % p->chunk != 0)
        return (*why = "(n_tokens - sink - w) must be a multiple of chunk"), false;
    if (!(p->eps >= 0.f) || !std::isfinite(p->eps) || !std::isfinite(p->lambda_L) ||
        !std::isfinite(p->beta) || !std::isfinite(p->gamma) || !std::isfinite(p->lambda_D))
        return (*why = "parameters must be finite, eps >= 0"), false;
    // the kernels' grids carry the units in gridDim.y (at most 65535), and K/V rows (unit, token)
    // and query rows (unit, query) are addressed with 32-bit indices and TMA coordinates
    const long long units = (long long)sh->n_seq * sh->n_layers * sh->n_kv_heads;
    const long long qu = (long long)(sh->n_q_heads / sh->n_kv_heads) * (p->w + p->M * p->T);
    if (units > 65535) return (*why = "n_seq * n_layers * n_kv_heads must be at most 65535"), false;
    if (units * sh->n_tokens >= (1LL << 31) || units * qu >= (1LL << 31))
        return (*why = "units * n_tokens and units * queries per unit must be below 2^31"), false;
    D->S = sh->n_seq;
    D->L = sh->n_layers;
    D->Hq = sh->n_q_heads;
    D->Hkv = sh->n_kv_heads;
    D->g = D->Hq / D->Hkv;
    D->d = sh->d_head;
    D->d_model = sh->d_model;
    D->n = sh->n_tokens;
    D->vocab = sh->vocab;
    D->dtype = sh->dtype;
    D->w = p->w;
    D->M = p->M;
    D->T = p->T;
    D->MT = p->M * p->T;
    D->nq = D->w + D->MT;
    D->Qu = D->g * D->nq;
    D->units = D->S * D->L * D->Hkv;
    D->chunk = p->chunk;
    D->sink = p->sink;
    D->B = p->budget_B;
    D->window_causal = p->window_causal ? 1 : 0;
    D->lambda_L = p->lambda_L;
    D->beta = p->beta;
    D->gamma = p->gamma;
    D->lambda_D = p->lambda_D;
    D->eps = p->eps;
    // shared-memory budget of the CUDA-core scoring kernel
    const size_t sc_smem = sizeof(float) * (2 * 32 * (D->d + 1) + 2 * (size_t)D->nq * D->d +
                                            (size_t)D->d * D->d + 3 * D->nq + 256);
    const size_t pu_smem = sizeof(float) * ((size_t)D->d * D->d + (size_t)((D->nq + 3) & ~3) * D->d);
    if (sc_smem > 227 * 1024 || pu_smem > 227 * 1024)
        return (*why = "w + M*T too large for d_head"), false;
    // token splits of the statistics pass: enough CTAs to fill the GPU several times
    const long qblocks = (D->Qu + 31) / 32;
    long want = (2432 + qblocks * D->units - 1) / (qblocks * D->units);
    const long max_split = (D->n + 127) / 128;
    if (want < 1) want = 1;
    if (want > max_split) want = max_split;
    long split_len = (D->n + want - 1) / want;
    split_len = (split_len + 127) / 128 * 128;
    D->split_len = (int)split_len;
    D->nsplit = (int)((D->n + split_len - 1) / split_len);
    D->at_qt = 2;
    if (tc_supported(*D)) tc_plan(D);
    long rs = (304 + (long)D->S * D->MT - 1) / ((long)D->S * D->MT);
    const long rs_max = (D->vocab + 2047) / 2048;
    if (rs > rs_max) rs = rs_max;
    if (rs < 1) rs = 1;
    D->rel_splits = (int)rs;
    return true;
}

LorekvWorkspace lorekv_ws_layout(const LorekvDims &D) {
    LorekvWorkspace W{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    const size_t uq = (size_t)D.units * D.Qu;
    W.part_ml = take(sizeof(float2) * uq * D.nsplit);
    W.part_o = take(sizeof(float) * uq * D.nsplit * D.d);
    W.lse2 = take(sizeof(float) * uq);
    W.o = take(sizeof(float) * uq * D.d);
    W.u32 = take(sizeof(float) * uq * D.d);
    W.cq = take(sizeof(float) * uq);
    W.wq = take(sizeof(float) * uq);
    const bool bf = D.dtype == KVE_BF16;
    W.u16 = take(bf ? 2 * uq * D.d : 0);
    W.q16 = take(bf ? 2 * uq * D.d : 0);
    // L^T packed per pair of query heads (256 rows of d each; an odd group size pads one head)
    W.lt16 = take(bf ? 2 * (size_t)D.L * D.Hkv * ((D.g + 1) / 2) * 256 * D.d : 0);
    W.part_s = take(bf ? sizeof(float) * (size_t)D.units * D.g * D.n : 0);
    W.qconst = take(bf ? sizeof(float4) * uq : 0);
    W.rel_part = take(sizeof(float4) * (size_t)D.S * D.MT * D.rel_splits);
    W.cosm = take(sizeof(float) * (size_t)D.S * D.L * D.Hq * D.M * D.M);
    W.part_mx = take(sizeof(float) * uq * D.nsplit);
    W.amax = take(sizeof(float) * uq);
    W.pk_cnt = take(sizeof(int) * uq);
    W.pk_tok = take(sizeof(int) * uq * kPeakSlots);
    W.pk_e = take(sizeof(float) * uq * kPeakSlots);
    W.total = off;
    return W;
}

}  // namespace kve

using namespace kve;

struct KveH2O {
    H2OState s;
};

// Refresh-cycle cache of the counter-causal method: two buffers of J + h rows per sequence (and
// head) for K, V, fresh queries, stored activations, token ids and original positions. Rows
// [0, mem) hold the memory M, rows [mem, mem + recent) the recent chunk; a refresh gathers the
// kept rows into the other buffer and swaps, so no row is overwritten while it is still read.
struct KveCcCache {
    CcDims D;  // n = J + h, ld = J + h
    int h;     // chunk size
    int mem = 0, recent = 0, seen = 0, cur = 0;
    struct Buf {
        void *K = nullptr, *V = nullptr, *Q = nullptr, *H = nullptr;
        int32_t *X = nullptr, *pos = nullptr;
    } buf[2];
    void *ws = nullptr;
    size_t ws_bytes = 0;
    float *surprise = nullptr;
    int32_t *kept = nullptr;
};

extern "C" {

const char *kve_last_error(void) { return g_err.c_str(); }

int kve_version(void) { return 10000; }

int kve_inject_failure(int status, int count) {
    g_inject_status.store(status);
    g_inject_count.store(count < 0 ? 0 : count);
    return KVE_OK;
}

int kve_profile_enable(int on) {
    g_prof_on.store(on ? 1 : 0);
    return KVE_OK;
}

int kve_profile_report(char *buf, size_t len) {
    if (!buf) return -KVE_EINVAL;
    std::vector<ProfRec> recs;
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        recs.swap(g_prof);
    }
    struct Agg {
        std::string name;
        int groups = 0, kernels = 0;
        double ms = 0.0;
    };
    std::vector<Agg> agg;
    for (auto &r : recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) == cudaSuccess) cudaEventElapsedTime(&ms, r.a, r.b);
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
        Agg *a = nullptr;
        for (auto &x : agg)
            if (x.name == r.name) a = &x;
        if (!a) {
            agg.push_back(Agg{r.name});
            a = &agg.back();
        }
        a->groups += 1;
        a->kernels += r.kernels;
        a->ms += ms;
    }
    std::string out;
    char line[256];
    for (auto &a : agg) {
        snprintf(line, sizeof(line), "%s %d %d %.6f\n", a.name.c_str(), a.groups, a.kernels, a.ms);
        out += line;
    }
    if (len > 0) {
        const size_t n = out.size() < len - 1 ? out.size() : len - 1;
        memcpy(buf, out.data(), n);
        buf[n] = 0;
    }
    return (int)agg.size();
}

int kve_check_device(void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "kve_check_device: stream synchronize");
    unsigned word = 0;
    e = cudaMemcpyFromSymbol(&word, g_kve_error_word, sizeof(word));
    if (e != cudaSuccess) return cuda_fail(e, "kve_check_device: read error word");
    if (word) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_kve_error_word, &zero, sizeof(zero));
        if (word & KVE_DEVERR_TIMEOUT)
            return fail(KVE_ETIMEOUT, "a bounded on-device wait gave up (error word 0x%x)", word);
        if (word & KVE_DEVERR_BADINDEX)
            return fail(KVE_EINVAL, "a token id outside [0, vocab) reached cc_surprise (error word 0x%x)",
                        word);
        return fail(KVE_ECUDA, "device error word 0x%x", word);
    }
    return KVE_OK;
}

int kve_selftest_wait_timeout(int limit_ms, void *stream) {
    if (int s = injected()) return s;
    if (limit_ms < 1 || limit_ms > 10000)
        return fail(KVE_EINVAL, "kve_selftest_wait_timeout: limit_ms must be in [1, 10000]");
    unsigned *err = device_error_word();
    if (!err) return fail(KVE_ECUDA, "kve_selftest_wait_timeout: no device error word");
    cudaError_t e = launch_wait_timeout_selftest((uint64_t)limit_ms * 1000000ull, err,
                                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kve_selftest_wait_timeout: launch");
    return KVE_OK;
}

int lorekv_prepare_wo(const KveShape *shape, const void *W_O, float *L_out, float *G_out,
                      void *stream) {
    if (int s = injected()) return s;
    if (!shape || !W_O || !L_out || !G_out) return fail(KVE_EINVAL, "lorekv_prepare_wo: null argument");
    if (shape->dtype != KVE_F32 && shape->dtype != KVE_BF16)
        return fail(KVE_EDTYPE, "lorekv_prepare_wo: dtype must be KVE_F32 or KVE_BF16");
    const int d = shape->d_head;
    if (d != 32 && d != 64 && d != 128) return fail(KVE_EINVAL, "lorekv_prepare_wo: d_head must be 32, 64 or 128");
    if (shape->n_layers < 1 || shape->n_q_heads < 1 || shape->d_model < 1)
        return fail(KVE_EINVAL, "lorekv_prepare_wo: sizes must be positive");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int *flag = nullptr;
    cudaError_t e = cudaMallocAsync(&flag, sizeof(int), st);
    if (e != cudaSuccess) return cuda_fail(e, "lorekv_prepare_wo: flag");
    cudaMemsetAsync(flag, 0, sizeof(int), st);
    e = launch_prepare_wo(shape->n_layers, shape->n_q_heads, d, shape->d_model, shape->dtype, W_O,
                          L_out, G_out, flag, st);
    if (e != cudaSuccess) {
        cudaFreeAsync(flag, st);
        return cuda_fail(e, "lorekv_prepare_wo: launch");
    }
    int h_flag = 0;
    e = cudaMemcpyAsync(&h_flag, flag, sizeof(int), cudaMemcpyDeviceToHost, st);
    cudaFreeAsync(flag, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "lorekv_prepare_wo: synchronize");
    if (h_flag) return fail(KVE_ENOTPD, "lorekv_prepare_wo: W_O^h^T W_O^h is not positive definite");
    return KVE_OK;
}

size_t lorekv_workspace_size(const KveShape *shape, const KveLorekvParams *params) {
    LorekvDims D;
    const char *why;
    if (!lorekv_dims(shape, params, &D, &why)) return 0;
    return lorekv_ws_layout(D).total;
}

int lorekv_kept_capacity(const KveShape *shape, const KveLorekvParams *params) {
    LorekvDims D;
    const char *why;
    if (!lorekv_dims(shape, params, &D, &why)) return -fail(KVE_EINVAL, "lorekv_kept_capacity: %s", why);
    const int mid = D.n - D.sink - D.w;
    return (mid <= D.B) ? D.n : D.sink + D.B + D.w;
}

static int score_common(const char *fn, const KveShape *shape, const KveLorekvParams *params,
                        const void *K, const void *V, const void *Q_W, const void *Q_look,
                        void *workspace, size_t ws_bytes, LorekvDims *D, LorekvWorkspace *W) {
    if (int s = injected()) return s;
    const char *why;
    if (!shape || !params) return fail(KVE_EINVAL, "%s: null shape or params", fn);
    if (shape->dtype != KVE_F32 && shape->dtype != KVE_BF16)
        return fail(KVE_EDTYPE, "%s: dtype must be KVE_F32 or KVE_BF16", fn);
    if (!lorekv_dims(shape, params, D, &why)) return fail(KVE_EINVAL, "%s: %s", fn, why);
    if (!K || !V || !Q_W || !Q_look) return fail(KVE_EINVAL, "%s: null tensor argument", fn);
    *W = lorekv_ws_layout(*D);
    if (!workspace || ws_bytes < W->total)
        return fail(KVE_EWORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, W->total,
                    workspace ? ws_bytes : (size_t)0);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(KVE_EINVAL, "%s: workspace must be 256-byte aligned", fn);
    return KVE_OK;
}

static cudaError_t run_attention(const LorekvDims &D, const LorekvWorkspace &W, const void *K,
                                 const void *V, const void *Q_W, const void *Q_look, void *ws,
                                 cudaStream_t st) {
    if (tc_supported(D)) {
        {
            ProfScope ps("pack_queries", 1, st);
            cudaError_t e = launch_pack_queries(D, Q_W, Q_look, ws, W, st);
            if (e != cudaSuccess) return e;
        }
        ProfScope ps("attention", 1, st);
        return launch_attention_tc(D, K, V, ws, W, device_error_word(), st);
    }
    ProfScope ps("attention", 1, st);
    return launch_attention_simt(D, K, V, Q_W, Q_look, ws, W, st);
}

int lorekv_attention_stats(const KveShape *shape, const KveLorekvParams *params, const void *K,
                           const void *V, const void *Q_W, const void *Q_look, float *lse_out,
                           float *o_out, void *workspace, size_t ws_bytes, void *stream) {
    LorekvDims D;
    LorekvWorkspace W;
    if (int s = score_common("lorekv_attention_stats", shape, params, K, V, Q_W, Q_look,
                             workspace, ws_bytes, &D, &W))
        return s;
    if (!lse_out || !o_out) return fail(KVE_EINVAL, "lorekv_attention_stats: null output");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = run_attention(D, W, K, V, Q_W, Q_look, workspace, st);
    if (e == cudaSuccess) {
        ProfScope ps("combine", 1, st);
        e = launch_combine(D, workspace, W, lse_out, o_out, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "lorekv_attention_stats: launch");
    return KVE_OK;
}

int lorekv_output_fidelity(const float *o_full, const float *o_comp, int rows, int d_head,
                           float *cos_out, float *mean_out, void *stream) {
    if (int s = injected()) return s;
    if (!o_full || !o_comp || !cos_out)
        return fail(KVE_EINVAL, "lorekv_output_fidelity: null argument");
    if (rows < 1 || d_head < 1)
        return fail(KVE_EINVAL, "lorekv_output_fidelity: rows and d_head must be >= 1");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    {
        ProfScope ps("fidelity", mean_out ? 2 : 1, st);
        e = launch_output_fidelity(o_full, o_comp, rows, d_head, cos_out, mean_out, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "lorekv_output_fidelity: launch");
    return KVE_OK;
}

// ---- counter-causal surprise refresh ----------------------------------------------------------

static int cc_dims(const char *fn, const KveCcShape *sh, CcDims *D) {
    if (!sh) return fail(KVE_EINVAL, "%s: null shape", fn);
    if (sh->dtype != KVE_F32 && sh->dtype != KVE_BF16)
        return fail(KVE_EDTYPE, "%s: dtype must be KVE_F32 or KVE_BF16", fn);
    if (sh->n_seq < 1 || sh->n_tokens < 1 || sh->n_q_heads < 1 || sh->n_kv_heads < 1 ||
        sh->d_model < 1 || sh->vocab < 1)
        return fail(KVE_EINVAL, "%s: sizes must be >= 1", fn);
    if (sh->n_q_heads % sh->n_kv_heads != 0)
        return fail(KVE_EINVAL, "%s: n_q_heads must be a multiple of n_kv_heads", fn);
    if (sh->d_head != 32 && sh->d_head != 64 && sh->d_head != 128)
        return fail(KVE_EINVAL, "%s: d_head must be 32, 64 or 128", fn);
    if (sh->sink < 0 || sh->sink > sh->n_tokens)
        return fail(KVE_EINVAL, "%s: sink must be in [0, n_tokens]", fn);
    if (sh->keep_J < 1 || sh->keep_J > sh->n_tokens)
        return fail(KVE_EINVAL, "%s: keep_J must be in [1, n_tokens]", fn);
    // launch-grid limits: y = query heads / column tiles, z = sequences
    if (sh->n_seq > 65535 || sh->n_q_heads > 65535 || sh->d_model > (1 << 22))
        return fail(KVE_EINVAL, "%s: n_seq, n_q_heads or d_model too large", fn);
    // query rows (sequence, head, token) are addressed with 32-bit indices and TMA coordinates
    if ((long long)sh->n_seq * sh->n_q_heads * sh->n_tokens >= (1LL << 31))
        return fail(KVE_EINVAL, "%s: n_seq * n_q_heads * n_tokens must be below 2^31", fn);
    *D = CcDims{sh->n_seq, sh->n_q_heads, sh->n_kv_heads, sh->d_head, sh->d_model, sh->n_tokens,
                sh->vocab, sh->dtype, sh->sink, sh->keep_J, sh->n_tokens};
    return KVE_OK;
}

size_t cc_workspace_size(const KveCcShape *shape) {
    CcDims D;
    if (cc_dims("cc_workspace_size", shape, &D) != KVE_OK) return 0;
    return cc_workspace_bytes(D);
}

int cc_surprise(const KveCcShape *shape, const void *K, const void *V, const void *Q_fresh,
                const void *H_last, const void *W_O, const void *W_U, const int32_t *tokens,
                float *surprise_out, void *workspace, size_t ws_bytes, void *stream) {
    if (int s = injected()) return s;
    CcDims D;
    if (int s = cc_dims("cc_surprise", shape, &D)) return s;
    if (!K || !V || !Q_fresh || !H_last || !W_O || !W_U || !tokens || !surprise_out)
        return fail(KVE_EINVAL, "cc_surprise: null argument");
    if (!workspace || ws_bytes < cc_workspace_bytes(D))
        return fail(KVE_EWORKSPACE, "cc_surprise: workspace of %zu bytes needed, %zu given",
                    cc_workspace_bytes(D), ws_bytes);
    unsigned *err = device_error_word();
    if (!err) return fail(KVE_ECUDA, "cc_surprise: no device error word");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    {
        ProfScope ps("cc_attention", 1, st);
        e = launch_cc_attention(D, K, V, Q_fresh, workspace, err, st);
    }
    if (e == cudaSuccess) {
        ProfScope ps("cc_logits", 2, st);
        e = launch_cc_logits(D, H_last, W_O, W_U, tokens, surprise_out, workspace, err, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "cc_surprise: launch");
    return KVE_OK;
}

int cc_select_compact(const KveCcShape *shape, const float *surprise, const void *K,
                      const void *V, const int32_t *tokens, int32_t *kept_idx, void *K_out,
                      void *V_out, int32_t *tokens_out, void *stream) {
    if (int s = injected()) return s;
    CcDims D;
    if (int s = cc_dims("cc_select_compact", shape, &D)) return s;
    if (!surprise || !K || !V || !tokens || !kept_idx || !K_out || !V_out || !tokens_out)
        return fail(KVE_EINVAL, "cc_select_compact: null argument");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    {
        ProfScope ps("cc_select_compact", 2, st);
        e = launch_cc_select(D, surprise, K, V, tokens, kept_idx, K_out, V_out, tokens_out, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "cc_select_compact: launch");
    return KVE_OK;
}

int lorekv_score(const KveShape *shape, const KveLorekvParams *params, const void *K,
                 const void *V, const void *Q_W, const void *Q_look, const float *L,
                 const float *G, const float *logits, const int32_t *sampled, float *scores_out,
                 float *omega_out, void *workspace, size_t ws_bytes, void *stream) {
    LorekvDims D;
    LorekvWorkspace W;
    if (int s = score_common("lorekv_score", shape, params, K, V, Q_W, Q_look, workspace,
                             ws_bytes, &D, &W))
        return s;
    if (!L || !G || !logits || !sampled || !scores_out || !omega_out)
        return fail(KVE_EINVAL, "lorekv_score: null argument");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool tc = tc_supported(D);
    cudaError_t e;
    {
        ProfScope ps("reliability", (D.lambda_D != 0.f && D.M > 1) ? 3 : 2, st);
        e = launch_reliability(D, Q_look, logits, sampled, omega_out, workspace, W, st);
    }
    if (e == cudaSuccess) e = run_attention(D, W, K, V, Q_W, Q_look, workspace, st);
    if (e == cudaSuccess) {
        ProfScope ps("combine", 1, st);
        e = launch_combine(D, workspace, W, nullptr, nullptr, st);
    }
    if (e == cudaSuccess) {
        ProfScope ps("prep_u", 1, st);
        e = launch_prep_u(D, G, omega_out, workspace, W, st, Q_W, Q_look, tc);
    }
    if (e == cudaSuccess) {
        ProfScope ps("scores", tc ? 4 : 1, st);
        if (tc)
            e = launch_scores_tc(D, K, V, L, workspace, W, scores_out, device_error_word(), st);
        else
            e = launch_scores_simt(D, K, V, Q_W, Q_look, L, workspace, W, scores_out, st);
    }
    if (e == cudaSuccess) {  // pairs with a > 1/4, left out above, evaluated exactly
        ProfScope ps("peak_fix", 2, st);
        e = launch_peak_fix(D, K, V, Q_W, Q_look, L, workspace, W, scores_out, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "lorekv_score: launch");
    return KVE_OK;
}

int lorekv_select_compact(const KveShape *shape, const KveLorekvParams *params,
                          const float *scores, const void *K, const void *V, int32_t *kept_idx,
                          int32_t *kept_len, void *K_out, void *V_out, void *workspace,
                          size_t ws_bytes, void *stream) {
    (void)workspace;
    (void)ws_bytes;
    if (int s = injected()) return s;
    LorekvDims D;
    const char *why;
    if (!shape || !params) return fail(KVE_EINVAL, "lorekv_select_compact: null shape or params");
    if (shape->dtype != KVE_F32 && shape->dtype != KVE_BF16)
        return fail(KVE_EDTYPE, "lorekv_select_compact: dtype must be KVE_F32 or KVE_BF16");
    if (!lorekv_dims(shape, params, &D, &why))
        return fail(KVE_EINVAL, "lorekv_select_compact: %s", why);
    if (!scores || !K || !V || !kept_idx || !kept_len || !K_out || !V_out)
        return fail(KVE_EINVAL, "lorekv_select_compact: null argument");
    const int mid = D.n - D.sink - D.w;
    const int cap = (mid <= D.B) ? D.n : D.sink + D.B + D.w;
    cudaError_t e;
    {
        ProfScope ps("select_compact", 1, static_cast<cudaStream_t>(stream));
        e = launch_select_compact(D, scores, K, V, kept_idx, kept_len, K_out, V_out, cap,
                                  static_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) return cuda_fail(e, "lorekv_select_compact: launch");
    return KVE_OK;
}

// ---- counter-causal refresh cycle ------------------------------------------------------------------
static size_t cc_row_bytes(const CcDims &D, int which) {  // 0 K/V, 1 Q, 2 H
    const size_t es = dtype_size(D.dtype);
    return which == 2 ? (size_t)D.dm * es : (size_t)D.d * es;
}

int cc_cache_create(KveCcCache **out, const KveCcShape *shape) {
    if (int s = injected()) return s;
    if (!out) return fail(KVE_EINVAL, "cc_cache_create: null out");
    *out = nullptr;
    CcDims D;
    if (int s = cc_dims("cc_cache_create", shape, &D)) return s;
    if (D.J >= D.n) return fail(KVE_EINVAL, "cc_cache_create: n_tokens must exceed keep_J (h = n_tokens - keep_J >= 1)");
    if (D.J < D.sink + 1) return fail(KVE_EINVAL, "cc_cache_create: keep_J must be at least sink + 1");
    if ((D.dm * dtype_size(D.dtype)) % 16 != 0)
        return fail(KVE_EINVAL, "cc_cache_create: d_model rows must be a multiple of 16 bytes");
    KveCcCache *c = new KveCcCache();
    c->D = D;
    c->h = D.n - D.J;
    const size_t rows = (size_t)D.batch * D.n;
    cudaError_t e = cudaSuccess;
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
        KveCcCache::Buf &b = c->buf[k];
        const size_t kv = rows * D.hkv * cc_row_bytes(D, 0), q = rows * D.hq * cc_row_bytes(D, 1),
                     hb = rows * cc_row_bytes(D, 2);
        // zero-filled: rows past the scored ones are read (and multiplied by 0) by the tensor-core
        // attention, so they must hold finite values
        if (e == cudaSuccess) e = cudaMalloc(&b.K, kv);
        if (e == cudaSuccess) e = cudaMemset(b.K, 0, kv);
        if (e == cudaSuccess) e = cudaMalloc(&b.V, kv);
        if (e == cudaSuccess) e = cudaMemset(b.V, 0, kv);
        if (e == cudaSuccess) e = cudaMalloc(&b.Q, q);
        if (e == cudaSuccess) e = cudaMemset(b.Q, 0, q);
        if (e == cudaSuccess) e = cudaMalloc(&b.H, hb);
        if (e == cudaSuccess) e = cudaMemset(b.H, 0, hb);
        if (e == cudaSuccess) e = cudaMalloc(&b.X, rows * sizeof(int32_t));
        if (e == cudaSuccess) e = cudaMemset(b.X, 0, rows * sizeof(int32_t));
        if (e == cudaSuccess) e = cudaMalloc(&b.pos, rows * sizeof(int32_t));
        if (e == cudaSuccess) e = cudaMemset(b.pos, 0xff, rows * sizeof(int32_t));
    }
    c->ws_bytes = cc_workspace_bytes(D);
    if (e == cudaSuccess) e = cudaMalloc(&c->ws, c->ws_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&c->surprise, rows * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&c->kept, (size_t)D.batch * D.J * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cc_cache_destroy(c);
        return cuda_fail(e, "cc_cache_create: allocate");
    }
    *out = c;
    return KVE_OK;
}

int cc_cache_append(KveCcCache *c, const void *K_new, const void *V_new, const void *Q_new,
                    const void *H_new, const int32_t *tokens_new, int count, void *stream) {
    if (int s = injected()) return s;
    if (!c || !K_new || !V_new || !Q_new || !H_new || !tokens_new)
        return fail(KVE_EINVAL, "cc_cache_append: null argument");
    if (count < 1 || count > c->h - c->recent)
        return fail(KVE_EINVAL, "cc_cache_append: count must be in [1, %d] (free rows of the chunk)",
                    c->h - c->recent);
    const CcDims &D = c->D;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    KveCcCache::Buf &b = c->buf[c->cur];
    const int at = c->mem + c->recent;
    cudaError_t e;
    {
        ProfScope ps("cc_append", 1, st);
        CcGatherSet G{};
        cc_gather_add(&G, K_new, b.K, D.batch, D.hkv, cc_row_bytes(D, 0), count);
        cc_gather_add(&G, V_new, b.V, D.batch, D.hkv, cc_row_bytes(D, 0), count);
        cc_gather_add(&G, Q_new, b.Q, D.batch, D.hq, cc_row_bytes(D, 1), count);
        cc_gather_add(&G, H_new, b.H, D.batch, 1, cc_row_bytes(D, 2), count);
        e = launch_cc_append(G, count, at, D.ld, tokens_new, b.X, b.pos, D.batch, c->seen, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "cc_cache_append: launch");
    c->recent += count;
    c->seen += count;
    return KVE_OK;
}

int cc_cache_refresh(KveCcCache *c, const void *W_O, const void *W_U, void *stream) {
    if (int s = injected()) return s;
    if (!c || !W_O || !W_U) return fail(KVE_EINVAL, "cc_cache_refresh: null argument");
    const int cand = c->mem + c->recent;
    if (cand <= c->D.J) {  // nothing to evict: every candidate is kept, in place and in order
        c->mem = cand;
        c->recent = 0;
        return KVE_OK;
    }
    unsigned *err = device_error_word();
    if (!err) return fail(KVE_ECUDA, "cc_cache_refresh: no device error word");
    CcDims D = c->D;
    D.n = cand;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const KveCcCache::Buf &a = c->buf[c->cur];
    KveCcCache::Buf &b = c->buf[c->cur ^ 1];
    cudaError_t e;
    {
        ProfScope ps("cc_attention", 1, st);
        e = launch_cc_attention(D, a.K, a.V, a.Q, c->ws, err, st);
    }
    if (e == cudaSuccess) {
        ProfScope ps("cc_logits", 2, st);
        e = launch_cc_logits(D, a.H, W_O, W_U, a.X, c->surprise, c->ws, err, st);
    }
    if (e == cudaSuccess) {
        ProfScope ps("cc_select_compact", 2, st);
        e = launch_cc_select_idx(D, c->surprise, a.X, a.pos, c->kept, b.X, b.pos, D.ld, st);
        if (e == cudaSuccess) {
            CcGatherSet G{};
            cc_gather_add(&G, a.K, b.K, D.batch, D.hkv, cc_row_bytes(D, 0), D.J);
            cc_gather_add(&G, a.V, b.V, D.batch, D.hkv, cc_row_bytes(D, 0), D.J);
            cc_gather_add(&G, a.Q, b.Q, D.batch, D.hq, cc_row_bytes(D, 1), D.J);
            cc_gather_add(&G, a.H, b.H, D.batch, 1, cc_row_bytes(D, 2), D.J);
            e = launch_cc_gather(G, c->kept, D.J, D.ld, D.ld, st);
        }
    }
    if (e != cudaSuccess) return cuda_fail(e, "cc_cache_refresh: launch");
    c->cur ^= 1;
    c->mem = D.J;
    c->recent = 0;
    return KVE_OK;
}

int cc_cache_step(KveCcCache *c, const void *K_new, const void *V_new, const void *Q_new,
                  const void *H_new, const int32_t *tokens_new, int count, const void *W_O,
                  const void *W_U, int *refreshed, void *stream) {
    if (refreshed) *refreshed = 0;
    if (!c || !W_O || !W_U) return fail(KVE_EINVAL, "cc_cache_step: null argument");
    if (int s = cc_cache_append(c, K_new, V_new, Q_new, H_new, tokens_new, count, stream))
        return s;
    if (c->recent < c->h) return KVE_OK;
    if (int s = cc_cache_refresh(c, W_O, W_U, stream)) return s;
    if (refreshed) *refreshed = 1;
    return KVE_OK;
}

int cc_cache_export(const KveCcCache *c, void *K, void *V, void *Q, void *H, int32_t *tokens,
                    int32_t *pos, void *stream) {
    if (int s = injected()) return s;
    if (!c) return fail(KVE_EINVAL, "cc_cache_export: null cache");
    const CcDims &D = c->D;
    const int len = c->mem + c->recent;
    if (len == 0) return KVE_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const KveCcCache::Buf &b = c->buf[c->cur];
    const size_t ld = (size_t)D.ld;
    struct Part {
        void *dst;
        const void *src;
        size_t row;
        size_t blocks;
    } parts[6] = {{K, b.K, cc_row_bytes(D, 0), (size_t)D.batch * D.hkv},
                  {V, b.V, cc_row_bytes(D, 0), (size_t)D.batch * D.hkv},
                  {Q, b.Q, cc_row_bytes(D, 1), (size_t)D.batch * D.hq},
                  {H, b.H, cc_row_bytes(D, 2), (size_t)D.batch},
                  {tokens, b.X, sizeof(int32_t), (size_t)D.batch},
                  {pos, b.pos, sizeof(int32_t), (size_t)D.batch}};
    for (const Part &p : parts) {
        if (!p.dst) continue;
        cudaError_t e = cudaMemcpy2DAsync(p.dst, len * p.row, p.src, ld * p.row, len * p.row,
                                          p.blocks, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "cc_cache_export: copy");
    }
    return KVE_OK;
}

int cc_cache_length(const KveCcCache *c) { return c ? c->mem + c->recent : -KVE_EINVAL; }
int cc_cache_seen(const KveCcCache *c) { return c ? c->seen : -KVE_EINVAL; }

void cc_cache_destroy(KveCcCache *c) {
    if (!c) return;
    for (auto &b : c->buf) {
        cudaFree(b.K);
        cudaFree(b.V);
        cudaFree(b.Q);
        cudaFree(b.H);
        cudaFree(b.X);
        cudaFree(b.pos);
    }
    cudaFree(c->ws);
    cudaFree(c->surprise);
    cudaFree(c->kept);
    delete c;
}

// ---- H2O -------------------------------------------------------------------------------------------
int h2o_state_create(KveH2O **out, int batch, int n_layers, int n_heads, int d_head, int max_len,
                     float budget_frac, int dtype) {
    if (int s = injected()) return s;
    if (!out) return fail(KVE_EINVAL, "h2o_state_create: null out");
    *out = nullptr;
    if (dtype != KVE_F16 && dtype != KVE_BF16)
        return fail(KVE_EDTYPE, "h2o_state_create: dtype must be KVE_F16 or KVE_BF16");
    if (batch < 1 || n_layers < 1 || n_heads < 1 || max_len < 1)
        return fail(KVE_EINVAL, "h2o_state_create: sizes must be positive");
    if (d_head != 64 && d_head != 128) return fail(KVE_EINVAL, "h2o_state_create: d_head must be 64 or 128");
    if (!(budget_frac > 0.f && budget_frac <= 1.f))
        return fail(KVE_EINVAL, "h2o_state_create: budget_frac must be in (0, 1]");
    const int cap = (int)floor((double)budget_frac * (double)max_len) + 1;
    if (cap > 4096) return fail(KVE_EINVAL, "h2o_state_create: slot capacity %d > 4096", cap);
    // prompt rows (unit, position) are addressed with 32-bit indices and TMA coordinates
    if ((long long)batch * n_layers * n_heads * max_len >= (1LL << 31))
        return fail(KVE_EINVAL, "h2o_state_create: batch * n_layers * n_heads * max_len must be below 2^31");
    KveH2O *h = new KveH2O();
    H2OState &s = h->s;
    s.batch = batch;
    s.L = n_layers;
    s.H = n_heads;
    s.d = d_head;
    s.max_len = max_len;
    s.cap = cap;
    s.dtype = dtype;
    s.frac = budget_frac;
    s.units = batch * n_layers * n_heads;
    s.t = 0;
    s.prefilled = 0;
    const size_t rows = (size_t)s.units * cap;
    cudaError_t e = cudaMalloc(&s.K, rows * d_head * 2);
    if (e == cudaSuccess) e = cudaMalloc(&s.V, rows * d_head * 2);
    if (e == cudaSuccess) e = cudaMalloc(&s.acc, rows * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&s.pos, rows * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&s.nslots, s.units * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&s.hole, s.units * sizeof(int32_t));
    // scratch of the prefill's partial column sums, sized for a prompt of max_len tokens
    if (e == cudaSuccess)
        e = cudaMalloc(&s.prefill_part, sizeof(float) * (size_t)s.units * kColsumTcParts * max_len);
    if (e == cudaSuccess) e = cudaMemset(s.K, 0, rows * d_head * 2);
    if (e == cudaSuccess) e = cudaMemset(s.V, 0, rows * d_head * 2);
    if (e == cudaSuccess) e = cudaMemset(s.acc, 0, rows * sizeof(float));
    if (e == cudaSuccess) e = cudaMemset(s.pos, 0xff, rows * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(s.nslots, 0, s.units * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(s.hole, 0xff, s.units * sizeof(int32_t));
    if (e != cudaSuccess) {
        h2o_state_destroy(h);
        return cuda_fail(e, "h2o_state_create: allocate");
    }
    *out = h;
    return KVE_OK;
}

int h2o_prefill(KveH2O *h, const void *K, const void *V, const void *Q, int prompt_len,
                void *stream) {
    if (int s = injected()) return s;
    if (!h || !K || !V || !Q) return fail(KVE_EINVAL, "h2o_prefill: null argument");
    H2OState &s = h->s;
    if (s.prefilled) return fail(KVE_EINVAL, "h2o_prefill: state already holds a prompt");
    if (prompt_len < 1 || prompt_len > s.max_len)
        return fail(KVE_EINVAL, "h2o_prefill: prompt_len must be in [1, max_len]");
    if (!h2o_prefill_fits(s.d, prompt_len, s.dtype))
        return fail(KVE_EINVAL, "h2o_prefill: prompt of %d tokens exceeds the on-chip prefill", prompt_len);
    cudaError_t e;
    {
        ProfScope ps("h2o_prefill", 1, static_cast<cudaStream_t>(stream));
        e = launch_h2o_prefill(s, K, V, Q, prompt_len, static_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) return cuda_fail(e, "h2o_prefill: launch");
    s.t = prompt_len;
    s.prefilled = 1;
    return KVE_OK;
}

int h2o_decode_step(KveH2O *h, const void *q, const void *k_new, const void *v_new,
                    void *attn_out, void *stream) {
    if (int s = injected()) return s;
    if (!h || !q || !k_new || !v_new || !attn_out) return fail(KVE_EINVAL, "h2o_decode_step: null argument");
    H2OState &s = h->s;
    if (!s.prefilled) return fail(KVE_EINVAL, "h2o_decode_step: call h2o_prefill first");
    if (s.t >= s.max_len) return fail(KVE_EINVAL, "h2o_decode_step: max_len reached");
    cudaError_t e;
    {
        ProfScope ps("h2o_step", 1, static_cast<cudaStream_t>(stream));
        e = launch_h2o_step(s, q, k_new, v_new, attn_out, static_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) return cuda_fail(e, "h2o_decode_step: launch");
    s.t += 1;
    return KVE_OK;
}

int h2o_export(const KveH2O *h, void *K, void *V, int32_t *pos, float *acc, int32_t *count,
               void *stream) {
    if (int s = injected()) return s;
    if (!h) return fail(KVE_EINVAL, "h2o_export: null state");
    cudaError_t e = launch_h2o_export(h->s, K, V, pos, acc, count, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "h2o_export: launch");
    return KVE_OK;
}

int h2o_capacity(const KveH2O *h) { return h ? h->s.cap : -KVE_EINVAL; }
int h2o_length(const KveH2O *h) { return h ? h->s.t : -KVE_EINVAL; }

void h2o_state_destroy(KveH2O *h) {
    if (!h) return;
    H2OState &s = h->s;
    cudaFree(s.K);
    cudaFree(s.V);
    cudaFree(s.acc);
    cudaFree(s.pos);
    cudaFree(s.nslots);
    cudaFree(s.hole);
    cudaFree(s.prefill_part);
    delete h;
}

}  // extern "C"

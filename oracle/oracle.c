/*
 * fp64 CPU oracle for the KV-cache eviction pass. TEST INFRASTRUCTURE ONLY: the library's CUDA
 * path never calls, links or loads this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.
 *
 * Everything here is written from the pages' statement of the method, in double precision, with
 * no blocking, fusion or reordering beyond what the definitions state:
 *
 *   LORE-KV (project page "LORE-KV: Monte Carlo Estimation for KV-Cache Eviction"):
 *     Method, "Reliability weights" (Eqs. 2-4, 10): c_u = log q(y_u|h_u) + H(q(.|h_u)),
 *        R_m = beta*cbar_m - gamma*Hbar_m - lambda_D*Dhat_m, omega = softmax(R).
 *     Method, "Projected deletion score" (Eqs. 5-7): Delta o = a/(1-a+eps) (v_i - o_q),
 *        e = ||W_O Delta o||, S_i = psi(E_{i,W}) + lambda_L sum_m omega_m psi(E_{i,m}).
 *     Method, "Evict and decode" (Eq. 8) and the "Hyperparameters" table: protected sink and
 *        window, chunks of 4 adjacent tokens, top-B per KV head.
 *   H2O (paper summary "H2O: Heavy-Hitter Oracle ..."):
 *     Section 2.1 (attention o_i = D_i^-1 exp(Q_i K^T)), Definitions 2.1/2.2, Section 4.1
 *     Algorithm 1 (accumulated score, greedy eviction with linear h), Appendix A (k/2 recent).
 *
 * Readings of points the pages leave open (the same readings the CUDA path implements):
 *   - attention logits are q.k / sqrt(d_head); inputs are post-rotary.
 *   - window query r (0-based) sits at position n-w+r and sees tokens i <= n-w+r when
 *     window_causal is set; lookahead queries see all n cached tokens.
 *   - psi is the arithmetic mean over the set's queries, taken over all g query heads that
 *     share the KV head; each query head uses its own W_O^h (columns h*d .. h*d+d-1).
 *   - ||W_O^h x|| is evaluated as ||L_h^T x|| with G_h = W_O^h^T W_O^h = L_h L_h^T (Cholesky);
 *     L_h^T (v_i - o_q) is formed as L_h^T v_i - L_h^T o_q (the linear map applied to both terms).
 *   - Dhat_m: qbar_m^{l,h} = mean over the T lookahead queries of trajectory m;
 *     D_m = 1 - mean_{m' != m} mean_{l,h} cos(qbar_m, qbar_m'); Dhat = (D - mean D) / std(D)
 *     (population std), Dhat = 0 when std < 1e-12 or M = 1.
 *   - protected set = [0, sink) U [n-w, n); chunk c covers [sink+4c, sink+4c+4); chunk score =
 *     mean S over the chunk; keep the top B/chunk chunks, higher score first, equal scores ->
 *     lower chunk index; kept positions ascending. If n - sink - w <= B every token is kept.
 *     S_i is reported as 0 for protected tokens.
 *   - H2O: t = tokens seen so far (including the new one); k_t = floor(frac*t),
 *     r_t = floor(k_t/2) most recent positions are never evicted; while more than k_t tokens are
 *     held, evict the minimum accumulated score among positions < t - r_t, ties -> oldest.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define KVO_OK 0
#define KVO_EINVAL 1
#define KVO_ENOTPD 4

/* ---------------------------------------------------------------------------------------------
 * Reliability weights (LORE-KV page, Method, "Reliability weights", Eqs. 2-4, 10)
 * ------------------------------------------------------------------------------------------- */

/* One vocabulary row: lse = log sum_v exp z_v, H = -sum_v p_v log p_v, logq = log p_{y}. */
void kvo_row_stats(long V, const double *z, long y, double *lse, double *H, double *logq)
{
    double mx = z[0];
    for (long v = 1; v < V; ++v)
        if (z[v] > mx) mx = z[v];
    double sum = 0.0;
    for (long v = 0; v < V; ++v) sum += exp(z[v] - mx);
    double l = mx + log(sum);
    double h = 0.0;
    for (long v = 0; v < V; ++v) {
        double logp = z[v] - l;
        double p = exp(logp);
        if (p > 0.0) h -= p * logp; /* 0 log 0 = 0: a -inf logit (masked token) adds nothing */
    }
    *lse = l;
    *H = h;
    *logq = z[y] - l;
}

/* Standardised cosine disagreement of each trajectory's mean lookahead query with the others.
 * qlook: [LH][M*T][d] for one sequence (LH = layers x query heads). */
void kvo_disagreement(int M, int T, int LH, int d, const double *qlook, double *Dhat)
{
    if (M <= 1) {
        for (int m = 0; m < M; ++m) Dhat[m] = 0.0;
        return;
    }
    double *qbar = (double *)calloc((size_t)M * d, sizeof(double));
    double *D = (double *)calloc((size_t)M, sizeof(double));
    for (int lh = 0; lh < LH; ++lh) {
        for (int m = 0; m < M; ++m) {
            for (int k = 0; k < d; ++k) {
                double s = 0.0;
                for (int t = 0; t < T; ++t) s += qlook[((size_t)lh * M * T + (size_t)m * T + t) * d + k];
                qbar[(size_t)m * d + k] = s / T;
            }
        }
        for (int m = 0; m < M; ++m) {
            for (int m2 = 0; m2 < M; ++m2) {
                if (m2 == m) continue;
                double dot = 0.0, na = 0.0, nb = 0.0;
                for (int k = 0; k < d; ++k) {
                    double a = qbar[(size_t)m * d + k], b = qbar[(size_t)m2 * d + k];
                    dot += a * b;
                    na += a * a;
                    nb += b * b;
                }
                double cs = (na > 0.0 && nb > 0.0) ? dot / (sqrt(na) * sqrt(nb)) : 0.0;
                D[m] += cs; /* summed over m2 != m and over (layer, head) */
            }
        }
    }
    for (int m = 0; m < M; ++m) D[m] = 1.0 - D[m] / ((double)(M - 1) * LH);
    double mean = 0.0;
    for (int m = 0; m < M; ++m) mean += D[m];
    mean /= M;
    double var = 0.0;
    for (int m = 0; m < M; ++m) var += (D[m] - mean) * (D[m] - mean);
    double sd = sqrt(var / M);
    for (int m = 0; m < M; ++m) Dhat[m] = (sd < 1e-12) ? 0.0 : (D[m] - mean) / sd;
    free(qbar);
    free(D);
}

/* Per-sequence reliability: rows u = m*T + t of logits [M*T][V], sampled ids y[M*T].
 * Outputs: c[M*T], H[M*T], Dhat[M], R[M], omega[M]. */
int kvo_reliability(int M, int T, long V, const double *logits, const int *y, int LH, int d,
                    const double *qlook, double beta, double gamma, double lambda_D, double *c,
                    double *H, double *Dhat, double *R, double *omega)
{
    if (M < 1 || T < 1 || V < 1) return KVO_EINVAL;
    for (int u = 0; u < M * T; ++u) {
        if (y[u] < 0 || y[u] >= V) return KVO_EINVAL;
        double lse, h, logq;
        kvo_row_stats(V, logits + (size_t)u * V, y[u], &lse, &h, &logq);
        H[u] = h;
        c[u] = logq + h;
    }
    if (lambda_D != 0.0)
        kvo_disagreement(M, T, LH, d, qlook, Dhat);
    else
        for (int m = 0; m < M; ++m) Dhat[m] = 0.0;
    double rmax = -INFINITY;
    for (int m = 0; m < M; ++m) {
        double cb = 0.0, hb = 0.0;
        for (int t = 0; t < T; ++t) {
            cb += c[m * T + t];
            hb += H[m * T + t];
        }
        cb /= T;
        hb /= T;
        R[m] = beta * cb - gamma * hb - lambda_D * Dhat[m];
        if (R[m] > rmax) rmax = R[m];
    }
    double z = 0.0;
    for (int m = 0; m < M; ++m) z += exp(R[m] - rmax);
    for (int m = 0; m < M; ++m) omega[m] = exp(R[m] - rmax) / z;
    return KVO_OK;
}

/* ---------------------------------------------------------------------------------------------
 * Output-projection Gram matrix and its Cholesky factor (LORE-KV page, Eqs. 5-7: e = ||W_O Delta o||)
 * W: [d_model][ncols] (row-major o_proj weight); head h owns columns h*d .. h*d+d-1.
 * G = W_h^T W_h, G = L L^T with L lower triangular. Returns KVO_ENOTPD if a pivot is <= 0.
 * ------------------------------------------------------------------------------------------- */
int kvo_gram_cholesky(int d_model, int ncols, int d, const double *W, int h, double *G, double *L)
{
    if ((long)(h + 1) * d > ncols) return KVO_EINVAL;
    for (int j = 0; j < d; ++j)
        for (int k = 0; k < d; ++k) {
            double s = 0.0;
            for (int r = 0; r < d_model; ++r)
                s += W[(size_t)r * ncols + (size_t)h * d + j] * W[(size_t)r * ncols + (size_t)h * d + k];
            G[(size_t)j * d + k] = s;
        }
    memset(L, 0, sizeof(double) * (size_t)d * d);
    for (int j = 0; j < d; ++j) {
        double s = G[(size_t)j * d + j];
        for (int k = 0; k < j; ++k) s -= L[(size_t)j * d + k] * L[(size_t)j * d + k];
        if (!(s > 0.0)) return KVO_ENOTPD;
        double piv = sqrt(s);
        L[(size_t)j * d + j] = piv;
        for (int i = j + 1; i < d; ++i) {
            double t = G[(size_t)i * d + j];
            for (int k = 0; k < j; ++k) t -= L[(size_t)i * d + k] * L[(size_t)j * d + k];
            L[(size_t)i * d + j] = t / piv;
        }
    }
    return KVO_OK;
}

/* ---------------------------------------------------------------------------------------------
 * One unit (sequence, layer, KV head): attention statistics of every query, projected deletion
 * scores and the aggregated token score S (LORE-KV page, Method, Eqs. 5-7).
 *
 * K, V : [n][d]; QW: [g][w][d] window queries; QL: [g][M*T][d] lookahead queries (row m*T+t);
 * Lf   : [g][d][d] Cholesky factors of the g query heads; omega: [M].
 * S    : [n] output, 0 for protected tokens.
 * lse_out (optional): [g][w+M*T] log-sum-exp of each query's logits;
 * o_out   (optional): [g][w+M*T][d] attention outputs o_q;
 * E       (optional): [g][w+M*T][n] e_{q,i} for every token (0 where a query cannot see i).
 * ------------------------------------------------------------------------------------------- */
int kvo_lorekv_unit(int n, int d, int g, int w, int M, int T, int window_causal, int sink,
                    const double *K, const double *V, const double *QW, const double *QL,
                    const double *Lf, const double *omega, double lambda_L, double eps, double *S,
                    double *lse_out, double *o_out, double *E)
{
    if (n < sink + w || d < 1 || g < 1 || w < 1 || M < 1 || T < 1) return KVO_EINVAL;
    const int MT = M * T, nq = w + MT;
    const double scale = 1.0 / sqrt((double)d);
    double *a = (double *)malloc(sizeof(double) * (size_t)n);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)n * d); /* y_i = L_h^T v_i */
    double *z = (double *)malloc(sizeof(double) * (size_t)d);     /* z_q = L_h^T o_q */
    double *LT = (double *)malloc(sizeof(double) * (size_t)d * d); /* LT[j][k] = L_h[k][j] */
    for (int i = 0; i < n; ++i) S[i] = 0.0;
    for (int h = 0; h < g; ++h) {
        const double *Lh = Lf + (size_t)h * d * d;
        for (int j = 0; j < d; ++j)
            for (int k = 0; k < d; ++k) LT[(size_t)j * d + k] = Lh[(size_t)k * d + j];
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < d; ++j) {
                double s = 0.0;
                for (int k = 0; k < d; ++k) s += LT[(size_t)j * d + k] * V[(size_t)i * d + k];
                y[(size_t)i * d + j] = s;
            }
        for (int q = 0; q < nq; ++q) {
            const int is_window = q < w;
            const double *qv = is_window ? QW + ((size_t)h * w + q) * d : QL + ((size_t)h * MT + (q - w)) * d;
            const int nvis = (is_window && window_causal) ? n - w + q + 1 : n;
            /* a_{q,i} = softmax_i(q . k_i / sqrt(d)) over the visible tokens */
            double mx = -INFINITY;
            for (int i = 0; i < nvis; ++i) {
                double s = 0.0;
                for (int k = 0; k < d; ++k) s += qv[k] * K[(size_t)i * d + k];
                a[i] = s * scale;
                if (a[i] > mx) mx = a[i];
            }
            double den = 0.0;
            for (int i = 0; i < nvis; ++i) den += exp(a[i] - mx);
            for (int i = 0; i < nvis; ++i) a[i] = exp(a[i] - mx) / den;
            for (int i = nvis; i < n; ++i) a[i] = 0.0;
            if (lse_out) lse_out[(size_t)h * nq + q] = mx + log(den);
            /* o_q = sum_i a_{q,i} v_i */
            for (int k = 0; k < d; ++k) o[k] = 0.0;
            for (int i = 0; i < nvis; ++i)
                for (int k = 0; k < d; ++k) o[k] += a[i] * V[(size_t)i * d + k];
            if (o_out) memcpy(o_out + ((size_t)h * nq + q) * d, o, sizeof(double) * d);
            for (int j = 0; j < d; ++j) {
                double s = 0.0;
                for (int k = 0; k < d; ++k) s += LT[(size_t)j * d + k] * o[k];
                z[j] = s;
            }
            /* weight of this query in S_i: psi = mean over the set's g*w (or g*T) queries */
            double wq;
            if (is_window)
                wq = 1.0 / ((double)g * w);
            else
                wq = lambda_L * omega[(q - w) / T] / ((double)g * T);
            for (int i = 0; i < n; ++i) {
                double e = 0.0;
                if (a[i] > 0.0) {
                    double nrm = 0.0;
                    for (int j = 0; j < d; ++j) {
                        double t = y[(size_t)i * d + j] - z[j];
                        nrm += t * t;
                    }
                    e = a[i] / (1.0 - a[i] + eps) * sqrt(nrm);
                }
                if (E) E[((size_t)h * nq + q) * n + i] = e;
                if (i >= sink && i < n - w) S[i] += wq * e;
            }
        }
    }
    free(a);
    free(o);
    free(y);
    free(z);
    free(LT);
    return KVO_OK;
}

/* Many units at once, in parallel over units (OpenMP). Arrays are the per-unit arrays above
 * stacked along a leading unit axis; omega is per unit as well ([units][M]). */
int kvo_lorekv_units(int units, int n, int d, int g, int w, int M, int T, int window_causal,
                     int sink, const double *K, const double *V, const double *QW,
                     const double *QL, const double *Lf, const double *omega, double lambda_L,
                     double eps, double *S)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int u = 0; u < units; ++u) {
        bad |= kvo_lorekv_unit(n, d, g, w, M, T, window_causal, sink, K + (size_t)u * n * d,
                               V + (size_t)u * n * d, QW + (size_t)u * g * w * d,
                               QL + (size_t)u * g * M * T * d, Lf + (size_t)u * g * d * d,
                               omega + (size_t)u * M, lambda_L, eps, S + (size_t)u * n, NULL,
                               NULL, NULL);
    }
    return bad ? KVO_EINVAL : KVO_OK;
}

int kvo_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------------------------
 * Top-B chunk selection (LORE-KV page, "Evict and decode", Eq. 8; "Hyperparameters": chunk 4)
 * kept: capacity n; receives the kept positions in ascending order. chunk_scores (optional):
 * [(n-sink-w)/chunk].
 * ------------------------------------------------------------------------------------------- */
typedef struct {
    double score;
    int idx;
} kvo_chunk;

static int kvo_chunk_cmp(const void *pa, const void *pb)
{
    const kvo_chunk *a = (const kvo_chunk *)pa, *b = (const kvo_chunk *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

int kvo_select(int n, int sink, int w, int chunk, int B, const double *S, int *kept,
               int *kept_len, double *chunk_scores)
{
    if (chunk < 1 || B < 0 || sink < 0 || w < 0 || n < sink + w) return KVO_EINVAL;
    const int mid = n - sink - w;
    if (mid % chunk != 0 || B % chunk != 0) return KVO_EINVAL;
    const int nch = mid / chunk, keep = B / chunk;
    if (nch <= keep) {
        for (int i = 0; i < n; ++i) kept[i] = i;
        *kept_len = n;
        if (chunk_scores)
            for (int c = 0; c < nch; ++c) {
                double s = 0.0;
                for (int j = 0; j < chunk; ++j) s += S[sink + c * chunk + j];
                chunk_scores[c] = s / chunk;
            }
        return KVO_OK;
    }
    kvo_chunk *ch = (kvo_chunk *)malloc(sizeof(kvo_chunk) * (size_t)nch);
    for (int c = 0; c < nch; ++c) {
        double s = 0.0;
        for (int j = 0; j < chunk; ++j) s += S[sink + c * chunk + j];
        ch[c].score = s / chunk;
        ch[c].idx = c;
        if (chunk_scores) chunk_scores[c] = ch[c].score;
    }
    qsort(ch, (size_t)nch, sizeof(kvo_chunk), kvo_chunk_cmp);
    char *take = (char *)calloc((size_t)nch, 1);
    for (int r = 0; r < keep; ++r) take[ch[r].idx] = 1;
    int len = 0;
    for (int i = 0; i < sink; ++i) kept[len++] = i;
    for (int c = 0; c < nch; ++c)
        if (take[c])
            for (int j = 0; j < chunk; ++j) kept[len++] = sink + c * chunk + j;
    for (int i = n - w; i < n; ++i) kept[len++] = i;
    *kept_len = len;
    free(ch);
    free(take);
    return KVO_OK;
}

/* ---------------------------------------------------------------------------------------------
 * H2O (paper summary "H2O: Heavy-Hitter Oracle", Section 2.1, Definitions 2.1/2.2, Section 4.1)
 * ------------------------------------------------------------------------------------------- */

/* Prompt of P tokens: acc_j = sum_{i >= j} softmax_i(q_i . K_{<=i} / sqrt d)_j (causal). */
int kvo_h2o_prefill_acc(int P, int d, const double *K, const double *Q, double *acc)
{
    const double scale = 1.0 / sqrt((double)d);
    double *s = (double *)malloc(sizeof(double) * (size_t)P);
    for (int j = 0; j < P; ++j) acc[j] = 0.0;
    for (int i = 0; i < P; ++i) {
        double mx = -INFINITY;
        for (int j = 0; j <= i; ++j) {
            double t = 0.0;
            for (int k = 0; k < d; ++k) t += Q[(size_t)i * d + k] * K[(size_t)j * d + k];
            s[j] = t * scale;
            if (s[j] > mx) mx = s[j];
        }
        double den = 0.0;
        for (int j = 0; j <= i; ++j) den += exp(s[j] - mx);
        for (int j = 0; j <= i; ++j) acc[j] += exp(s[j] - mx) / den;
    }
    free(s);
    return KVO_OK;
}

/* Attention of one query over the cnt retained tokens: p = softmax(q . K / sqrt d), out = p V. */
int kvo_h2o_attend(int cnt, int d, const double *Kc, const double *Vc, const double *q, double *p,
                   double *out)
{
    const double scale = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (int j = 0; j < cnt; ++j) {
        double t = 0.0;
        for (int k = 0; k < d; ++k) t += q[k] * Kc[(size_t)j * d + k];
        p[j] = t * scale;
        if (p[j] > mx) mx = p[j];
    }
    double den = 0.0;
    for (int j = 0; j < cnt; ++j) den += exp(p[j] - mx);
    for (int j = 0; j < cnt; ++j) p[j] = exp(p[j] - mx) / den;
    for (int k = 0; k < d; ++k) out[k] = 0.0;
    for (int j = 0; j < cnt; ++j)
        for (int k = 0; k < d; ++k) out[k] += p[j] * Vc[(size_t)j * d + k];
    return KVO_OK;
}

/* Evictions at length t: k_t = floor(frac*t) tokens stay, the r_t = floor(k_t/2) most recent
 * (positions >= t - r_t) are protected; while more than k_t remain, drop the minimum accumulated
 * score among the others, ties -> oldest position. evict[j] is set to 1 for every dropped entry.
 * Returns the number of evictions, or -1 if no candidate is left. */
int kvo_h2o_evict(int cnt, const int *pos, const double *acc, int t, double frac, char *evict)
{
    const int k = (int)floor(frac * (double)t);
    const int r = k / 2;
    int alive = cnt, ne = 0;
    for (int j = 0; j < cnt; ++j) evict[j] = 0;
    while (alive > k) {
        int best = -1;
        for (int j = 0; j < cnt; ++j) {
            if (evict[j] || pos[j] >= t - r) continue;
            if (best < 0 || acc[j] < acc[best] || (acc[j] == acc[best] && pos[j] < pos[best])) best = j;
        }
        if (best < 0) return -1;
        evict[best] = 1;
        --alive;
        ++ne;
    }
    return ne;
}

// Reliability weights of the lookahead trajectories (LORE-KV page, Method, "Reliability
// weights", Eqs. 2-4, 10):
//   per logits row u: lse, H = -sum p log p, log q(y_u) = z_y - lse, c_u = log q(y_u) + H;
//   cbar_m, Hbar_m = means over the T rows of trajectory m; Dhat_m = standardised cosine
//   disagreement of the trajectory's mean lookahead query with the others (all layers and query
//   heads); R_m = beta cbar_m - gamma Hbar_m - lambda_D Dhat_m; omega = softmax(R).
//
// Three kernels: per-row partial statistics (several CTAs per row, streaming the vocabulary once
// with an online max), per-(layer, head) cosine matrices of the trajectory means (only when
// lambda_D != 0), and a per-sequence finaliser that merges everything in a fixed order.
#include "kve_internal.cuh"

namespace kve {

namespace {

struct RowAcc {
    float m, a, b;  // running max, sum exp(z-m), sum exp(z-m)*z
};

__device__ __forceinline__ RowAcc row_merge(RowAcc x, RowAcc y) {
    float m = fmaxf(x.m, y.m);
    if (m == -INFINITY) return x;
    float sx = (x.m == -INFINITY) ? 0.f : expf(x.m - m);
    float sy = (y.m == -INFINITY) ? 0.f : expf(y.m - m);
    return RowAcc{m, x.a * sx + y.a * sy, x.b * sx + y.b * sy};
}

// grid (rel_splits, MT, S), block 256
__global__ void __launch_bounds__(256) rel_rows_kernel(const float *__restrict__ logits, int MT,
                                                       long vocab, int splits,
                                                       float4 *__restrict__ part) {
    const int sp = blockIdx.x, u = blockIdx.y, s = blockIdx.z;
    const float *z = logits + ((size_t)s * MT + u) * vocab;
    const long per = (vocab + splits - 1) / splits;
    const long v0 = (long)sp * per, v1 = min(vocab, v0 + per);
    RowAcc acc{-INFINITY, 0.f, 0.f};
    for (long v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
        float x = __ldg(z + v);
        // a -inf logit (a masked token) has p = 0 and adds nothing to the sums (0 log 0 = 0)
        if (x == -INFINITY) continue;
        if (x > acc.m) {
            float sc = (acc.m == -INFINITY) ? 0.f : expf(acc.m - x);
            acc.a = acc.a * sc + 1.f;
            acc.b = acc.b * sc + x;
            acc.m = x;
        } else {
            float e = expf(x - acc.m);
            acc.a += e;
            acc.b += e * x;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        RowAcc y{__shfl_xor_sync(0xffffffffu, acc.m, o), __shfl_xor_sync(0xffffffffu, acc.a, o),
                 __shfl_xor_sync(0xffffffffu, acc.b, o)};
        acc = row_merge(acc, y);
    }
    __shared__ RowAcc wacc[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) wacc[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        RowAcc t = wacc[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) t = row_merge(t, wacc[w]);
        part[((size_t)s * MT + u) * splits + sp] = make_float4(t.m, t.a, t.b, 0.f);
    }
}

// grid (L*Hq, S), block 128. cosm[s][lh][m][m2] = cos(qbar_m, qbar_m2) of query head lh.
template <typename T>
__global__ void __launch_bounds__(128) rel_cos_kernel(const T *__restrict__ QL, int LH, int M,
                                                      int Tn, int d, float *__restrict__ cosm) {
    extern __shared__ float qbar[];  // [M][d]
    const int lh = blockIdx.x, s = blockIdx.y;
    const T *q = QL + ((size_t)s * LH + lh) * (size_t)M * Tn * d;
    for (int idx = threadIdx.x; idx < M * d; idx += blockDim.x) {
        const int m = idx / d, k = idx % d;
        float acc = 0.f;
        for (int t = 0; t < Tn; ++t) acc += to_f(q[((size_t)m * Tn + t) * d + k]);
        qbar[idx] = acc / (float)Tn;
    }
    __syncthreads();
    for (int pr = threadIdx.x; pr < M * M; pr += blockDim.x) {
        const int m = pr / M, m2 = pr % M;
        float dot = 0.f, na = 0.f, nb = 0.f;
        for (int k = 0; k < d; ++k) {
            const float a = qbar[m * d + k], b = qbar[m2 * d + k];
            dot = fmaf(a, b, dot);
            na = fmaf(a, a, na);
            nb = fmaf(b, b, nb);
        }
        const float cs = (na > 0.f && nb > 0.f) ? dot / (sqrtf(na) * sqrtf(nb)) : 0.f;
        cosm[(((size_t)s * LH + lh) * M + m) * M + m2] = cs;
    }
}

// grid S, block kRelFinalThreads (one thread per logits row; MT <= 64). Fixed-order merges,
// double precision; the disagreement sums over the L*Hq query heads are split over the threads
// (head lh goes to thread lh % kRelFinalThreads) and the partial sums added by a pairwise tree of
// fixed shape.
constexpr int kRelFinalThreads = 256;
__global__ void rel_final_kernel(const float *__restrict__ logits, const int32_t *__restrict__ y,
                                 const float4 *__restrict__ part, const float *__restrict__ cosm,
                                 int M, int Tn, long vocab, int splits, int LH, float beta,
                                 float gamma, float lambda_D, float *__restrict__ omega) {
    __shared__ double c_s[64], h_s[64], R_s[32], red[kRelFinalThreads], dsum[32];
    const int s = blockIdx.x, u = threadIdx.x, MT = M * Tn;
    if (u < MT) {
        const float4 *p = part + ((size_t)s * MT + u) * splits;
        double m = -INFINITY;
        for (int k = 0; k < splits; ++k) m = fmax(m, (double)p[k].x);
        double a = 0.0, b = 0.0;
        for (int k = 0; k < splits; ++k) {
            if (p[k].x == -INFINITY) continue;
            const double sc = exp((double)p[k].x - m);
            a += (double)p[k].y * sc;
            b += (double)p[k].z * sc;
        }
        const double lse = m + log(a);
        const double H = lse - b / a;  // -sum p log p = lse - sum p z
        const int yy = y[(size_t)s * MT + u];
        // an id outside the vocabulary yields NaN weights instead of an out-of-range read
        const double logq = (yy >= 0 && yy < vocab)
                                ? (double)logits[((size_t)s * MT + u) * vocab + yy] - lse
                                : (double)NAN;
        c_s[u] = logq + H;
        h_s[u] = H;
    }
    __syncthreads();
    const bool disagree = lambda_D != 0.f && M > 1;
    if (disagree) {
        for (int mm = 0; mm < M; ++mm) {
            double acc = 0.0;
            for (int lh = u; lh < LH; lh += blockDim.x)
                for (int m2 = 0; m2 < M; ++m2)
                    if (m2 != mm) acc += cosm[(((size_t)s * LH + lh) * M + mm) * M + m2];
            red[u] = acc;
            __syncthreads();
            for (int stride = kRelFinalThreads / 2; stride > 0; stride >>= 1) {
                if (u < stride) red[u] += red[u + stride];
                __syncthreads();
            }
            if (u == 0) dsum[mm] = red[0];
            __syncthreads();
        }
    }
    if (u == 0) {
        double D[32], Dh[32];
        for (int mm = 0; mm < M; ++mm) Dh[mm] = 0.0;
        if (disagree) {
            double mean = 0.0;
            for (int mm = 0; mm < M; ++mm) {
                D[mm] = 1.0 - dsum[mm] / ((double)(M - 1) * LH);
                mean += D[mm];
            }
            mean /= M;
            double var = 0.0;
            for (int mm = 0; mm < M; ++mm) var += (D[mm] - mean) * (D[mm] - mean);
            const double sd = sqrt(var / M);
            for (int mm = 0; mm < M; ++mm) Dh[mm] = (sd < 1e-12) ? 0.0 : (D[mm] - mean) / sd;
        }
        double rmax = -INFINITY;
        for (int mm = 0; mm < M; ++mm) {
            double cb = 0.0, hb = 0.0;
            for (int t = 0; t < Tn; ++t) {
                cb += c_s[mm * Tn + t];
                hb += h_s[mm * Tn + t];
            }
            cb /= Tn;
            hb /= Tn;
            R_s[mm] = (double)beta * cb - (double)gamma * hb - (double)lambda_D * Dh[mm];
            rmax = fmax(rmax, R_s[mm]);
        }
        double zsum = 0.0;
        for (int mm = 0; mm < M; ++mm) zsum += exp(R_s[mm] - rmax);
        for (int mm = 0; mm < M; ++mm) omega[(size_t)s * M + mm] = (float)(exp(R_s[mm] - rmax) / zsum);
    }
}

}  // namespace

cudaError_t launch_reliability(const LorekvDims &D, const void *Q_look, const float *logits,
                               const int32_t *sampled, float *omega_out, void *ws,
                               const LorekvWorkspace &W, cudaStream_t st) {
    char *base = static_cast<char *>(ws);
    float4 *part = reinterpret_cast<float4 *>(base + W.rel_part);
    float *cosm = reinterpret_cast<float *>(base + W.cosm);
    rel_rows_kernel<<<dim3(D.rel_splits, D.MT, D.S), 256, 0, st>>>(logits, D.MT, D.vocab,
                                                                  D.rel_splits, part);
    const int LH = D.L * D.Hq;
    if (D.lambda_D != 0.f && D.M > 1) {
        const size_t smem = sizeof(float) * D.M * D.d;
        if (D.dtype == KVE_F32)
            rel_cos_kernel<float><<<dim3(LH, D.S), 128, smem, st>>>(
                static_cast<const float *>(Q_look), LH, D.M, D.T, D.d, cosm);
        else
            rel_cos_kernel<__nv_bfloat16><<<dim3(LH, D.S), 128, smem, st>>>(
                static_cast<const __nv_bfloat16 *>(Q_look), LH, D.M, D.T, D.d, cosm);
    }
    rel_final_kernel<<<D.S, kRelFinalThreads, 0, st>>>(logits, sampled, part, cosm, D.M, D.T, D.vocab,
                                         D.rel_splits, LH, D.beta, D.gamma, D.lambda_D, omega_out);
    return cudaGetLastError();
}

}  // namespace kve

// LORE-KV scoring on CUDA cores (FP32 FMA). This is the path for fp32 inputs and for shapes the
// tensor-core kernels do not cover; it computes exactly what the tensor-core path computes.
//
// Attention statistics (LORE-KV page, Method: a_{q,i} = softmax_i(q.k_i/sqrt d), o_q =
// sum_i a_{q,i} v_i): each CTA takes 32 queries of one unit and one split of the tokens, with an
// online softmax in the log2 domain; a combine kernel merges the splits.
//
// Per-query prep: u_q = G_h o_q and c_q = o_q^T G_h o_q, so that
//   ||L_h^T (v_i - o_q)||^2 = ||L_h^T v_i||^2 - 2 v_i.u_q + c_q,
// plus the weight of the query in S_i (1/(g w) for window queries, lambda_L omega_m/(g T) for
// the lookahead queries of trajectory m; psi = mean).
//
// Scores (Eqs. 5-7): e_{q,i} = a_{q,i}/(1-a_{q,i}+eps) * sqrt(x_{q,i}), S_i = sum_q weight_q e_{q,i}.
#include "kve_internal.cuh"

namespace kve {

namespace {

constexpr int kQB = 32;  // queries per CTA in the statistics pass
constexpr int kTT = 32;  // tokens per shared-memory tile

template <typename T>
__device__ __forceinline__ const T *query_ptr(const T *QW, const T *QL, const LorekvDims &D,
                                              int unit, int qi) {
    const int kh = unit % D.Hkv;
    const int sl = unit / D.Hkv;  // s*L + l
    const int j = qi / D.nq, r = qi % D.nq;
    const int h = kh * D.g + j;
    if (r < D.w) return QW + (((size_t)sl * D.Hq + h) * D.w + r) * D.d;
    return QL + (((size_t)sl * D.Hq + h) * D.MT + (r - D.w)) * D.d;
}

__device__ __forceinline__ int visible_tokens(const LorekvDims &D, int qi) {
    const int r = qi % D.nq;
    return (r < D.w && D.window_causal) ? D.n - D.w + r + 1 : D.n;
}

// grid (ceil(Qu/32), nsplit, units), block 256 (8 warps x 4 queries). DPL = d/32 dims per lane.
template <typename T, int DPL>
__global__ void __launch_bounds__(256) attn_partial_kernel(const T *__restrict__ K,
                                                           const T *__restrict__ V,
                                                           const T *__restrict__ QW,
                                                           const T *__restrict__ QL, LorekvDims D,
                                                           float2 *__restrict__ part_ml,
                                                           float *__restrict__ part_o,
                                                           float *__restrict__ part_mx) {
    constexpr int d = DPL * 32;
    extern __shared__ float sm[];
    float *qs = sm;                       // [kQB][d]
    float *ks = qs + kQB * d;             // [kTT][d+1]
    float *vs = ks + kTT * (d + 1);       // [kTT][d+1]
    const int qb = blockIdx.x, sp = blockIdx.y, unit = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float qscale = kLog2e * rsqrtf((float)d);
    for (int idx = threadIdx.x; idx < kQB * d; idx += blockDim.x) {
        const int qq = idx / d, k = idx % d;
        const int qi = qb * kQB + qq;
        qs[idx] = (qi < D.Qu) ? to_f(query_ptr(QW, QL, D, unit, qi)[k]) * qscale : 0.f;
    }
    const int t0 = sp * D.split_len, t1 = min(D.n, t0 + D.split_len);
    const T *Ku = K + (size_t)unit * D.n * d;
    const T *Vu = V + (size_t)unit * D.n * d;
    float m[4], l[4], o[4][DPL], mnp[4];  // mnp: largest visible non-protected logit
    int nvis[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        m[a] = -INFINITY;
        mnp[a] = -INFINITY;
        l[a] = 0.f;
        const int qi = qb * kQB + warp * 4 + a;
        nvis[a] = (qi < D.Qu) ? visible_tokens(D, qi) : 0;
#pragma unroll
        for (int c = 0; c < DPL; ++c) o[a][c] = 0.f;
    }
    for (int base = t0; base < t1; base += kTT) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kTT * d; idx += blockDim.x) {
            const int tt = idx / d, k = idx % d;
            const int tok = base + tt;
            ks[tt * (d + 1) + k] = (tok < t1) ? to_f(Ku[(size_t)tok * d + k]) : 0.f;
            vs[tt * (d + 1) + k] = (tok < t1) ? to_f(Vu[(size_t)tok * d + k]) : 0.f;
        }
        __syncthreads();
        const int tok = base + lane;
        const bool np_tok = tok >= D.sink && tok < D.n - D.w;
        // the tile holds sink or window tokens (block-uniform)
        const bool has_prot = base < D.sink || base + kTT > D.n - D.w;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        const float *kr = ks + lane * (d + 1);
        const float *qr = qs + (warp * 4) * d;
        for (int k = 0; k < d; ++k) {
            const float kv = kr[k];
#pragma unroll
            for (int a = 0; a < 4; ++a) s[a] = fmaf(qr[a * d + k], kv, s[a]);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const bool valid = tok < t1 && tok < nvis[a];
            const float sv = valid ? s[a] : -INFINITY;
            const float mt = warp_max(sv);
            mnp[a] = fmaxf(mnp[a], has_prot ? warp_max(np_tok ? sv : -INFINITY) : mt);
            const float mn = fmaxf(m[a], mt);
            if (mn == -INFINITY) continue;  // nothing visible yet
            const float corr = (m[a] == -INFINITY) ? 0.f : exp2f(m[a] - mn);
            const float p = valid ? exp2f(sv - mn) : 0.f;
            l[a] = l[a] * corr + warp_sum(p);
            m[a] = mn;
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[a][c] *= corr;
            for (int t2 = 0; t2 < kTT; ++t2) {
                const float pt = __shfl_sync(0xffffffffu, p, t2);
                const float *vr = vs + t2 * (d + 1);
#pragma unroll
                for (int c = 0; c < DPL; ++c) o[a][c] = fmaf(pt, vr[lane + 32 * c], o[a][c]);
            }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int qi = qb * kQB + warp * 4 + a;
        if (qi >= D.Qu) continue;
        const size_t row = ((size_t)unit * D.nsplit + sp) * D.Qu + qi;
        if (lane == 0) {
            part_ml[row] = make_float2(m[a], l[a]);
            part_mx[row] = mnp[a];
        }
#pragma unroll
        for (int c = 0; c < DPL; ++c) part_o[row * d + lane + 32 * c] = o[a][c];
    }
}

// grid (ceil(Qu/8), units), block 256: one warp per query, 4 dimensions per lane (d = 128) or
// fewer. Merges the token splits of the query.
__global__ void __launch_bounds__(256) combine_kernel(LorekvDims D, const float2 *__restrict__ part_ml,
                                                      const float *__restrict__ part_o,
                                                      const float *__restrict__ part_mx,
                                                      float *__restrict__ lse2,
                                                      float *__restrict__ o,
                                                      float *__restrict__ amax,
                                                      int *__restrict__ pk_cnt,
                                                      float *__restrict__ lse_out,
                                                      float *__restrict__ o_out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qi = blockIdx.x * 8 + warp, unit = blockIdx.y;
    if (qi >= D.Qu) return;
    const size_t base = (size_t)unit * D.nsplit * D.Qu + qi;
    float mx = -INFINITY;
    for (int sp = 0; sp < D.nsplit; ++sp) mx = fmaxf(mx, part_ml[base + (size_t)sp * D.Qu].x);
    const int dpl = D.d / 32;  // dimensions per lane, contiguous
    float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int sp = 0; sp < D.nsplit; ++sp) {
        const float2 ml = part_ml[base + (size_t)sp * D.Qu];
        if (ml.x == -INFINITY) continue;
        const float sc = exp2f(ml.x - mx);
        l = fmaf(ml.y, sc, l);
        const float *src = part_o + (base + (size_t)sp * D.Qu) * D.d + lane * dpl;
        if (dpl == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(src);
            acc[0] = fmaf(v.x, sc, acc[0]);
            acc[1] = fmaf(v.y, sc, acc[1]);
            acc[2] = fmaf(v.z, sc, acc[2]);
            acc[3] = fmaf(v.w, sc, acc[3]);
        } else {
            for (int c = 0; c < dpl; ++c) acc[c] = fmaf(src[c], sc, acc[c]);
        }
    }
    const size_t row = (size_t)unit * D.Qu + qi;
    const float inv = 1.f / l;
    for (int c = 0; c < dpl; ++c) {
        const float ov = acc[c] * inv;
        o[row * D.d + lane * dpl + c] = ov;
        if (o_out) o_out[row * D.d + lane * dpl + c] = ov;
    }
    if (lane == 0) {
        const float v = mx + log2f(l);
        lse2[row] = v;
        if (lse_out) lse_out[row] = v * kLn2;
        // a_max over non-protected tokens: flags the queries whose pairs may be peaked
        float mnp = -INFINITY;
        for (int sp = 0; sp < D.nsplit; ++sp) mnp = fmaxf(mnp, part_mx[base + (size_t)sp * D.Qu]);
        amax[row] = mnp > -1e30f ? exp2f(mnp - v) : 0.f;
        pk_cnt[row] = 0;
    }
}

// grid (g, units), block 256. u_q = G_h o_q, c_q = o_q^T G_h o_q and the query's weight, for the
// nq queries of one query head; bf16 copy of u for the tensor-core path. G_h and the head's o rows
// (transposed: [dimension][query]) are staged in shared memory; a thread computes a 4-query x
// 8-dimension block of U, reading its 4 queries' o values for a dimension as one 16-byte word
// (consecutive threads hold consecutive query groups: no bank conflict).
template <typename T>
__global__ void __launch_bounds__(256) prep_u_kernel(LorekvDims D, const float *__restrict__ G,
                                                     const float *__restrict__ omega,
                                                     const T *__restrict__ QW,
                                                     const T *__restrict__ QL,
                                                     const float *__restrict__ o,
                                                     float *__restrict__ u32,
                                                     float *__restrict__ cq,
                                                     float *__restrict__ wq,
                                                     __nv_bfloat16 *__restrict__ u16,
                                                     __nv_bfloat16 *__restrict__ q16) {
    extern __shared__ float sm[];
    const int d = D.d;
    float *Gs = sm;                 // [d][d]
    float *OsT = sm + d * d;        // [d][nq_pad]: o transposed
    const int j = blockIdx.x, unit = blockIdx.y;
    const int kh = unit % D.Hkv, l = (unit / D.Hkv) % D.L, s = unit / (D.Hkv * D.L);
    const int h = kh * D.g + j;
    const float *Gh = G + ((size_t)l * D.Hq + h) * d * d;
    const size_t row0 = (size_t)unit * D.Qu + (size_t)j * D.nq;
    const int nq_pad = (D.nq + 3) & ~3;
    {
        const float4 *g4 = reinterpret_cast<const float4 *>(Gh);
        float4 *s4 = reinterpret_cast<float4 *>(Gs);
#pragma unroll 4
        for (int idx = threadIdx.x; idx < d * d / 4; idx += blockDim.x) s4[idx] = g4[idx];
        // query fastest, so that the transposed stores of a warp hit consecutive words
        const float4 *o4 = reinterpret_cast<const float4 *>(o + row0 * d);
        for (int idx = threadIdx.x; idx < nq_pad * d / 4; idx += blockDim.x) {
            const int q = idx % nq_pad, k4 = idx / nq_pad;
            const float4 v = q < D.nq ? o4[(size_t)q * (d / 4) + k4] : make_float4(0.f, 0.f, 0.f, 0.f);
            OsT[(4 * k4 + 0) * nq_pad + q] = v.x;
            OsT[(4 * k4 + 1) * nq_pad + q] = v.y;
            OsT[(4 * k4 + 2) * nq_pad + q] = v.z;
            OsT[(4 * k4 + 3) * nq_pad + q] = v.w;
        }
    }
    __syncthreads();
    // gsz threads share 4 queries; thread jb takes dimensions 4 jb .. 4 jb + 3 and d/2 + 4 jb ..
    // d/2 + 4 jb + 3, so that each 16-byte G load of the group covers consecutive words (no bank
    // conflict)
    const int gsz = d / 8;
    const int jb = threadIdx.x % gsz, qg = threadIdx.x / gsz;
    const int c0 = 4 * jb, c1 = d / 2 + 4 * jb;
    const int qstep = blockDim.x / gsz;
    for (int base = 0; base < nq_pad; base += qstep * 4) {  // uniform trip count: shuffles below
        const bool active = base + qg * 4 < nq_pad;
        const int q0 = active ? base + qg * 4 : 0;
        float acc[4][8];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
        for (int k = 0; k < d; ++k) {
            const float4 g0 = *reinterpret_cast<const float4 *>(Gs + k * d + c0);
            const float4 g1 = *reinterpret_cast<const float4 *>(Gs + k * d + c1);
            const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const float4 o4k = *reinterpret_cast<const float4 *>(OsT + k * nq_pad + q0);
            const float ov[4] = {o4k.x, o4k.y, o4k.z, o4k.w};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(gv[b], ov[a], acc[a][b]);  // G symmetric
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int r = q0 + a;
            float cpart = 0.f;
            if (r < D.nq) {  // o_q . u_q over this thread's 8 dimensions (o from global: L2)
                const float *orow = o + (row0 + r) * d;
                const float4 x0 = *reinterpret_cast<const float4 *>(orow + c0);
                const float4 x1 = *reinterpret_cast<const float4 *>(orow + c1);
                const float ox[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int b = 0; b < 8; ++b) cpart = fmaf(ox[b], acc[a][b], cpart);
            }
            for (int off = gsz / 2; off > 0; off >>= 1)
                cpart += __shfl_xor_sync(0xffffffffu, cpart, off);
            if (active && r < D.nq) {
                const size_t row = row0 + r;
#pragma unroll
                for (int b = 0; b < 8; ++b) u32[row * d + (b < 4 ? c0 + b : c1 + b - 4)] = acc[a][b];
                if (u16)  // -2 u_q (exact scaling of the rounded u_q): B operand of X = -2 V U^T
#pragma unroll
                    for (int b = 0; b < 8; ++b)
                        u16[row * d + (b < 4 ? c0 + b : c1 + b - 4)] =
                            __float2bfloat16_rn(-2.f * acc[a][b]);
                if (jb == 0) cq[row] = cpart;
            }
        }
    }
    for (int r = threadIdx.x; r < D.nq; r += blockDim.x) {
        const size_t row = row0 + r;
        float wt;
        if (r < D.w)
            wt = 1.f / (float)(D.g * D.w);
        else
            wt = D.lambda_L * omega[(size_t)s * D.M + (r - D.w) / D.T] / (float)(D.g * D.T);
        wq[row] = wt;
        if (q16) {
            const T *qp = query_ptr(QW, QL, D, unit, j * D.nq + r);
            for (int k = 0; k < d; ++k) q16[row * d + k] = __float2bfloat16_rn(to_f(qp[k]));
        }
    }
}

// grid (ceil(n/32), units), block 256. Lane = token of the tile, warp = a subset of the queries.
template <typename T, int DPL>
__global__ void __launch_bounds__(256) scores_simt_kernel(
    const T *__restrict__ K, const T *__restrict__ V, const T *__restrict__ QW,
    const T *__restrict__ QL, const float *__restrict__ Lf, LorekvDims D,
    const float *__restrict__ lse2, const float *__restrict__ u32, const float *__restrict__ cq,
    const float *__restrict__ wq, float *__restrict__ scores, int *__restrict__ pk_cnt,
    int *__restrict__ pk_tok) {
    constexpr int d = DPL * 32;
    extern __shared__ float sm[];
    float *ks = sm;                        // [kTT][d+1]
    float *vs = ks + kTT * (d + 1);        // [kTT][d+1]
    float *qs = vs + kTT * (d + 1);        // [nq][d] pre-scaled by log2e/sqrt(d)
    float *us = qs + D.nq * d;             // [nq][d]
    float *ls = us + D.nq * d;             // [d][d]
    float *qc = ls + d * d;                // [3][nq]: lse2, c, weight
    float *red = qc + 3 * D.nq;            // [8][32]
    const int tile = blockIdx.x, unit = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = tile * kTT;
    const int tok = i0 + lane;
    const bool scored = tok >= D.sink && tok < D.n - D.w;
    float *Su = scores + (size_t)unit * D.n;
    if (i0 + kTT <= D.sink || i0 >= D.n - D.w) {  // the whole tile is protected
        if (threadIdx.x < kTT && tok < D.n) Su[tok] = 0.f;
        return;
    }
    const T *Ku = K + (size_t)unit * D.n * d;
    const T *Vu = V + (size_t)unit * D.n * d;
    for (int idx = threadIdx.x; idx < kTT * d; idx += blockDim.x) {
        const int tt = idx / d, k = idx % d;
        const int t = i0 + tt;
        ks[tt * (d + 1) + k] = (t < D.n) ? to_f(Ku[(size_t)t * d + k]) : 0.f;
        vs[tt * (d + 1) + k] = (t < D.n) ? to_f(Vu[(size_t)t * d + k]) : 0.f;
    }
    const int kh = unit % D.Hkv, l = (unit / D.Hkv) % D.L;
    const float qscale = kLog2e * rsqrtf((float)d);
    float Sacc = 0.f;
    for (int j = 0; j < D.g; ++j) {
        __syncthreads();
        const int h = kh * D.g + j;
        for (int idx = threadIdx.x; idx < D.nq * d; idx += blockDim.x) {
            const int r = idx / d, k = idx % d;
            const int qi = j * D.nq + r;
            qs[idx] = to_f(query_ptr(QW, QL, D, unit, qi)[k]) * qscale;
            us[idx] = u32[((size_t)unit * D.Qu + qi) * d + k];
        }
        const float *Lh = Lf + ((size_t)l * D.Hq + h) * d * d;
        for (int idx = threadIdx.x; idx < d * d; idx += blockDim.x) ls[idx] = Lh[idx];
        for (int r = threadIdx.x; r < D.nq; r += blockDim.x) {
            const size_t row = (size_t)unit * D.Qu + j * D.nq + r;
            qc[r] = lse2[row];
            qc[D.nq + r] = cq[row];
            qc[2 * D.nq + r] = wq[row];
        }
        __syncthreads();
        // ||L_h^T v||^2: warp w owns output dims jj = w, w+8, ...
        const float *vr = vs + lane * (d + 1);
        const float *kr = ks + lane * (d + 1);
        float nvp = 0.f;
        for (int jj = warp; jj < d; jj += 8) {
            float y = 0.f;
            for (int k = jj; k < d; ++k) y = fmaf(ls[k * d + jj], vr[k], y);  // L lower triangular
            nvp = fmaf(y, y, nvp);
        }
        red[warp * 32 + lane] = nvp;
        __syncthreads();
        float nv = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) nv += red[w * 32 + lane];
        for (int r = warp; r < D.nq; r += 8) {
            const float *qr = qs + r * d;
            const float *ur = us + r * d;
            float s = 0.f, vu = 0.f;
            for (int k = 0; k < d; ++k) {
                s = fmaf(qr[k], kr[k], s);
                vu = fmaf(ur[k], vr[k], vu);
            }
            float a = exp2f(s - qc[r]);
            if (scored && a > kPeakTau) {  // peaked pair: left out here, evaluated exactly later
                const size_t row = (size_t)unit * D.Qu + j * D.nq + r;
                const int slot = atomicAdd(pk_cnt + row, 1);
                if (slot < kPeakSlots) {
                    pk_tok[row * kPeakSlots + slot] = tok;
                    a = 0.f;
                }
            }
            const float x = fmaxf(fmaf(-2.f, vu, nv + qc[D.nq + r]), 0.f);
            const float e = a / (1.f - a + D.eps) * sqrtf(x);
            Sacc = fmaf(qc[2 * D.nq + r], e, Sacc);
        }
    }
    __syncthreads();
    red[warp * 32 + lane] = Sacc;
    __syncthreads();
    if (threadIdx.x < kTT && tok < D.n) {
        float S = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) S += red[w * 32 + threadIdx.x];
        Su[tok] = scored ? S : 0.f;
    }
}

template <typename T>
cudaError_t attn_dispatch(const LorekvDims &D, const void *K, const void *V, const void *QW,
                          const void *QL, float2 *ml, float *po, float *mx, cudaStream_t st) {
    const dim3 grid((D.Qu + kQB - 1) / kQB, D.nsplit, D.units);
    const size_t smem = sizeof(float) * (kQB * D.d + 2 * kTT * (D.d + 1));
#define KVE_ATTN_CASE(DPL)                                                                     \
    case DPL: {                                                                                \
        auto kern = attn_partial_kernel<T, DPL>;                                               \
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);    \
        kern<<<grid, 256, smem, st>>>((const T *)K, (const T *)V, (const T *)QW, (const T *)QL, \
                                      D, ml, po, mx);                                          \
        break;                                                                                 \
    }
    switch (D.d / 32) {
        KVE_ATTN_CASE(1)
        KVE_ATTN_CASE(2)
        KVE_ATTN_CASE(4)
        default: return cudaErrorInvalidValue;
    }
#undef KVE_ATTN_CASE
    return cudaGetLastError();
}

template <typename T>
cudaError_t scores_dispatch(const LorekvDims &D, const void *K, const void *V, const void *QW,
                            const void *QL, const float *Lf, const float *lse2, const float *u32,
                            const float *cq, const float *wq, float *scores, int *pk_cnt,
                            int *pk_tok, cudaStream_t st) {
    const dim3 grid((D.n + kTT - 1) / kTT, D.units);
    const size_t smem = sizeof(float) * (2 * kTT * (D.d + 1) + 2 * D.nq * D.d + D.d * D.d +
                                         3 * D.nq + 8 * 32);
#define KVE_SC_CASE(DPL)                                                                        \
    case DPL: {                                                                                 \
        auto kern = scores_simt_kernel<T, DPL>;                                                 \
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
        kern<<<grid, 256, smem, st>>>((const T *)K, (const T *)V, (const T *)QW, (const T *)QL, \
                                      Lf, D, lse2, u32, cq, wq, scores, pk_cnt, pk_tok);        \
        break;                                                                                  \
    }
    switch (D.d / 32) {
        KVE_SC_CASE(1)
        KVE_SC_CASE(2)
        KVE_SC_CASE(4)
        default: return cudaErrorInvalidValue;
    }
#undef KVE_SC_CASE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_simt(const LorekvDims &D, const void *K, const void *V,
                                  const void *QW, const void *QL, void *ws,
                                  const LorekvWorkspace &W, cudaStream_t st) {
    char *b = static_cast<char *>(ws);
    float2 *ml = reinterpret_cast<float2 *>(b + W.part_ml);
    float *po = reinterpret_cast<float *>(b + W.part_o);
    float *mx = reinterpret_cast<float *>(b + W.part_mx);
    if (D.dtype == KVE_F32) return attn_dispatch<float>(D, K, V, QW, QL, ml, po, mx, st);
    return attn_dispatch<__nv_bfloat16>(D, K, V, QW, QL, ml, po, mx, st);
}

cudaError_t launch_combine(const LorekvDims &D, void *ws, const LorekvWorkspace &W,
                           float *lse_out, float *o_out, cudaStream_t st) {
    char *b = static_cast<char *>(ws);
    combine_kernel<<<dim3((D.Qu + 7) / 8, D.units), 256, 0, st>>>(
        D, reinterpret_cast<const float2 *>(b + W.part_ml),
        reinterpret_cast<const float *>(b + W.part_o),
        reinterpret_cast<const float *>(b + W.part_mx), reinterpret_cast<float *>(b + W.lse2),
        reinterpret_cast<float *>(b + W.o), reinterpret_cast<float *>(b + W.amax),
        reinterpret_cast<int *>(b + W.pk_cnt), lse_out, o_out);
    return cudaGetLastError();
}

cudaError_t launch_prep_u(const LorekvDims &D, const float *G, const float *omega, void *ws,
                          const LorekvWorkspace &W, cudaStream_t st, const void *QW,
                          const void *QL, bool want_bf16);

cudaError_t launch_prep_u(const LorekvDims &D, const float *G, const float *omega, void *ws,
                          const LorekvWorkspace &W, cudaStream_t st) {
    return launch_prep_u(D, G, omega, ws, W, st, nullptr, nullptr, false);
}

cudaError_t launch_prep_u(const LorekvDims &D, const float *G, const float *omega, void *ws,
                          const LorekvWorkspace &W, cudaStream_t st, const void *QW,
                          const void *QL, bool want_bf16) {
    char *b = static_cast<char *>(ws);
    const size_t smem = sizeof(float) * (D.d * D.d + (size_t)((D.nq + 3) & ~3) * D.d);
    __nv_bfloat16 *u16 = want_bf16 ? reinterpret_cast<__nv_bfloat16 *>(b + W.u16) : nullptr;
    __nv_bfloat16 *q16 = nullptr;  // the tensor-core path packs the queries itself
    const float *o = reinterpret_cast<const float *>(b + W.o);
    float *u32 = reinterpret_cast<float *>(b + W.u32);
    float *cq = reinterpret_cast<float *>(b + W.cq);
    float *wq = reinterpret_cast<float *>(b + W.wq);
    if (D.dtype == KVE_F32) {
        auto kern = prep_u_kernel<float>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<dim3(D.g, D.units), 256, smem, st>>>(D, G, omega, (const float *)QW,
                                                    (const float *)QL, o, u32, cq, wq, u16, q16);
    } else {
        auto kern = prep_u_kernel<__nv_bfloat16>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<dim3(D.g, D.units), 256, smem, st>>>(D, G, omega, (const __nv_bfloat16 *)QW,
                                                    (const __nv_bfloat16 *)QL, o, u32, cq, wq,
                                                    u16, q16);
    }
    return cudaGetLastError();
}

cudaError_t launch_scores_simt(const LorekvDims &D, const void *K, const void *V,
                               const void *QW, const void *QL, const float *Lf, void *ws,
                               const LorekvWorkspace &W, float *scores, cudaStream_t st) {
    char *b = static_cast<char *>(ws);
    const float *lse2 = reinterpret_cast<const float *>(b + W.lse2);
    const float *u32 = reinterpret_cast<const float *>(b + W.u32);
    const float *cq = reinterpret_cast<const float *>(b + W.cq);
    const float *wq = reinterpret_cast<const float *>(b + W.wq);
    int *pk_cnt = reinterpret_cast<int *>(b + W.pk_cnt);
    int *pk_tok = reinterpret_cast<int *>(b + W.pk_tok);
    if (D.dtype == KVE_F32)
        return scores_dispatch<float>(D, K, V, QW, QL, Lf, lse2, u32, cq, wq, scores, pk_cnt,
                                      pk_tok, st);
    return scores_dispatch<__nv_bfloat16>(D, K, V, QW, QL, Lf, lse2, u32, cq, wq, scores, pk_cnt,
                                          pk_tok, st);
}

}  // namespace kve

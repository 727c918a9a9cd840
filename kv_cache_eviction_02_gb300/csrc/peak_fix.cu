// Exact projected deletion scores of peaked pairs (LORE-KV page, Method, "Projected deletion
// score", Eqs. 5-7): e_{q,i} = a_{q,i}/(1 - a_{q,i} + eps) ||L_h^T (v_i - o_q)|| for the pairs the
// scoring kernels left out because a_{q,i} > 1/4.
//
// Near a = 1 every shortcut of the scoring pass loses the result: 1 - a is a difference of two
// numbers close to 1, o_q is close to v_i so that the expanded ||L^T v||^2 - 2 v.(G o) + o^T G o
// cancels, and the bf16 rounding of a_{q,i} inside o_q is of the size of v_i - o_q itself. Here
// each recorded query is evaluated again over its visible tokens with the recorded tokens B held
// apart. With r_j = exp(s_j - s_ref):
//   R_i = sum_{j != i} r_j = W + sum_{b in B, b != i} r_b,   W = sum_{j not in B} r_j,
//   a_i = r_i / (r_i + R_i),  1 - a_i = R_i / (r_i + R_i),
//   v_i - o_q = (R_i v_i - sum_{j != i} r_j v_j) / (r_i + R_i)
//            = (W v_i - O + sum_{b != i} r_b (v_i - v_b)) / (r_i + R_i),   O = sum_{j not in B} r_j v_j,
// so neither 1 - a nor v_i - o_q is formed as a difference of nearly equal numbers, and the norm
// is taken of L_h^T (v_i - o_q) directly (the difference form of Eqs. 5-7). fp32 inputs
// accumulate in fp64; bf16 inputs in fp32 (per-lane partial sums, then a warp tree).
//
// peak_apply_kernel then adds w_q e_{q,i} to S_i for every recorded pair, one unit per warp,
// queries in index order and the tokens of a query ascending, so the result does not depend on
// the order in which the scoring kernels recorded the pairs.
#include "kve_internal.cuh"

namespace kve {

namespace {

constexpr int kFixQ = 8;    // queries (warps) per CTA
constexpr int kFixTT = 32;  // tokens per shared-memory tile

template <typename T>
__device__ __forceinline__ const T *fix_query_ptr(const T *QW, const T *QL, const LorekvDims &D,
                                                  int unit, int qi) {
    const int kh = unit % D.Hkv, sl = unit / D.Hkv;
    const int j = qi / D.nq, r = qi % D.nq;
    const int h = kh * D.g + j;
    if (r < D.w) return QW + (((size_t)sl * D.Hq + h) * D.w + r) * D.d;
    return QL + (((size_t)sl * D.Hq + h) * D.MT + (r - D.w)) * D.d;
}

template <typename Acc> __device__ __forceinline__ Acc acc_exp(Acc x);
template <> __device__ __forceinline__ float acc_exp<float>(float x) { return expf(x); }
template <> __device__ __forceinline__ double acc_exp<double>(double x) { return exp(x); }

template <typename Acc> __device__ __forceinline__ Acc warp_sum_acc(Acc v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// grid (ceil(Qu / kFixQ), units), block 32 kFixQ: warp w takes query blockIdx.x kFixQ + w. A CTA
// none of whose queries recorded a pair returns at once.
template <typename T, typename Acc, int DPL>
__global__ void __launch_bounds__(32 * kFixQ) peak_fix_kernel(
    const T *__restrict__ K, const T *__restrict__ V, const T *__restrict__ QW,
    const T *__restrict__ QL, const float *__restrict__ Lf, LorekvDims D,
    const int *__restrict__ pk_cnt, int *__restrict__ pk_tok, float *__restrict__ pk_e,
    const float *__restrict__ wq) {
    constexpr int d = DPL * 32;
    extern __shared__ __align__(16) unsigned char fix_smem[];
    float *ks = reinterpret_cast<float *>(fix_smem);      // [kFixTT][d + 1]
    float *vs = ks + kFixTT * (d + 1);                     // [kFixTT][d + 1]
    float *qs = vs + kFixTT * (d + 1);                     // [kFixQ][d]
    Acc *df = reinterpret_cast<Acc *>(qs + kFixQ * d);     // [kFixQ][d]: v_i - o_q
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.y, qi = blockIdx.x * kFixQ + warp;
    const size_t row = (size_t)unit * D.Qu + qi;
    int cnt = 0;
    if (qi < D.Qu) cnt = min(pk_cnt[row], kPeakSlots);
    if (!__syncthreads_or(cnt > 0)) return;

    // the recorded tokens of this query, ascending (lane b holds token b)
    int tb = 0x7fffffff;
    if (cnt > 0) {
        if (lane < cnt) tb = pk_tok[row * kPeakSlots + lane];
        // rank sort of at most kPeakSlots distinct tokens: lane r takes the r-th smallest
        int rank = 0;
        for (int b = 0; b < cnt; ++b) {
            const int o = __shfl_sync(0xffffffffu, tb, b);
            rank += (o < tb) ? 1 : 0;
        }
        int mine = 0x7fffffff;
        for (int b = 0; b < cnt; ++b) {
            const int o = __shfl_sync(0xffffffffu, tb, b);
            const int rb = __shfl_sync(0xffffffffu, rank, b);
            if (rb == lane) mine = o;
        }
        tb = mine;
        if (lane < cnt) pk_tok[row * kPeakSlots + lane] = tb;
    }
    const T *Ku = K + (size_t)unit * D.n * d;
    const T *Vu = V + (size_t)unit * D.n * d;
    int tok_b[kPeakSlots];
#pragma unroll
    for (int b = 0; b < kPeakSlots; ++b) tok_b[b] = __shfl_sync(0xffffffffu, tb, b);
    const Acc scale = Acc(1) / sqrt(Acc(d));
    Acc s_b[kPeakSlots], vb[kPeakSlots][DPL];
    Acc s_ref = Acc(0);
    int nvis = D.n;
    if (cnt > 0) {
        const T *q = fix_query_ptr(QW, QL, D, unit, qi);
        for (int k = lane; k < d; k += 32) qs[warp * d + k] = to_f(q[k]);
        __syncwarp();
        const int r = qi % D.nq;
        nvis = (r < D.w && D.window_causal) ? D.n - D.w + r + 1 : D.n;
#pragma unroll
        for (int b = 0; b < kPeakSlots; ++b) {
            s_b[b] = Acc(0);
#pragma unroll
            for (int c = 0; c < DPL; ++c) vb[b][c] = Acc(0);
            if (b < cnt) {
                Acc part = Acc(0);
#pragma unroll
                for (int c = 0; c < DPL; ++c) {
                    const int k = lane + 32 * c;
                    part += (Acc)qs[warp * d + k] * (Acc)to_f(Ku[(size_t)tok_b[b] * d + k]);
                    vb[b][c] = (Acc)to_f(Vu[(size_t)tok_b[b] * d + k]);
                }
                s_b[b] = warp_sum_acc(part) * scale;
            }
        }
        s_ref = s_b[0];
        for (int b = 1; b < cnt; ++b) s_ref = s_b[b] > s_ref ? s_b[b] : s_ref;
    }

    // W = sum r_j and O = sum r_j v_j over the visible tokens outside B
    Acc Wl = Acc(0), O[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) O[c] = Acc(0);
    for (int base = 0; base < D.n; base += kFixTT) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kFixTT * d; idx += blockDim.x) {
            const int tt = idx / d, k = idx % d;
            const int t = base + tt;
            ks[tt * (d + 1) + k] = t < D.n ? to_f(Ku[(size_t)t * d + k]) : 0.f;
            vs[tt * (d + 1) + k] = t < D.n ? to_f(Vu[(size_t)t * d + k]) : 0.f;
        }
        __syncthreads();
        if (cnt == 0 || base >= nvis) continue;
        const int t = base + lane;
        bool in_b = false;
#pragma unroll
        for (int b = 0; b < kPeakSlots; ++b) in_b |= (b < cnt && t == tok_b[b]);
        Acc sdot = Acc(0);
        const float *kr = ks + lane * (d + 1);
        const float *qr = qs + warp * d;
        for (int k = 0; k < d; ++k) sdot += (Acc)qr[k] * (Acc)kr[k];
        const Acc rj = (t < nvis && !in_b) ? acc_exp<Acc>(sdot * scale - s_ref) : Acc(0);
        Wl += rj;
        for (int t2 = 0; t2 < kFixTT; ++t2) {
            const Acc rt = __shfl_sync(0xffffffffu, rj, t2);
            const float *vr = vs + t2 * (d + 1);
#pragma unroll
            for (int c = 0; c < DPL; ++c) O[c] += rt * (Acc)vr[lane + 32 * c];
        }
    }
    if (cnt == 0) return;  // after the last block-wide barrier
    const Acc W = warp_sum_acc(Wl);
    const int l = (unit / D.Hkv) % D.L, kh = unit % D.Hkv;
    const int h = kh * D.g + qi / D.nq;
    const float *Lh = Lf + ((size_t)l * D.Hq + h) * d * d;
    Acc r_b[kPeakSlots];
#pragma unroll
    for (int b = 0; b < kPeakSlots; ++b) r_b[b] = b < cnt ? acc_exp<Acc>(s_b[b] - s_ref) : Acc(0);
    const float w = wq[row];
    for (int i = 0; i < cnt; ++i) {
        Acc rest = W;
#pragma unroll
        for (int b = 0; b < kPeakSlots; ++b)
            if (b != i) rest += r_b[b];
        Acc ri = Acc(0);
#pragma unroll
        for (int b = 0; b < kPeakSlots; ++b)
            if (b == i) ri = r_b[b];
        const Acc tot = ri + rest;
        // v_i - o_q for this lane's dimensions
#pragma unroll
        for (int c = 0; c < DPL; ++c) {
            Acc vi = Acc(0);
#pragma unroll
            for (int b = 0; b < kPeakSlots; ++b)
                if (b == i) vi = vb[b][c];
            Acc dsum = W * vi - O[c];
#pragma unroll
            for (int b = 0; b < kPeakSlots; ++b)
                if (b != i) dsum += r_b[b] * (vi - vb[b][c]);
            df[warp * d + lane + 32 * c] = dsum / tot;
        }
        __syncwarp();
        // ||L_h^T (v_i - o_q)||^2: lane owns output columns lane + 32 c; L_h[k][c] = 0 for k < c
        Acc y[DPL];
#pragma unroll
        for (int c = 0; c < DPL; ++c) y[c] = Acc(0);
        for (int k = 0; k < d; ++k) {
            const Acc dk = df[warp * d + k];
#pragma unroll
            for (int c = 0; c < DPL; ++c) y[c] += (Acc)Lh[(size_t)k * d + lane + 32 * c] * dk;
        }
        Acc nrm2 = Acc(0);
#pragma unroll
        for (int c = 0; c < DPL; ++c) nrm2 += y[c] * y[c];
        nrm2 = warp_sum_acc(nrm2);
        const Acc a = ri / tot, oma = rest / tot;
        const Acc e = a / (oma + (Acc)D.eps) * sqrt(nrm2);
        if (lane == 0) pk_e[row * kPeakSlots + i] = (float)((Acc)w * e);
        __syncwarp();
    }
}

// grid units, block 32: S_i += w_q e_{q,i} for every recorded pair of the unit, queries in index
// order, tokens of a query ascending (a fixed order: the result is deterministic).
__global__ void peak_apply_kernel(LorekvDims D, const int *__restrict__ pk_cnt,
                                  const int *__restrict__ pk_tok, const float *__restrict__ pk_e,
                                  float *__restrict__ scores) {
    const int unit = blockIdx.x, lane = threadIdx.x;
    float *Su = scores + (size_t)unit * D.n;
    for (int base = 0; base < D.Qu; base += 32) {
        const int qi = base + lane;
        const size_t row = (size_t)unit * D.Qu + qi;
        const int c = qi < D.Qu ? min(pk_cnt[row], kPeakSlots) : 0;
        unsigned mask = __ballot_sync(0xffffffffu, c > 0);
        while (mask) {
            const int src = __ffs(mask) - 1;
            mask &= mask - 1;
            const int cs = __shfl_sync(0xffffffffu, c, src);
            if (lane == 0) {
                const size_t r = (size_t)unit * D.Qu + base + src;
                for (int b = 0; b < cs; ++b)
                    Su[pk_tok[r * kPeakSlots + b]] += pk_e[r * kPeakSlots + b];
            }
        }
    }
}

template <typename T, typename Acc>
cudaError_t fix_dispatch(const LorekvDims &D, const void *K, const void *V, const void *QW,
                         const void *QL, const float *Lf, const int *cnt, int *tok, float *e,
                         const float *wq, cudaStream_t st) {
    const dim3 grid((D.Qu + kFixQ - 1) / kFixQ, D.units);
    const size_t smem = sizeof(float) * (2 * kFixTT * (D.d + 1) + kFixQ * D.d) +
                        sizeof(Acc) * kFixQ * D.d;
#define KVE_FIX_CASE(DPL)                                                                        \
    case DPL: {                                                                                  \
        auto kern = peak_fix_kernel<T, Acc, DPL>;                                                \
        cudaError_t ae =                                                                         \
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);  \
        if (ae != cudaSuccess) return ae;                                                        \
        kern<<<grid, 32 * kFixQ, smem, st>>>((const T *)K, (const T *)V, (const T *)QW,          \
                                             (const T *)QL, Lf, D, cnt, tok, e, wq);             \
        break;                                                                                   \
    }
    switch (D.d / 32) {
        KVE_FIX_CASE(1)
        KVE_FIX_CASE(2)
        KVE_FIX_CASE(4)
        default: return cudaErrorInvalidValue;
    }
#undef KVE_FIX_CASE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_peak_fix(const LorekvDims &D, const void *K, const void *V, const void *QW,
                            const void *QL, const float *Lf, void *ws, const LorekvWorkspace &W,
                            float *scores, cudaStream_t st) {
    char *b = static_cast<char *>(ws);
    const int *cnt = reinterpret_cast<const int *>(b + W.pk_cnt);
    int *tok = reinterpret_cast<int *>(b + W.pk_tok);
    float *e = reinterpret_cast<float *>(b + W.pk_e);
    const float *wq = reinterpret_cast<const float *>(b + W.wq);
    cudaError_t err = D.dtype == KVE_F32
                          ? fix_dispatch<float, double>(D, K, V, QW, QL, Lf, cnt, tok, e, wq, st)
                          : fix_dispatch<__nv_bfloat16, float>(D, K, V, QW, QL, Lf, cnt, tok, e,
                                                               wq, st);
    if (err != cudaSuccess) return err;
    peak_apply_kernel<<<D.units, 32, 0, st>>>(D, cnt, tok, e, scores);
    return cudaGetLastError();
}

}  // namespace kve

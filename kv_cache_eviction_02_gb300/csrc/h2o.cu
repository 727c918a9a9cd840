// H2O heavy-hitter + recent-window eviction (paper summary "H2O: Heavy-Hitter Oracle ...").
//
// State per (batch, layer, head) unit: `cap` preallocated slots of K and V, the accumulated
// attention score and the position of the token each slot holds (Appendix A: preallocated memory;
// an evicted slot is overwritten in place by the next token, nothing moves). Slots 0..nslots-1
// are in use except `hole`, the slot freed by the last eviction, which the next append fills.
// The recent window is the r_t most recent positions (positions >= t - r_t); it is recomputed from
// the positions each step instead of being kept as a separate circular queue.
//
// Decode step (Section 4.1, Algorithm 1 with linear h; Section 2.1 / Definition 2.2 for attention
// over the retained set; Definition 2.1 for at most one eviction per step): one warp per unit.
// The unit's K/V rows are streamed twice (scores, then the weighted sum of V) with 16-byte loads;
// the work is bound by HBM bandwidth.
#include "kve_internal.cuh"

namespace kve {

namespace {

template <typename T> struct Vec8;  // 8 elements = 16 bytes
template <> struct Vec8<__half> {
    static __device__ __forceinline__ void load(const __half *p, float *f) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __half22float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    static __device__ __forceinline__ void store(__half *p, const float *f) {
        uint4 u;
        __half2 *h = reinterpret_cast<__half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        *reinterpret_cast<uint4 *>(p) = u;
    }
};
template <> struct Vec8<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float *f) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float *f) {
        uint4 u;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        *reinterpret_cast<uint4 *>(p) = u;
    }
};

constexpr int kPrefThreads = 256;

// ---- prefill, CUDA-core column sums ---------------------------------------------------------------
// acc_j = sum_{i >= j} softmax_i(q_i . K_{<=i} / sqrt d)_j over the prompt (H2O summary, Section 4.1,
// prompt handled as one block). grid units, block 256. Shared: Kt [d][P] (transposed keys, input
// type), colsum [8][P] f32, qst [8][4][d] f32. Writes acc_out [unit][P].
template <typename T>
__global__ void __launch_bounds__(kPrefThreads) h2o_colsum_kernel(
    const T *__restrict__ K, const T *__restrict__ Q, int P, int d, float *__restrict__ acc_out) {
    extern __shared__ __align__(16) unsigned char smraw[];
    T *Kt = reinterpret_cast<T *>(smraw);                                  // [d][P]
    float *colsum = reinterpret_cast<float *>(smraw + sizeof(T) * d * P);  // [8][P]
    float *qst = colsum + 8 * P;                                           // [8][4][d]
    const int unit = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T *Ku = K + (size_t)unit * P * d;
    const T *Qu = Q + (size_t)unit * P * d;
    for (int e = threadIdx.x; e < P * d; e += blockDim.x) {
        const int j = e / d, k = e % d;
        Kt[k * P + j] = Ku[e];
    }
    for (int e = threadIdx.x; e < 8 * P; e += blockDim.x) colsum[e] = 0.f;
    __syncthreads();
    const float qscale = kLog2e * rsqrtf((float)d);
    float *qw = qst + warp * 4 * d;
    float *cs = colsum + warp * P;
    const int ngroups = (P + 3) / 4;
    for (int grp = warp; grp < ngroups; grp += 8) {
        const int i0 = grp * 4;
        __syncwarp();
        for (int e = lane; e < 4 * d; e += 32) {
            const int a = e / d, k = e % d;
            qw[e] = (i0 + a < P) ? to_f(Qu[(size_t)(i0 + a) * d + k]) * qscale : 0.f;
        }
        __syncwarp();
        const int jmax = min(P - 1, i0 + 3);
        float m[4], l[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            m[a] = -INFINITY;
            l[a] = 0.f;
        }
        // pass 1: row max and normaliser (online per lane, then warp merge)
        for (int jb = 0; jb <= jmax; jb += 32) {
            const int j = jb + lane;
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            if (j <= jmax)
                for (int k = 0; k < d; ++k) {
                    const float kv = to_f(Kt[k * P + j]);
#pragma unroll
                    for (int a = 0; a < 4; ++a) s[a] = fmaf(qw[a * d + k], kv, s[a]);
                }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                if (j <= i0 + a && i0 + a < P) {
                    if (s[a] > m[a]) {
                        l[a] = l[a] * exp2f(m[a] - s[a]) + 1.f;
                        m[a] = s[a];
                    } else {
                        l[a] += exp2f(s[a] - m[a]);
                    }
                }
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float mw = warp_max(m[a]);
            const float lw = warp_sum((m[a] == -INFINITY) ? 0.f : l[a] * exp2f(m[a] - mw));
            m[a] = mw;
            l[a] = 1.f / lw;
        }
        // pass 2: p_ij = exp2(s - m) / l added to this warp's column sums
        for (int jb = 0; jb <= jmax; jb += 32) {
            const int j = jb + lane;
            if (j > jmax) continue;
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k = 0; k < d; ++k) {
                const float kv = to_f(Kt[k * P + j]);
#pragma unroll
                for (int a = 0; a < 4; ++a) s[a] = fmaf(qw[a * d + k], kv, s[a]);
            }
            float add = 0.f;
#pragma unroll
            for (int a = 0; a < 4; ++a)
                if (j <= i0 + a && i0 + a < P) add += exp2f(s[a] - m[a]) * l[a];
            cs[j] += add;
        }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < P; j += blockDim.x) {
        float t = 0.f;
        for (int w2 = 0; w2 < 8; ++w2) t += colsum[w2 * P + j];
        acc_out[(size_t)unit * P + j] = t;
    }
}

// ---- prefill, first compression ---------------------------------------------------------------------
// The r most recent prompt tokens stay; among the rest the keep_k - r highest acc (equal acc: the
// newer token stays, i.e. eviction takes the oldest first). Kept tokens fill slots 0.. in position
// order. acc_in [unit][parts][P] holds partial sums of the prefill scores, added in part order.
// The (keep_k - r)-th largest score tau is found by an MSB-first radix select (4 passes of 8 bits
// over shared-memory histograms); scores above tau stay, and among those equal to tau the newest
// fill the remainder. grid units, block 256. Shared: accs [P] f32, slot [P] int, src [P] int.

__device__ __forceinline__ uint32_t score_key(float f) {  // order-preserving for all floats
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide scan of one value per thread; *total = the block's sum. All threads call.
__device__ __forceinline__ int block_scan_excl(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int before = 0, tot = 0;
    for (int w2 = 0; w2 < nw; ++w2) {
        const int t = warp_tot[w2];
        before += (w2 < warp) ? t : 0;
        tot += t;
    }
    __syncthreads();
    *total = tot;
    return before + x - v;
}

template <typename T>
__global__ void __launch_bounds__(kPrefThreads) h2o_compress_kernel(
    const T *__restrict__ K, const T *__restrict__ V, const float *__restrict__ acc_in, int parts,
    int P, int d, int keep_k, int cap, T *__restrict__ Ks, T *__restrict__ Vs, float *__restrict__ acc,
    int32_t *__restrict__ pos, int32_t *__restrict__ nslots, int32_t *__restrict__ hole) {
    extern __shared__ __align__(16) unsigned char smraw[];
    float *colsum = reinterpret_cast<float *>(smraw);  // [P]
    int *slot_of = reinterpret_cast<int *>(colsum + P);  // [P] slot of position j, or -1
    int *src_of = slot_of + P;                           // [P] position held by slot s
    __shared__ int warp_tot[32];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_prefix;
    __shared__ int s_krem;
    const int unit = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T *Ku = K + (size_t)unit * P * d;
    const T *Vu = V + (size_t)unit * P * d;
    for (int j = threadIdx.x; j < P; j += blockDim.x) {
        float t = 0.f;
        for (int p = 0; p < parts; ++p) t += acc_in[((size_t)unit * parts + p) * P + j];
        colsum[j] = t;
    }
    const int r = keep_k / 2;
    const int heavy = keep_k - r;
    const int ncand = keep_k >= P ? 0 : P - r;  // candidates for the heavy part: [0, ncand)
    if (threadIdx.x == 0) {
        s_prefix = 0u;
        s_krem = heavy;
    }
    __syncthreads();
    if (ncand > 0 && heavy > 0) {
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            const uint32_t mask = pass == 0 ? 0u : (0xffffffffu << (shift + 8));
            for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
            __syncthreads();
            const uint32_t prefix = s_prefix;
            for (int j = threadIdx.x; j < ncand; j += blockDim.x) {
                const uint32_t key = score_key(colsum[j]);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                // lane l holds bins 255-8l .. 248-8l (descending); find the bin of the krem-th
                // largest key among those matching the prefix
                uint32_t c[8];
                int sum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    c[i] = hist[255 - 8 * lane - i];
                    sum += (int)c[i];
                }
                int incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const int krem = s_krem;
                const unsigned ball = __ballot_sync(0xffffffffu, incl >= krem);
                if (ball != 0u && lane == __ffs(ball) - 1) {
                    int kr = krem - (incl - sum);
                    int bsel = 248 - 8 * lane;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if ((int)c[i] >= kr) {
                            bsel = 255 - 8 * lane - i;
                            break;
                        }
                        kr -= (int)c[i];
                    }
                    s_krem = kr;
                    s_prefix = prefix | ((uint32_t)bsel << shift);
                }
            }
            __syncthreads();
        }
    }
    const uint32_t tau = s_prefix;
    const int take_eq = s_krem;  // candidates equal to tau that stay, newest first
    // keep flags; ranks among the candidates equal to tau by descending position
    int run_eq = 0;
    for (int base = 0; base < P; base += blockDim.x) {
        const int j = P - 1 - (base + (int)threadIdx.x);  // descending positions
        int keep = 0, eq = 0;
        if (j >= 0) {
            if (j >= ncand) {
                keep = 1;
            } else if (heavy > 0) {
                const uint32_t key = score_key(colsum[j]);
                keep = key > tau ? 1 : 0;
                eq = key == tau ? 1 : 0;
            }
        }
        int tot_eq;
        const int rank_eq = run_eq + block_scan_excl(eq, warp_tot, &tot_eq);
        if (j >= 0) slot_of[j] = (keep || (eq && rank_eq < take_eq)) ? 1 : 0;
        run_eq += tot_eq;
    }
    __syncthreads();
    // ordered slot assignment (block scan over ascending positions)
    int run = 0;
    for (int base = 0; base < P; base += blockDim.x) {
        const int j = base + threadIdx.x;
        const int v = j < P ? slot_of[j] : 0;
        int tot;
        const int before = run + block_scan_excl(v, warp_tot, &tot);
        if (j < P) {
            slot_of[j] = v ? before : -1;
            if (v) src_of[before] = j;
        }
        run += tot;
    }
    __syncthreads();
    const int kept = run;
    float *accu = acc + (size_t)unit * cap;
    int32_t *posu = pos + (size_t)unit * cap;
    for (int sl = threadIdx.x; sl < cap; sl += blockDim.x) {
        if (sl < kept) {
            const int j = src_of[sl];
            accu[sl] = colsum[j];
            posu[sl] = j;
        } else {
            accu[sl] = 0.f;
            posu[sl] = -1;
        }
    }
    const int vpr = d * (int)sizeof(T) / 16;
    const uint4 *Ksrc = reinterpret_cast<const uint4 *>(Ku);
    const uint4 *Vsrc = reinterpret_cast<const uint4 *>(Vu);
    uint4 *Kd = reinterpret_cast<uint4 *>(Ks + (size_t)unit * cap * d);
    uint4 *Vd = reinterpret_cast<uint4 *>(Vs + (size_t)unit * cap * d);
    for (int e = threadIdx.x; e < kept * vpr; e += blockDim.x) {
        const int sl = e / vpr, c = e % vpr;
        const size_t src = (size_t)src_of[sl] * vpr + c;
        Kd[e] = Ksrc[src];
        Vd[e] = Vsrc[src];
    }
    if (threadIdx.x == 0) {
        nslots[unit] = kept;
        hole[unit] = -1;
    }
}

// ---- decode step ---------------------------------------------------------------------------------
constexpr int kStepWarps = 8;

template <typename T, int D>
__global__ void __launch_bounds__(kStepWarps * 32) h2o_step_kernel(
    const T *__restrict__ q, const T *__restrict__ kn, const T *__restrict__ vn,
    T *__restrict__ out, int units, int cap, int t, int k_t, int r_t, T *__restrict__ Ks,
    T *__restrict__ Vs, float *__restrict__ acc, int32_t *__restrict__ pos,
    int32_t *__restrict__ nslots, int32_t *__restrict__ hole) {
    constexpr int LPR = D / 8;       // lanes per row (16 bytes each)
    constexpr int RPI = 32 / LPR;    // rows per warp iteration
    extern __shared__ float sbuf_all[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x * kStepWarps + warp;
    if (unit >= units) return;
    float *sb = sbuf_all + warp * cap;  // scores, then probabilities
    const int sub = lane / LPR, part = lane % LPR;
    T *Ku = Ks + (size_t)unit * cap * D;
    T *Vu = Vs + (size_t)unit * cap * D;
    float *au = acc + (size_t)unit * cap;
    int32_t *pu = pos + (size_t)unit * cap;
    // 1. append into the free slot
    const int ns = nslots[unit], hl = hole[unit];
    const int slot = (hl >= 0) ? hl : ns;
    const int nsn = (hl >= 0) ? ns : ns + 1;
    const size_t urow = (size_t)unit * D;
    float qf[8];
    Vec8<T>::load(q + urow + part * 8, qf);
    const float qscale = kLog2e * rsqrtf((float)D);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[i] *= qscale;
    if (sub == 0)
        *reinterpret_cast<uint4 *>(Ku + (size_t)slot * D + part * 8) =
            *reinterpret_cast<const uint4 *>(kn + urow + part * 8);
    if (sub == 1)
        *reinterpret_cast<uint4 *>(Vu + (size_t)slot * D + part * 8) =
            *reinterpret_cast<const uint4 *>(vn + urow + part * 8);
    if (lane == 0) pu[slot] = t - 1;
    __syncwarp();
    // 2. scores s_j = q.k_j (log2 domain)
    for (int j0 = 0; j0 < nsn; j0 += RPI * 4) {
        float dot[4];
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
            const int j = j0 + uu * RPI + sub;
            float kf[8];
            dot[uu] = 0.f;
            if (j < nsn) {
                Vec8<T>::load(Ku + (size_t)j * D + part * 8, kf);
#pragma unroll
                for (int i = 0; i < 8; ++i) dot[uu] = fmaf(qf[i], kf[i], dot[uu]);
            }
        }
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) dot[uu] += __shfl_xor_sync(0xffffffffu, dot[uu], o);
            const int j = j0 + uu * RPI + sub;
            if (part == 0 && j < nsn) sb[j] = dot[uu];
        }
    }
    __syncwarp();
    // 3. softmax over the retained tokens, accumulate
    float mx = -INFINITY;
    for (int j = lane; j < nsn; j += 32) mx = fmaxf(mx, sb[j]);
    mx = warp_max(mx);
    float sum = 0.f;
    for (int j = lane; j < nsn; j += 32) sum += exp2f(sb[j] - mx);
    sum = warp_sum(sum);
    const float inv = 1.f / sum;
    for (int j = lane; j < nsn; j += 32) {
        const float p = exp2f(sb[j] - mx) * inv;
        sb[j] = p;
        const float prev = (j == slot) ? 0.f : au[j];
        au[j] = prev + p;
    }
    __syncwarp();
    // 4. out = sum_j p_j v_j
    float of[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) of[i] = 0.f;
    for (int j0 = 0; j0 < nsn; j0 += RPI * 4) {
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
            const int j = j0 + uu * RPI + sub;
            if (j < nsn) {
                float vf[8];
                Vec8<T>::load(Vu + (size_t)j * D + part * 8, vf);
                const float p = sb[j];
#pragma unroll
                for (int i = 0; i < 8; ++i) of[i] = fmaf(p, vf[i], of[i]);
            }
        }
    }
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i) of[i] += __shfl_xor_sync(0xffffffffu, of[i], o);
    if (sub == 0) Vec8<T>::store(out + urow + part * 8, of);
    // 5. evict: the lowest accumulated score among positions < t - r_t (ties: oldest)
    int new_hole = -1;
    if (nsn > k_t) {
        float ba = INFINITY;
        int bp = 0x7fffffff, bj = -1;
        for (int j = lane; j < nsn; j += 32) {
            const int pj = pu[j];
            if (pj < 0 || pj >= t - r_t) continue;
            const float aj = au[j];
            if (aj < ba || (aj == ba && pj < bp)) {
                ba = aj;
                bp = pj;
                bj = j;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float oa = __shfl_xor_sync(0xffffffffu, ba, o);
            const int op = __shfl_xor_sync(0xffffffffu, bp, o);
            const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
            if (oj >= 0 && (bj < 0 || oa < ba || (oa == ba && op < bp))) {
                ba = oa;
                bp = op;
                bj = oj;
            }
        }
        new_hole = bj;
    }
    __syncwarp();
    if (lane == 0) {
        if (new_hole >= 0) pu[new_hole] = -1;
        nslots[unit] = nsn;
        hole[unit] = new_hole;
    }
}

__global__ void h2o_count_kernel(const int32_t *__restrict__ nslots,
                                 const int32_t *__restrict__ hole, int units,
                                 int32_t *__restrict__ count) {
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u < units) count[u] = nslots[u] - (hole[u] >= 0 ? 1 : 0);
}

template <typename T>
cudaError_t prefill_t(H2OState &s, const void *K, const void *V, const void *Q, int P,
                      int keep_k, float *acc_tmp, cudaStream_t st) {
    cudaError_t e;
    const bool tc = h2o_colsum_tc_supported(s.d, P, s.dtype);
    if (tc) {
        e = launch_h2o_colsum_tc(s.units, P, K, Q, s.dtype, acc_tmp, st);
    } else {
        const size_t smem = h2o_prefill_smem(s.d, P, s.dtype);
        auto kern = h2o_colsum_kernel<T>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<s.units, kPrefThreads, smem, st>>>((const T *)K, (const T *)Q, P, s.d, acc_tmp);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    const size_t smem = (sizeof(float) + 2 * sizeof(int)) * P;
    auto comp = h2o_compress_kernel<T>;
    e = cudaFuncSetAttribute(comp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    comp<<<s.units, kPrefThreads, smem, st>>>((const T *)K, (const T *)V, acc_tmp,
                                              tc ? kColsumTcParts : 1, P, s.d, keep_k,
                                              s.cap, (T *)s.K, (T *)s.V, s.acc, s.pos, s.nslots,
                                              s.hole);
    return cudaGetLastError();
}

template <typename T>
cudaError_t step_t(H2OState &s, const void *q, const void *k, const void *v, void *out, int t,
                   int k_t, int r_t, cudaStream_t st) {
    const dim3 grid((s.units + kStepWarps - 1) / kStepWarps);
    const size_t smem = sizeof(float) * kStepWarps * s.cap;
    if (s.d == 128) {
        h2o_step_kernel<T, 128><<<grid, kStepWarps * 32, smem, st>>>(
            (const T *)q, (const T *)k, (const T *)v, (T *)out, s.units, s.cap, t, k_t, r_t,
            (T *)s.K, (T *)s.V, s.acc, s.pos, s.nslots, s.hole);
    } else if (s.d == 64) {
        h2o_step_kernel<T, 64><<<grid, kStepWarps * 32, smem, st>>>(
            (const T *)q, (const T *)k, (const T *)v, (T *)out, s.units, s.cap, t, k_t, r_t,
            (T *)s.K, (T *)s.V, s.acc, s.pos, s.nslots, s.hole);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

size_t h2o_prefill_smem(int d, int P, int dtype) {
    return dtype_size(dtype) * d * P + sizeof(float) * (8 * P + 8 * 4 * d);
}

bool h2o_prefill_fits(int d, int P, int dtype) {
    return h2o_colsum_tc_supported(d, P, dtype) || h2o_prefill_smem(d, P, dtype) <= 227 * 1024;
}

cudaError_t launch_h2o_prefill(H2OState &s, const void *K, const void *V, const void *Q, int P,
                               cudaStream_t st) {
    int keep_k = (int)floor((double)s.frac * (double)P);
    if (keep_k > P) keep_k = P;
    // partial prefill scores [units][parts][P] go to the state's preallocated scratch (sized for
    // P = max_len when the state was created): the prefill allocates nothing
    if (s.dtype == KVE_F16) return prefill_t<__half>(s, K, V, Q, P, keep_k, s.prefill_part, st);
    return prefill_t<__nv_bfloat16>(s, K, V, Q, P, keep_k, s.prefill_part, st);
}

cudaError_t launch_h2o_step(H2OState &s, const void *q, const void *k, const void *v, void *out,
                            cudaStream_t st) {
    const int t = s.t + 1;
    const int k_t = (int)floor((double)s.frac * (double)t);
    const int r_t = k_t / 2;
    if (s.dtype == KVE_F16) return step_t<__half>(s, q, k, v, out, t, k_t, r_t, st);
    return step_t<__nv_bfloat16>(s, q, k, v, out, t, k_t, r_t, st);
}

cudaError_t launch_h2o_export(const H2OState &s, void *K, void *V, int32_t *pos, float *acc,
                              int32_t *count, cudaStream_t st) {
    const size_t rows = (size_t)s.units * s.cap;
    const size_t rb = (size_t)s.d * dtype_size(s.dtype);
    cudaError_t e = cudaSuccess;
    if (K && e == cudaSuccess) e = cudaMemcpyAsync(K, s.K, rows * rb, cudaMemcpyDeviceToDevice, st);
    if (V && e == cudaSuccess) e = cudaMemcpyAsync(V, s.V, rows * rb, cudaMemcpyDeviceToDevice, st);
    if (pos && e == cudaSuccess)
        e = cudaMemcpyAsync(pos, s.pos, rows * sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    if (acc && e == cudaSuccess)
        e = cudaMemcpyAsync(acc, s.acc, rows * sizeof(float), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return e;
    if (count) h2o_count_kernel<<<(s.units + 255) / 256, 256, 0, st>>>(s.nslots, s.hole, s.units,
                                                                        count);
    return cudaGetLastError();
}

}  // namespace kve

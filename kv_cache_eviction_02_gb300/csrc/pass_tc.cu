// LORE-KV scoring on the 5th-generation tensor cores (tcgen05, sm_103a), bf16 inputs, fp32 TMEM
// accumulators, TMA-staged 128-byte-swizzled operand tiles.
//
// Attention statistics (LORE-KV page, Method: a_{q,i} = softmax_i(q.k_i/sqrt d), o_q =
// sum_i a_{q,i} v_i), one CTA per (unit, 256 or 128 queries, token split):
//   S_t = Q_t K^T (M = 128 queries, N = 128 tokens) per query tile t, an online softmax per query
//   row in a 4-warp group per tile (rows = TMEM lanes), P written back into TMEM as bf16 pairs
//   and O_t += P_t V issued with P read from TMEM (V as the MN-major B operand). O stays in TMEM;
//   it is rescaled only when a row's running maximum grows by more than 2^8. A CTA with two query
//   tiles alternates them on the tensor pipe (one tile's S is computed while the other tile's
//   softmax runs); a CTA with one tile double-buffers S instead.
//
// Projected deletion scores (Eqs. 5-7), one CTA per (unit, pair of query heads, token range),
// tokens on M: S = K [Q_h0; Q_h1]^T, X = V [U_h0; U_h1]^T (U holds -2 G_h o_q) and Y = V L_h
// (||L_h^T v||^2 = ||row of Y||^2; the zero upper-right block of L_h^T is skipped) for 128 tokens
// per tile, one extra K step adding the per-query constants inside the MMAs; two 4-warp epilogue
// groups (one per head) evaluate e = a/(1-a+eps) sqrt(||L^T v||^2 - 2 v.u + c) with
// a = exp2(s log2e/sqrt(d) - lse2) for the head's 64 queries, weighted per query set. Per-head
// partial sums go to the workspace and a small kernel adds the g heads in a fixed order.
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace kve {

constexpr int kSms = 152;  // GB300
constexpr long kScSetupTiles = 4;  // a scoring CTA's set-up, in 128-token tiles of its loop

bool tc_supported(const LorekvDims &D) {
    return D.dtype == KVE_BF16 && D.d == 128 && D.nq >= 1 && D.nq <= 64;
}

// ---- host: tensor maps ---------------------------------------------------------------------------
bool make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                       uint32_t box_inner, uint32_t box_rows, bool f16) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return false;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    if (reinterpret_cast<uintptr_t>(base) % 16 != 0) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token splits (attention) or ranges (scores) that spread `items * parts` CTAs evenly over the
// SMs: minimise ceil(items*parts / SMs) * (ceil(tiles / parts) + setup), where `setup` is a CTA's
// fixed cost in tiles (the scoring CTA stages 112 KB of Q, U and L^T and sets up its TMEM and
// constant tiles before its first token tile).
static int balance_parts(long items, long tiles, int max_parts, long setup = 0) {
    int best = 1;
    long best_cost = -1;
    for (int p = 1; p <= max_parts && p <= tiles; ++p) {
        const long waves = (items * p + kSms - 1) / kSms;
        const long per = (tiles + p - 1) / p;
        const long cost = waves * (per + setup);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = p;
        }
    }
    return best;
}

void tc_plan(LorekvDims *D) {
    const long ntiles = (D->n + 127) / 128;
    // attention CTAs hold two 128-query tiles when the unit's queries fill whole pairs (one
    // K/V stream serves 256 queries); otherwise one tile each, with S double-buffered and a
    // deeper K/V ring (the CTAs of a unit share the stream through L2)
    D->at_qt = D->Qu % 256 == 0 ? 2 : 1;
    const long nqp = (D->Qu + 128 * D->at_qt - 1) / (128 * D->at_qt);
    // Each split writes and the combine re-reads a 256-query partial (o, m, l: ~128 KB, the DRAM
    // traffic of two 128-token K/V tiles) and pays a CTA's set-up; counted as four tiles next to
    // the per-SM tile load (at 128K this picks 7 splits, measured faster than 13 or 16).
    const long items = (long)D->units * nqp;
    int ns = 1;
    long best = -1;
    for (int p = 1; p <= 64 && p <= ntiles; ++p) {
        const long waves = (items * p + kSms - 1) / kSms;
        const long cost = waves * ((ntiles + p - 1) / p) + 4 * waves;
        if (best < 0 || cost < best) {
            best = cost;
            ns = p;
        }
    }
    const long per = (ntiles + ns - 1) / ns;
    D->split_len = (int)(per * 128);
    D->nsplit = (int)((D->n + D->split_len - 1) / D->split_len);
}

namespace {

// ---- small packing kernels -------------------------------------------------------------------------
// The B operand (N = j, K = k, K-major) of Y = V L_h for the two query heads of a CTA, d = 128:
// lt16[l][kv head][pair][r][k] = bf16(L_h[k][j]). Rows 0-127 hold columns j < 64 and rows
// 128-255 columns j >= 64, both in groups of 16 columns alternating between the pair's heads
// (r = 32 g + 16 head + t <-> j = 16 g + t, offset by 64 for the second half). Since L_h is
// lower triangular, column j only gets contributions from k >= j: at the 16-wide K step s only
// the first groups are non-zero, and the MMA over K step s reads just those leading rows. A
// missing second head (odd group size) is zero.
// grid (L * Hkv * npairs, 8), block 256: CTA (blk, rb) writes the 32 packed rows 32 rb .. 32 rb +
// 31, i.e. one 16-column group of both heads: it stages those 16 columns of the two L_h (all 128
// k, rows padded to 17 floats) in shared memory, so that the reads of L (64 bytes along j) and the
// writes of the packed rows (along k, two values a thread) are coalesced and many CTAs share an
// SM.
__global__ void __launch_bounds__(256) pack_lt_kernel(const float *__restrict__ L,
                                                      __nv_bfloat16 *__restrict__ lt, int Hq,
                                                      int Hkv, int g, int npairs) {
    constexpr int d = 128;
    __shared__ float lsm[2][d][17];  // L_h[k][j0 + t] of the pair's two heads
    const int blk = blockIdx.x;     // (l * Hkv + kh) * npairs + pair
    const int rb = blockIdx.y;      // packed rows 32 rb .. 32 rb + 31
    const int pair = blk % npairs, kh = (blk / npairs) % Hkv, l = blk / (npairs * Hkv);
    const int j0 = 64 * (rb >> 2) + 16 * (rb & 3);
    for (int e = threadIdx.x; e < 2 * d * 16; e += blockDim.x) {
        const int hd = e / (d * 16), k = (e / 16) % d, t = e % 16;
        const int hin = 2 * pair + hd;
        lsm[hd][k][t] = hin < g ? L[(((size_t)l * Hq + kh * g + hin) * d + k) * d + j0 + t] : 0.f;
    }
    __syncthreads();
    __nv_bfloat162 *dst =
        reinterpret_cast<__nv_bfloat162 *>(lt + ((size_t)blk * 256 + 32 * rb) * d);
    for (int e = threadIdx.x; e < 32 * d / 2; e += blockDim.x) {
        const int r = e / (d / 2), k = 2 * (e % (d / 2));
        const int hd = r >> 4, t = r & 15;  // row r of the group: head hd, column j0 + t
        dst[e] = __floats2bfloat162_rn(lsm[hd][k][t], lsm[hd][k + 1][t]);
    }
}

// q16[unit][qi][:] = the query of row qi (head-major, window rows then lookahead rows).
// grid (ceil(Qu * d / 8 / 256), units), block 256: one 16-byte word (8 values) per thread.
__global__ void pack_queries_kernel(const __nv_bfloat16 *__restrict__ QW,
                                    const __nv_bfloat16 *__restrict__ QL, LorekvDims D,
                                    __nv_bfloat16 *__restrict__ q16) {
    const int unit = blockIdx.y;
    const int per_row = D.d / 8;
    const long e = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (long)D.Qu * per_row) return;
    const int qi = (int)(e / per_row), k8 = (int)(e % per_row);
    const int kh = unit % D.Hkv, sl = unit / D.Hkv;
    const int j = qi / D.nq, r = qi % D.nq, h = kh * D.g + j;
    const __nv_bfloat16 *src = (r < D.w) ? QW + (((size_t)sl * D.Hq + h) * D.w + r) * D.d
                                         : QL + (((size_t)sl * D.Hq + h) * D.MT + (r - D.w)) * D.d;
    __nv_bfloat16 *dst = q16 + ((size_t)unit * D.Qu + qi) * D.d;
    reinterpret_cast<uint4 *>(dst)[k8] = __ldg(reinterpret_cast<const uint4 *>(src) + k8);
}

// Per-query constants of the scoring epilogue: {-lse2, c, w, a_max}.
__global__ void pack_qconst_kernel(const float *__restrict__ lse2, const float *__restrict__ cq,
                                   const float *__restrict__ wq, const float *__restrict__ amax,
                                   long rows, float4 *__restrict__ qconst) {
    const long r = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (r < rows) qconst[r] = make_float4(-lse2[r], cq[r], wq[r], amax[r]);
}

// S_i = sum over query heads of the partial scores (fixed order); 0 for protected tokens.
__global__ void reduce_heads_kernel(const float *__restrict__ part, int g, int n, int sink, int w,
                                    float *__restrict__ S) {
    const int unit = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float acc = 0.f;
    for (int j = 0; j < g; ++j) acc += part[((size_t)unit * g + j) * n + i];
    S[(size_t)unit * n + i] = (i >= sink && i < n - w) ? acc : 0.f;
}

// ---- scores kernel -----------------------------------------------------------------------------------
struct ScoresArgs {
    int n, g, Hkv, L, Hq, nq, Qu, sink, w;
    int ntiles, tpr, nranges;
    float eps, k1;
    const float4 *qconst;
    float *part_s;
    int *pk_cnt, *pk_tok;  // pairs left out for the exact peaked-pair evaluation
    unsigned *err;
};

constexpr int kScThreads = 320;  // TMA, MMA issuer, 2 epilogue groups (one per head)
// One CTA scores two query heads of a unit over a token range: every staged K/V tile serves both,
// and the heads' operands are interleaved so that each MMA is wide (N = 128 or 256).
// Shared memory:
//   Q    2 K-blocks x 16 KB: rows [Q_h0 (64) | Q_h1 (64)]           -> B of S = K [Q_h0;Q_h1]^T
//   B2   rows [U_h0 | U_h1 | Lt rows for Y columns 0-63 | Lt rows for Y columns 64-127] -> B of
//        V B2^T, where the L_h^T rows of the two heads alternate in groups of 16 (the packing
//        in pack_lt_kernel). Rows of L_h^T for columns >= 64 are zero for k < 64, so K-block 0
//        holds rows 0-255 (32 KB) and K-block 1 rows 0-383 (48 KB).
//   ring 3 x 32 KB TMA boxes (V_i, K_i, V_i+1, ...).
//   one extra K step (32-byte swizzle, 16 bf16 per row) that adds per-query constants inside the
//   MMAs: A_aug (128 token rows [1, 1, 1, 0, ...]), B_aug_S (the 128 query rows of S: -lse2/k1
//   split into three bf16 terms) and B_aug_V (the 128 query rows of X: c split into three bf16
//   terms, then 128 zero rows under Y). With U staged as -2u, the MMAs give S' = s - lse2/k1 and
//   X' = c - 2 v.u directly.
//   per-query weights (general query layout) | per-set weights | barriers.
// TMEM (512 columns, one buffer): S_h0 | S_h1 | X_h0 | X_h1 (64 columns each) | Ya | Yb (128
// each: columns 0-63 / 64-127 of Y = V L_h of both heads, in alternating groups of 16). Yb only
// takes the second K-block of V, and each 16-column group only the K steps at or after its
// diagonal block.
constexpr int SC_HPC = 2;                                  // query heads per CTA
constexpr uint32_t SC_Q = 0, SC_B2 = 32768;
constexpr uint32_t SC_B2_K0 = 0, SC_B2_K1 = 32768;         // K-block offsets inside B2
constexpr uint32_t SC_RING = SC_B2 + 32768 + 49152;        // 112 KB
constexpr int SC_SLOTS = 3;
constexpr uint32_t SC_AUG_A = SC_RING + SC_SLOTS * 32768;  // 128 rows x 32 B
constexpr uint32_t SC_AUG_S = SC_AUG_A + 4096;             // 128 rows x 32 B
constexpr uint32_t SC_AUG_V = SC_AUG_S + 4096;             // 256 rows x 32 B
constexpr uint32_t SC_QW = SC_AUG_V + 8192;                // [2][32] float2 weight pairs
constexpr uint32_t SC_SW = SC_QW + SC_HPC * 32 * 8;        // [2][8] per-set weights
constexpr uint32_t SC_BAR = SC_SW + SC_HPC * 8 * 4;
constexpr size_t SC_SMEM = SC_BAR + 256 + 1024;
// Query layout with compile-time sets: w = 32 window queries, then M = 4 trajectories of T = 8
// lookahead queries; pairs 0-15 are the window, pairs 16 + 4m .. 19 + 4m trajectory m.
constexpr int kSetW = 32, kSetM = 4, kSetT = 8;

// v as the sum of three bf16 terms (relative error about 2^-24); a value below -1e30 (a padded
// query's -inf) becomes (-1e30, 0, 0).
__device__ __forceinline__ void split3_bf16(float v, __nv_bfloat16 *dst0, __nv_bfloat16 *dst1,
                                            __nv_bfloat16 *dst2) {
    if (!(v > -1e30f)) {
        *dst0 = __float2bfloat16_rn(-1e30f);
        *dst1 = *dst2 = __float2bfloat16_rn(0.f);
        return;
    }
    const __nv_bfloat16 a = __float2bfloat16_rn(v);
    float r = v - __bfloat162float(a);
    const __nv_bfloat16 b = __float2bfloat16_rn(r);
    r -= __bfloat162float(b);
    *dst0 = a;
    *dst1 = b;
    *dst2 = __float2bfloat16_rn(r);
}

// The pair terms of one token row against the 64 queries of one head (two per packed FP32
// instruction): unweighted per-set sums (kFixedSets) or weighted sums into acc2. With kPeak,
// a pair whose a exceeds tau is left out (a := 0) and recorded for the exact evaluation of
// peaked pairs; a query takes at most kPeakSlots such tokens (a record that finds the slots
// full keeps its pair in the sum instead).
template <bool kFixedSets, bool kPeak>
__device__ __forceinline__ void score_pairs(const float (&s0)[32], const float (&s1)[32],
                                            const float (&x0)[32], const float (&x1)[32],
                                            float nv, uint64_t (&acc2)[8],
                                            const float2 *qwh, uint64_t k1_2, uint64_t one_2,
                                            uint64_t neg1_2, float tau, int tok, int *pk_cnt,
                                            int *pk_tok) {
    const uint64_t nv_2 = tc::pk2(nv, nv);
#pragma unroll
    for (int p = 0; p < 32; ++p) {
        const float sa = (p < 16) ? s0[2 * p] : s1[2 * p - 32];
        const float sb = (p < 16) ? s0[2 * p + 1] : s1[2 * p - 31];
        const float xa = (p < 16) ? x0[2 * p] : x1[2 * p - 32];
        const float xb = (p < 16) ? x0[2 * p + 1] : x1[2 * p - 31];
        float ea, eb;
        tc::upk2(tc::mul2(tc::pk2(sa, sb), k1_2), ea, eb);
        float aa = tc::ex2_approx(ea), ab = tc::ex2_approx(eb);
        if (kPeak && (aa > tau || ab > tau)) {
            if (aa > tau) {
                const int slot = atomicAdd(pk_cnt + 2 * p, 1);
                if (slot < kPeakSlots) {
                    pk_tok[(2 * p) * kPeakSlots + slot] = tok;
                    aa = 0.f;
                }
            }
            if (ab > tau) {
                const int slot = atomicAdd(pk_cnt + 2 * p + 1, 1);
                if (slot < kPeakSlots) {
                    pk_tok[(2 * p + 1) * kPeakSlots + slot] = tok;
                    ab = 0.f;
                }
            }
        }
        const uint64_t a2 = tc::pk2(aa, ab);
        float ya, yb;
        tc::upk2(tc::add2(tc::pk2(xa, xb), nv_2), ya, yb);
        const uint64_t x2 = tc::pk2(fmaxf(ya, 1e-30f), fmaxf(yb, 1e-30f));
        const uint64_t dd2 = tc::fma2(a2, neg1_2, one_2);
        float za, zb;
        tc::upk2(tc::mul2(tc::mul2(x2, dd2), dd2), za, zb);
        const uint64_t r2 = tc::pk2(tc::rsqrt_approx(za), tc::rsqrt_approx(zb));
        if (kFixedSets) {  // unweighted; the set's weight is applied once at the end
            const int slot = p < 16 ? (p & 3) : 4 + ((p - 16) >> 2);
            acc2[slot] = tc::fma2(tc::mul2(a2, x2), r2, acc2[slot]);
        } else {
            const float2 cw = qwh[p];
            acc2[p & 3] = tc::fma2(tc::mul2(tc::mul2(a2, tc::pk2(cw.x, cw.y)), x2), r2,
                                   acc2[p & 3]);
        }
    }
}

template <bool kFixedSets>
__global__ void __launch_bounds__(kScThreads, 1)
    scores_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_u,
                     const __grid_constant__ CUtensorMap tm_lt, ScoresArgs A) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int npairs = (A.g + SC_HPC - 1) / SC_HPC;
    const int b = blockIdx.x;
    const int hp = b % npairs;
    const int range = (b / npairs) % A.nranges;
    const int unit = b / (npairs * A.nranges);
    const int j0 = hp * SC_HPC;
    const int nh = min(SC_HPC, A.g - j0);         // heads of this CTA (1 for an odd last pair)
    const int t_begin = range * A.tpr;
    const int ntl = min(A.ntiles, t_begin + A.tpr) - t_begin;
    if (ntl <= 0) return;
    const int kh = unit % A.Hkv, l = (unit / A.Hkv) % A.L;

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + SC_BAR);
    // tfull1/tfree1: the V-tile products X, Y (columns 128-511); tfull2/tfree2: S (columns 0-127)
    uint64_t *ops_full = bars + 0, *rfull = bars + 1, *rempty = bars + 1 + SC_SLOTS,
             *tfull1 = bars + 1 + 2 * SC_SLOTS, *tfree1 = tfull1 + 1, *tfull2 = tfull1 + 2,
             *tfree2 = tfull1 + 3, *drain = tfull1 + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tfull1 + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tfull1 + 6);
    float *sw = reinterpret_cast<float *>(sm + SC_SW);
    float2 *qw = reinterpret_cast<float2 *>(sm + SC_QW);

    if (threadIdx.x == 0) {
        tc::mbar_init(ops_full, 1);
        for (int s = 0; s < SC_SLOTS; ++s) {
            tc::mbar_init(&rfull[s], 1);
            tc::mbar_init(&rempty[s], 1);
        }
        tc::mbar_init(tfull1, 1);
        tc::mbar_init(tfull2, 1);
        tc::mbar_init(tfree1, 128 * nh);  // every epilogue thread has read the columns
        tc::mbar_init(tfree2, 128 * nh);
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::fence_before_sync();
    }
    // the augmentation K step: zero it, then write the ones of A_aug and the constants of the queries
    for (int e = threadIdx.x; e < 16384 / 16; e += blockDim.x)
        reinterpret_cast<uint4 *>(sm + SC_AUG_A)[e] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (threadIdx.x < 128) {
        __nv_bfloat16 *aa = reinterpret_cast<__nv_bfloat16 *>(sm + SC_AUG_A);
        const __nv_bfloat16 one = __float2bfloat16_rn(1.f);
        for (int k = 0; k < 3; ++k) aa[tc::sw32_offset(threadIdx.x, k) / 2] = one;
    }
    int peaked = 0;  // a query of this CTA has a non-protected pair with a > kPeakFlag
    if (threadIdx.x >= 128 && threadIdx.x < 128 + 64 * SC_HPC) {  // one query each
        const int q = threadIdx.x - 128;                           // B row: head q / 64
        const int hh = q >> 6, r = q & 63;
        float4 c = make_float4(-INFINITY, 0.f, 0.f, 0.f);
        if (hh < nh && r < A.nq) c = A.qconst[(size_t)unit * A.Qu + (size_t)(j0 + hh) * A.nq + r];
        peaked = c.w > kPeakFlag;
        __nv_bfloat16 *bs = reinterpret_cast<__nv_bfloat16 *>(sm + SC_AUG_S);
        __nv_bfloat16 *bv = reinterpret_cast<__nv_bfloat16 *>(sm + SC_AUG_V);
        const uint32_t o0 = tc::sw32_offset(q, 0) / 2, o1 = tc::sw32_offset(q, 1) / 2,
                       o2 = tc::sw32_offset(q, 2) / 2;
        split3_bf16(c.x / A.k1, bs + o0, bs + o1, bs + o2);  // -lse2 / k1
        split3_bf16(c.y, bv + o0, bv + o1, bv + o2);         // c
        if (kFixedSets) {
            // the weight is per set: window, then one per trajectory
            if (r == 0) sw[hh * 8] = c.z;
            if (r >= kSetW && (r - kSetW) % kSetT == 0) sw[hh * 8 + 1 + (r - kSetW) / kSetT] = c.z;
        } else {
            reinterpret_cast<float *>(qw)[hh * 64 + r] = c.z;  // weight pairs (2t, 2t+1)
        }
    }
    tc::fence_proxy_async_smem();  // generic-proxy writes -> MMA operand reads
    const int peak_cta = __syncthreads_or(peaked);
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer ----
            tc::mbar_expect_tx(ops_full, 32768u * nh + 49152u);
            for (int hh = 0; hh < nh; ++hh) {
                const int qrow = unit * A.Qu + (j0 + hh) * A.nq;
                for (int kb = 0; kb < 2; ++kb) {
                    uint8_t *b2 = sm + SC_B2 + (kb ? SC_B2_K1 : SC_B2_K0) + hh * 8192;
                    tc::tma_load_2d(sm + SC_Q + kb * 16384 + hh * 8192, &tm_q, 64 * kb, qrow,
                                    ops_full);
                    tc::tma_load_2d(b2, &tm_u, 64 * kb, qrow, ops_full);
                }
            }
            // the pair's packed L^T rows: 0-127 (Y columns 0-63) into both K-blocks, 128-255
            // (Y columns 64-127) into the second
            const int lrow = ((l * A.Hkv + kh) * npairs + hp) * 256;
            for (int kb = 0; kb < 2; ++kb) {
                uint8_t *b2 = sm + SC_B2 + (kb ? SC_B2_K1 : SC_B2_K0);
                tc::tma_load_2d(b2 + 16384, &tm_lt, 64 * kb, lrow, ops_full);
                tc::tma_load_2d(b2 + 16384 + 8192, &tm_lt, 64 * kb, lrow + 64, ops_full);
            }
            tc::tma_load_2d(sm + SC_B2 + SC_B2_K1 + 32768, &tm_lt, 64, lrow + 128, ops_full);
            tc::tma_load_2d(sm + SC_B2 + SC_B2_K1 + 32768 + 8192, &tm_lt, 64, lrow + 192,
                            ops_full);
            int issued = 0;
            for (int c = 0; c < 2 * ntl; ++c) {
                const int slot = c % SC_SLOTS;
                const uint32_t ph = (c / SC_SLOTS) & 1;
                if (!tc::mbar_wait(&rempty[slot], ph ^ 1, abort_flag, A.err)) break;
                tc::mbar_expect_tx(&rfull[slot], 32768);
                const int row = unit * A.n + (t_begin + (c >> 1)) * 128;
                const CUtensorMap *map = (c & 1) ? &tm_k : &tm_v;  // V_i, K_i, V_i+1, ...
                uint8_t *dst = sm + SC_RING + slot * 32768;
                tc::tma_load_2d(dst, map, 0, row, &rfull[slot]);
                tc::tma_load_2d(dst + 16384, map, 64, row, &rfull[slot]);
                issued = c + 1;
            }
            // copies still in flight land before the CTA exits (immediate on the normal path)
            tc::mbar_drain(ops_full, 0);
            for (int c = issued - SC_SLOTS < 0 ? 0 : issued - SC_SLOTS; c < issued; ++c)
                tc::mbar_drain(&rfull[c % SC_SLOTS], (c / SC_SLOTS) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0 && tc::mbar_wait(ops_full, 0, abort_flag, A.err)) {  // ---- MMA issuer ----
            tc::fence_after_sync();
            const uint32_t ring = tc::smem_u32(sm + SC_RING);
            const uint32_t q_addr = tc::smem_u32(sm + SC_Q);
            const uint32_t b2_addr = tc::smem_u32(sm + SC_B2);
            const uint32_t aug_a = tc::smem_u32(sm + SC_AUG_A), aug_s = tc::smem_u32(sm + SC_AUG_S),
                           aug_v = tc::smem_u32(sm + SC_AUG_V);
            constexpr uint32_t id128 = tc::idesc_bf16(128, 128, 0);
            constexpr uint32_t id256 = tc::idesc_bf16(128, 256, 0);
            for (int i = 0; i < ntl; ++i) {
                const int cv = 2 * i, ck = 2 * i + 1;
                const int sv = cv % SC_SLOTS, sk = ck % SC_SLOTS;
                // group 1: [X_h0 | X_h1 | Ya_h0 | Ya_h1] = V [U_h0; U_h1; L_h0^T(0:64); L_h1^T(0:64)]^T
                // and [Yb_h0 | Yb_h1] from the second K-block of V
                if (!tc::mbar_wait(&rfull[sv], (cv / SC_SLOTS) & 1, abort_flag, A.err)) break;
                if (!tc::mbar_wait(tfree1, (i & 1) ^ 1, abort_flag, A.err)) break;
                tc::fence_after_sync();
                const uint32_t v_addr = ring + sv * 32768;
                // K steps from the last down: the first product covers every column; at K step
                // s the Y_a columns of groups above s are zero (L lower triangular) and are left
                // out by narrowing N to the leading B rows
#pragma unroll
                for (int k = 7; k >= 0; --k) {
                    const uint32_t ao = (k >> 2) * 16384 + (k & 3) * 32;
                    const uint32_t bo = ((k >> 2) ? SC_B2_K1 : SC_B2_K0) + (k & 3) * 32;
                    const int nn = 128 + 32 * (k < 3 ? k + 1 : 4);
                    tc::mma_bf16(tmem + 128, tc::sdesc_sw128(v_addr + ao, 16, 1024),
                                 tc::sdesc_sw128(b2_addr + bo, 16, 1024),
                                 tc::idesc_bf16(128, nn, 0), k < 7);
                }
                tc::mma_bf16(tmem + 128, tc::sdesc_sw32(aug_a), tc::sdesc_sw32(aug_v), id256, 1);
#pragma unroll
                for (int k = 7; k >= 4; --k) {  // Y_b: groups g need K steps >= 4 + g
                    const uint32_t ao = 16384 + (k & 3) * 32;
                    const uint32_t bo = SC_B2_K1 + 32768 + (k & 3) * 32;
                    tc::mma_bf16(tmem + 384, tc::sdesc_sw128(v_addr + ao, 16, 1024),
                                 tc::sdesc_sw128(b2_addr + bo, 16, 1024),
                                 tc::idesc_bf16(128, 32 * (k - 3), 0), k < 7);
                }
                tc::mma_commit(&rempty[sv]);
                tc::mma_commit(tfull1);
                // group 2: [S_h0 | S_h1] = K [Q_h0; Q_h1]^T
                if (!tc::mbar_wait(&rfull[sk], (ck / SC_SLOTS) & 1, abort_flag, A.err)) break;
                if (!tc::mbar_wait(tfree2, (i & 1) ^ 1, abort_flag, A.err)) break;
                tc::fence_after_sync();
                const uint32_t k_addr = ring + sk * 32768;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
                    tc::mma_bf16(tmem, tc::sdesc_sw128(k_addr + o, 16, 1024),
                                 tc::sdesc_sw128(q_addr + o, 16, 1024), id128, k > 0);
                }
                tc::mma_bf16(tmem, tc::sdesc_sw32(aug_a), tc::sdesc_sw32(aug_s), id128, 1);
                tc::mma_commit(&rempty[sk]);
                tc::mma_commit(tfull2);
            }
        }
        if (lane == 0) {  // every product issued has completed before the tensor memory is freed
            tc::mma_commit(drain);
            tc::mbar_drain(drain, 0);
        }
    } else if ((warp - 2) >> 2 < nh) {
        // ---- epilogue: group hh (warps 2-5 -> head 0, 6-9 -> head 1); warp w reads TMEM lanes
        // 32 (w % 4) .. +31 ----
        const int hh = (warp - 2) >> 2, lg = warp & 3;
        const int row = lg * 32 + lane;
        const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
        float *out = A.part_s + ((size_t)unit * A.g + j0 + hh) * A.n;
        const size_t qrow0 = (size_t)unit * A.Qu + (size_t)(j0 + hh) * A.nq;
        int *pk_cnt = A.pk_cnt + qrow0, *pk_tok = A.pk_tok + qrow0 * kPeakSlots;
        const float one_eps = 1.f + A.eps;
        const float2 *qwh = qw + hh * 32;
        const uint64_t k1_2 = tc::pk2(A.k1, A.k1);
        const uint64_t one_2 = tc::pk2(one_eps, one_eps), neg1_2 = tc::pk2(-1.f, -1.f);
        float wset[1 + kSetM];
#pragma unroll
        for (int k = 0; k < 1 + kSetM; ++k) wset[k] = kFixedSets ? sw[hh * 8 + k] : 0.f;
        for (int i = 0; i < ntl; ++i) {
            if (!tc::mbar_wait_warp(tfull1, i & 1, abort_flag, A.err)) break;
            tc::fence_after_sync();
            const uint32_t tb = tmem + lane_off;
            // ||L_h^T v||^2 of this thread's token (the 128 columns of Y), and X
            float x0[32], x1[32];
            uint64_t np2[4] = {0, 0, 0, 0};  // bit pattern 0 = (0.f, 0.f)
            {
                // this head's 64 Y_a and 64 Y_b columns: groups of 16 at 32 g + 16 hh
                float y[4][16];
#pragma unroll
                for (int gi = 0; gi < 4; ++gi) tc::tmem_ld16(tb + 256 + 32 * gi + 16 * hh, y[gi]);
                tc::tmem_wait_ld();
#pragma unroll
                for (int gi = 0; gi < 4; ++gi)
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        const uint64_t a = tc::pk2(y[gi][c], y[gi][c + 1]);
                        np2[(c >> 1) & 3] = tc::fma2(a, a, np2[(c >> 1) & 3]);
                    }
#pragma unroll
                for (int gi = 0; gi < 4; ++gi) tc::tmem_ld16(tb + 384 + 32 * gi + 16 * hh, y[gi]);
                tc::tmem_ld32(tb + 128 + 64 * hh, x0);
                tc::tmem_ld32(tb + 160 + 64 * hh, x1);
                tc::tmem_wait_ld();
                tc::fence_before_sync();
                tc::mbar_arrive(tfree1);
#pragma unroll
                for (int gi = 0; gi < 4; ++gi)
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        const uint64_t a = tc::pk2(y[gi][c], y[gi][c + 1]);
                        np2[(c >> 1) & 3] = tc::fma2(a, a, np2[(c >> 1) & 3]);
                    }
            }
            float nv;
            {
                float n[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) tc::upk2(np2[k], n[2 * k], n[2 * k + 1]);
                nv = ((n[0] + n[1]) + (n[2] + n[3])) + ((n[4] + n[5]) + (n[6] + n[7]));
            }
            if (!tc::mbar_wait_warp(tfull2, i & 1, abort_flag, A.err)) break;
            tc::fence_after_sync();
            float s0[32], s1[32];
            tc::tmem_ld32(tb + 64 * hh, s0);
            tc::tmem_ld32(tb + 64 * hh + 32, s1);
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            tc::mbar_arrive(tfree2);
            // e = a sqrt(x) / (1 - a + eps) for two queries per packed FP32 instruction, with
            // a = exp2(S' k1) (S' = s - lse2/k1), x = ||L^T v||^2 + X' (X' = c - 2 v.u) and
            // sqrt(x) / dd = x rsqrt(x dd^2)
            const int tok = (t_begin + i) * 128 + row;
            uint64_t acc2[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (peak_cta) {
                // pairs of non-protected tokens with a > kPeakTau are left out and recorded
                const float tau = (tok >= A.sink && tok < A.n - A.w) ? kPeakTau : INFINITY;
                score_pairs<kFixedSets, true>(s0, s1, x0, x1, nv, acc2, qwh, k1_2, one_2, neg1_2,
                                              tau, tok, pk_cnt, pk_tok);
            } else {
                score_pairs<kFixedSets, false>(s0, s1, x0, x1, nv, acc2, qwh, k1_2, one_2, neg1_2,
                                               INFINITY, tok, pk_cnt, pk_tok);
            }
            float acc = 0.f;
            if (kFixedSets) {
                float win = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float u, v;
                    tc::upk2(acc2[k], u, v);
                    win += u + v;
                }
                acc = wset[0] * win;
#pragma unroll
                for (int m = 0; m < kSetM; ++m) {
                    float u, v;
                    tc::upk2(acc2[4 + m], u, v);
                    acc = fmaf(wset[1 + m], u + v, acc);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float u, v;
                    tc::upk2(acc2[k], u, v);
                    acc += u + v;
                }
            }
            if (tok < A.n) out[tok] = (tok >= A.sink && tok < A.n - A.w) ? acc : 0.f;
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ---- attention-statistics kernel ------------------------------------------------------------------
struct AttnArgs {
    int n, Qu, nq, w, sink, window_causal, nsplit, split_len, nqp;
    float k1;
    float2 *part_ml;
    float *part_o;
    float *part_mx;  // largest visible non-protected logit of the split (log2 domain)
    unsigned *err;
};

// TMA, MMA issuer, 2 idle, one softmax group of 4 warps per query tile
template <int QT>
constexpr int at_threads() { return (4 + 4 * QT) * 32; }
// Shared memory of a CTA holding QT query tiles: the Q tiles (32 KB each), then the K/V ring of
// 32 KB items (K_0, V_0, K_1, ...: 5 slots next to two Q tiles, 6 next to one), then barriers.
template <int QT>
struct AtLayout {
    static constexpr int SLOTS = QT == 2 ? 5 : 6;
    static constexpr uint32_t Q = 0, RING = QT * 32768;
    static constexpr uint32_t BAR = RING + SLOTS * 32768;
    static constexpr size_t SMEM = BAR + 256 + 1024;
};
constexpr int AT_SLOTS = AtLayout<2>::SLOTS;  // the two-tile issue helpers below
constexpr uint32_t AT_Q = AtLayout<2>::Q, AT_RING = AtLayout<2>::RING;
constexpr float kRescaleLog2 = 8.f;  // rescale O only when a row maximum grows by > 2^8
constexpr float kNoMax = -1e30f;     // running maximum before any visible token

// S_t = Q_t K_i^T for query tile t (K_i = ring item 2i) into TMEM columns [128 t, 128 t + 128).
// Issued after P_t(i-1) V_(i-1) by the same thread: MMAs execute in issue order, so the product
// has read P_t (which lives in these columns) before S_t(i) overwrites it.
__device__ __forceinline__ bool attn_issue_s(uint32_t base, uint32_t tmem, int t, int i, int nqt,
                                             uint64_t *rfull, uint64_t *rempty, uint64_t *s_full,
                                             volatile int *abort_flag, unsigned *err) {
    constexpr uint32_t id_s = tc::idesc_bf16(128, 128, 0);
    const int c = 2 * i, slot = c % AT_SLOTS;
    if (t == 0 && !tc::mbar_wait(&rfull[slot], (c / AT_SLOTS) & 1, abort_flag, err))
        return false;
    tc::fence_after_sync();
    const uint32_t q_addr = base + AT_Q + t * 32768;
    const uint32_t k_addr = base + AT_RING + slot * 32768;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
        tc::mma_bf16(tmem + t * 128, tc::sdesc_sw128(q_addr + o, 16, 1024),
                     tc::sdesc_sw128(k_addr + o, 16, 1024), id_s, k > 0);
    }
    tc::mma_commit(&s_full[t]);
    if (t == nqt - 1) tc::mma_commit(&rempty[slot]);  // K_i is done once every tile used it
    return true;
}

// O_t += P_t V_i for query tile t: P_t is read from TMEM (bf16 pairs in the first 64 columns of
// S_t, 8 columns per 16 tokens), V_i (ring item 2i+1) is the MN-major B operand.
__device__ __forceinline__ bool attn_issue_pv(uint32_t base, uint32_t tmem, int t, int i, int nqt,
                                              uint64_t *rfull, uint64_t *rempty, uint64_t *p_full,
                                              uint64_t *o_done, volatile int *abort_flag,
                                              unsigned *err) {
    constexpr uint32_t id_pv = tc::idesc_bf16(128, 128, 1);
    const int c = 2 * i + 1, slot = c % AT_SLOTS;
    if (t == 0 && !tc::mbar_wait(&rfull[slot], (c / AT_SLOTS) & 1, abort_flag, err))
        return false;
    if (!tc::mbar_wait(&p_full[t], i & 1, abort_flag, err)) return false;
    tc::fence_after_sync();
    const uint32_t v_addr = base + AT_RING + slot * 32768;
#pragma unroll
    for (int k = 0; k < 8; ++k)  // K = 16 tokens per step: 8 TMEM columns of P, 16 rows of V
        tc::mma_bf16_ts(tmem + 256 + t * 128, tmem + t * 128 + 8 * k,
                        tc::sdesc_sw128(v_addr + k * 2048, 16384, 1024), id_pv,
                        (i > 0 || k > 0) ? 1u : 0u);
    tc::mma_commit(&o_done[t]);
    if (t == nqt - 1) tc::mma_commit(&rempty[slot]);  // V_i is done once every tile used it
    return true;
}

// One query tile (the CTA's second 128 queries hold no valid row): S is double-buffered in the
// columns the two tiles use otherwise, so S(i + 1) is computed while the softmax of S(i) runs.
// S(i) goes to buffer i % 2 (TMEM columns 128 (i % 2)); it is issued right after P(i - 2) V,
// which read its P from the same columns (MMAs execute in issue order).
template <int QT>
__device__ __forceinline__ bool attn_db_issue_s(uint32_t base, uint32_t tmem, int i,
                                                uint64_t *rfull, uint64_t *rempty,
                                                uint64_t *s_full, volatile int *abort_flag,
                                                unsigned *err) {
    constexpr uint32_t id_s = tc::idesc_bf16(128, 128, 0);
    using L = AtLayout<QT>;
    const int c = 2 * i, slot = c % L::SLOTS, b = i & 1;
    if (!tc::mbar_wait(&rfull[slot], (c / L::SLOTS) & 1, abort_flag, err)) return false;
    tc::fence_after_sync();
    const uint32_t q_addr = base + L::Q;
    const uint32_t k_addr = base + L::RING + slot * 32768;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
        tc::mma_bf16(tmem + b * 128, tc::sdesc_sw128(q_addr + o, 16, 1024),
                     tc::sdesc_sw128(k_addr + o, 16, 1024), id_s, k > 0);
    }
    tc::mma_commit(&s_full[b]);
    tc::mma_commit(&rempty[slot]);
    return true;
}
// O += P(i) V_i with P(i) in buffer i % 2; the last product also completes the single-use
// o_final barrier (o_done alone can be two phases behind the softmax here: S(i + 1) is issued
// before P(i) V).
template <int QT>
__device__ __forceinline__ bool attn_db_issue_pv(uint32_t base, uint32_t tmem, int i, int ntl,
                                                 uint64_t *rfull, uint64_t *rempty,
                                                 uint64_t *p_full, uint64_t *o_done,
                                                 uint64_t *o_final, volatile int *abort_flag,
                                                 unsigned *err) {
    constexpr uint32_t id_pv = tc::idesc_bf16(128, 128, 1);
    using L = AtLayout<QT>;
    const int c = 2 * i + 1, slot = c % L::SLOTS, b = i & 1;
    if (!tc::mbar_wait(&rfull[slot], (c / L::SLOTS) & 1, abort_flag, err)) return false;
    if (!tc::mbar_wait(&p_full[b], (i >> 1) & 1, abort_flag, err)) return false;
    tc::fence_after_sync();
    const uint32_t v_addr = base + L::RING + slot * 32768;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        tc::mma_bf16_ts(tmem + 256, tmem + b * 128 + 8 * k,
                        tc::sdesc_sw128(v_addr + k * 2048, 16384, 1024), id_pv,
                        (i > 0 || k > 0) ? 1u : 0u);
    tc::mma_commit(&o_done[0]);
    if (i == ntl - 1) tc::mma_commit(o_final);
    tc::mma_commit(&rempty[slot]);
    return true;
}

// ---- softmax groups: warps 4-7 own query tile 0, 8-11 tile 1. DB: one query tile, S(i) in
// buffer i % 2 (TMEM columns 128 (i % 2)), each buffer's barriers completing every second tile.
// The two layouts are separate instantiations so each keeps its own register allocation.
template <bool DB>
__device__ __forceinline__ void attn_softmax(const AttnArgs &A, uint32_t tmem, int warp, int lane,
                                             int qbase, int t0, int t1, int ntl, int unit, int sp,
                                             uint64_t *s_full, uint64_t *p_full, uint64_t *o_done,
                                             uint64_t *o_final, volatile int *abort_flag) {
    const int t = DB ? 0 : (warp - 4) >> 2, lg = warp & 3;
    const int r = lg * 32 + lane;
    const int qi = qbase + 128 * t + r;
    const bool valid_row = qi < A.Qu;
    const int rr = qi % A.nq;
    const int nvis = (valid_row && rr < A.w && A.window_causal) ? A.n - A.w + rr + 1 : A.n;
    const int vend = min(t1, nvis);
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const uint32_t o_col = tmem + lane_off + 256 + t * 128;
    float m_used = kNoMax, l = 0.f;  // finite sentinel: exp2(x - kNoMax) = 0
    float m_np = kNoMax;             // true maximum over visible non-protected tokens
    bool ok = true;
    for (int i = 0; i < ntl; ++i) {
        const int sb = DB ? (i & 1) : t;  // S buffer (TMEM columns 128 sb) and its barriers
        const uint32_t s_col = tmem + lane_off + sb * 128;
        if (!tc::mbar_wait_warp(&s_full[sb], DB ? ((i >> 1) & 1) : (i & 1), abort_flag,
                                A.err)) {
            ok = false;
            break;
        }
        tc::fence_after_sync();
        float s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld32(s_col + c * 32, s[c]);
        tc::tmem_wait_ld();
        const int nv_tile = vend - (t0 + i * 128);  // valid columns of this row in the tile
        float mt = -INFINITY;
        if (nv_tile < 128) {  // the tile crosses the end of the split, the unit or a causal window row
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (c * 32 + e >= nv_tile) s[c][e] = -INFINITY;
        }
        {
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 32; e += 2) m4[c] = tc::max3(m4[c], s[c][e], s[c][e + 1]);
            mt = tc::max3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
        }
        {
            // the largest a over non-protected tokens flags queries with peaked pairs; only
            // the tiles holding sink or window tokens (CTA-uniform) need a masked maximum
            const int tbase = t0 + i * 128;
            float mnp = mt;
            if (tbase < A.sink || tbase + 128 > A.n - A.w) {
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int tok = tbase + c * 32 + e;
                        if (tok >= A.sink && tok < A.n - A.w) m4[c] = fmaxf(m4[c], s[c][e]);
                    }
                mnp = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
            m_np = fmaxf(m_np, mnp * A.k1);
        }
        const float m_new = fmaxf(m_used, mt * A.k1);
        // O is rescaled only when the row maximum grew by more than 2^8 (and O holds data)
        const bool rescale = m_new > m_used + kRescaleLog2;
        const float f = (rescale && i > 0) ? tc::ex2_approx(m_used - m_new) : 1.f;
        if (rescale) m_used = m_new;
        const float neg_m = -m_used;
        // p = exp2(s log2e/sqrt(d) - m), packed at once as bf16 pairs: column j of P holds
        // tokens 2j, 2j+1
        const uint64_t k1_2 = tc::pk2(A.k1, A.k1), negm_2 = tc::pk2(neg_m, neg_m);
        uint64_t lsum2[4] = {0, 0, 0, 0};  // bit pattern 0 = (0.f, 0.f)
        float pk[2][32];
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            float t0, t1;
            tc::upk2(tc::fma2(tc::pk2(s[j >> 4][(2 * j) & 31], s[j >> 4][(2 * j + 1) & 31]),
                              k1_2, negm_2),
                     t0, t1);
            const float p0 = tc::ex2_approx(t0), p1 = tc::ex2_approx(t1);
            lsum2[j & 3] = tc::add2(lsum2[j & 3], tc::pk2(p0, p1));
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
            pk[j >> 5][j & 31] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&h2));
        }
        float lsum;
        {
            float a[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) tc::upk2(lsum2[k], a[2 * k], a[2 * k + 1]);
            lsum = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
        }
        l = fmaf(l, f, lsum);
        // tcgen05.ld/st are warp-collective (.sync.aligned): the rescale branch is taken by the
        // whole warp when any of its rows needs it (f = 1 leaves the other rows unchanged)
        if (__any_sync(0xffffffffu, f != 1.f)) {
            // O must hold the previous product before it is rescaled
            if (!tc::mbar_wait_warp(&o_done[t], (i - 1) & 1, abort_flag, A.err)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tc::tmem_ld32(o_col + c * 32, o);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] *= f;
                tc::tmem_st32(o_col + c * 32, o);
            }
        }
        // P row -> TMEM over the first 64 columns of S_t (S_t is in registers; the previous
        // P_t V product completed before S_t(i) was written)
        tc::tmem_st32(s_col, pk[0]);
        tc::tmem_st32(s_col + 32, pk[1]);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::mbar_arrive(&p_full[sb]);
    }
    // warp-uniform condition before the warp-collective TMEM loads
    if (__all_sync(0xffffffffu,
                   ok && (DB ? tc::mbar_wait(o_final, 0, abort_flag, A.err)
                             : tc::mbar_wait(&o_done[t], (ntl - 1) & 1, abort_flag,
                                             A.err)))) {
        tc::fence_after_sync();
        const size_t rowi = ((size_t)unit * A.nsplit + sp) * A.Qu + qi;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float o[32];
            tc::tmem_ld32(o_col + c * 32, o);
            tc::tmem_wait_ld();
            if (valid_row) {
                float4 *dst = reinterpret_cast<float4 *>(A.part_o + rowi * 128 + c * 32);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
            }
        }
        if (valid_row) {
            A.part_ml[rowi] = make_float2(m_used, l);
            A.part_mx[rowi] = m_np;
        }
    }
}

// QT: 128-query tiles per CTA (2: one K/V stream for 256 queries; 1: S double-buffered). With 12
// warps three share a sub-partition's 16K registers (at most 168 a thread), with 8 two (255).
template <int QT>
__global__ void __launch_bounds__(at_threads<QT>(), 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q, AttnArgs A) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    using L = AtLayout<QT>;
    // with one tile per CTA, the CTAs of a (unit, split) are adjacent, so they stream its K/V
    // tiles together and meet in L2
    const int sp = QT == 2 ? blockIdx.x % A.nsplit : (blockIdx.x / A.nqp) % A.nsplit;
    const int qp = QT == 2 ? (blockIdx.x / A.nsplit) % A.nqp : blockIdx.x % A.nqp;
    const int unit = blockIdx.x / (A.nsplit * A.nqp);
    const int t0 = sp * A.split_len, t1 = min(A.n, t0 + A.split_len);
    const int ntl = (t1 - t0 + 127) / 128;
    if (ntl <= 0) return;
    const int qbase = qp * 128 * QT;
    // query tiles with a valid row: with two tiles per CTA, the last CTA of a unit whose queries
    // are not a multiple of 256 holds only one (the planner gives such units one-tile CTAs, but
    // the case is handled); an empty second tile is neither computed nor waited on
    const int nqt = QT == 2 && qbase + 128 < A.Qu ? 2 : 1;

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint64_t *q_full = bars + 0, *rfull = bars + 1, *rempty = bars + 1 + L::SLOTS,
             *s_full = bars + 1 + 2 * L::SLOTS, *p_full = bars + 3 + 2 * L::SLOTS,
             *o_done = bars + 5 + 2 * L::SLOTS, *drain = bars + 7 + 2 * L::SLOTS,
             *o_final = bars + 8 + 2 * L::SLOTS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 9 + 2 * L::SLOTS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 10 + 2 * L::SLOTS);

    if (threadIdx.x == 0) {
        tc::mbar_init(q_full, 1);
        for (int s = 0; s < L::SLOTS; ++s) {
            tc::mbar_init(&rfull[s], 1);
            tc::mbar_init(&rempty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            tc::mbar_init(&s_full[t], 1);
            tc::mbar_init(&p_full[t], 128);
            tc::mbar_init(&o_done[t], 1);
        }
        tc::mbar_init(drain, 1);
        tc::mbar_init(o_final, 1);
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer: Q once, then K_i, V_i through the ring ----
            const int qrow = unit * A.Qu + qbase;
            tc::mbar_expect_tx(q_full, 32768u * nqt);
            for (int t = 0; t < nqt; ++t) {
                tc::tma_load_2d(sm + L::Q + t * 32768, &tm_q, 0, qrow + 128 * t, q_full);
                tc::tma_load_2d(sm + L::Q + t * 32768 + 16384, &tm_q, 64, qrow + 128 * t, q_full);
            }
            int issued = 0;
            for (int c = 0; c < 2 * ntl; ++c) {
                const int slot = c % L::SLOTS;
                const uint32_t ph = (c / L::SLOTS) & 1;
                if (!tc::mbar_wait(&rempty[slot], ph ^ 1, abort_flag, A.err)) break;
                tc::mbar_expect_tx(&rfull[slot], 32768);
                const int row = unit * A.n + t0 + (c >> 1) * 128;
                const CUtensorMap *map = (c & 1) ? &tm_v : &tm_k;
                uint8_t *dst = sm + L::RING + slot * 32768;
                tc::tma_load_2d(dst, map, 0, row, &rfull[slot]);
                tc::tma_load_2d(dst + 16384, map, 64, row, &rfull[slot]);
                issued = c + 1;
            }
            // copies still in flight land before the CTA exits (immediate on the normal path)
            tc::mbar_drain(q_full, 0);
            for (int c = issued - L::SLOTS < 0 ? 0 : issued - L::SLOTS; c < issued; ++c)
                tc::mbar_drain(&rfull[c % L::SLOTS], (c / L::SLOTS) & 1);
        }
    } else if (warp == 1) {
        // ---- MMA issuer. Per K/V tile it submits [P_0 V, S_0 next] then [P_1 V, S_1 next] as
        // blocks, so the tensor pipe serves the two softmax groups in turn and they settle half a
        // cycle apart (one group's exponentials run while the other's products do).
        if (lane == 0 && tc::mbar_wait(q_full, 0, abort_flag, A.err)) {
            const uint32_t base = tc::smem_u32(sm);
            bool ok = true;
            if (nqt == 1) {  // one query tile, S double-buffered
                for (int i = 0; ok && i < 2 && i < ntl; ++i)
                    ok = attn_db_issue_s<QT>(base, tmem, i, rfull, rempty, s_full, abort_flag,
                                             A.err);
                for (int i = 0; ok && i < ntl; ++i) {
                    ok = attn_db_issue_pv<QT>(base, tmem, i, ntl, rfull, rempty, p_full, o_done,
                                              o_final, abort_flag, A.err);
                    if (ok && i + 2 < ntl)
                        ok = attn_db_issue_s<QT>(base, tmem, i + 2, rfull, rempty, s_full,
                                                 abort_flag, A.err);
                }
            }
            for (int t = 0; ok && nqt == 2 && t < nqt; ++t)
                ok = attn_issue_s(base, tmem, t, 0, nqt, rfull, rempty, s_full, abort_flag, A.err);
            for (int i = 0; ok && nqt == 2 && i < ntl; ++i) {
                for (int t = 0; ok && t < nqt; ++t) {
                    ok = attn_issue_pv(base, tmem, t, i, nqt, rfull, rempty, p_full, o_done,
                                       abort_flag, A.err);
                    if (ok && i + 1 < ntl)
                        ok = attn_issue_s(base, tmem, t, i + 1, nqt, rfull, rempty, s_full,
                                          abort_flag, A.err);
                }
            }
        }
        if (lane == 0) {  // every product issued has completed before the tensor memory is freed
            tc::mma_commit(drain);
            tc::mbar_drain(drain, 0);
        }
    } else if (warp >= 4 && ((warp - 4) >> 2) < nqt) {
        if (nqt == 1)
            attn_softmax<true>(A, tmem, warp, lane, qbase, t0, t1, ntl, unit, sp, s_full, p_full,
                               o_done, o_final, abort_flag);
        else
            attn_softmax<false>(A, tmem, warp, lane, qbase, t0, t1, ntl, unit, sp, s_full, p_full,
                                o_done, o_final, abort_flag);
    }
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// One thread waits on an mbarrier that nothing signals, through the same bounded wait the
// kernels above use; the wait gives up after limit_ns and records the timeout.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, unsigned *err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        abort_flag = 0;
        tc::mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, unsigned *err, cudaStream_t st) {
    wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, err);
    return cudaGetLastError();
}

cudaError_t launch_pack_queries(const LorekvDims &D, const void *QW, const void *QL, void *ws,
                                const LorekvWorkspace &W, cudaStream_t st) {
    __nv_bfloat16 *q16 = reinterpret_cast<__nv_bfloat16 *>(static_cast<char *>(ws) + W.q16);
    const long words = (long)D.Qu * (D.d / 8);
    pack_queries_kernel<<<dim3((unsigned)((words + 255) / 256), D.units), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(QW), static_cast<const __nv_bfloat16 *>(QL), D, q16);
    return cudaGetLastError();
}

cudaError_t launch_attention_tc(const LorekvDims &D, const void *K, const void *V, void *ws,
                                const LorekvWorkspace &W, unsigned *err, cudaStream_t st) {
    char *b = static_cast<char *>(ws);
    CUtensorMap tk, tv, tq;
    const uint64_t rows = (uint64_t)D.units * D.n;
    if (!make_tmap_bf16_2d(&tk, K, 128, rows, 64, 128) ||
        !make_tmap_bf16_2d(&tv, V, 128, rows, 64, 128) ||
        !make_tmap_bf16_2d(&tq, b + W.q16, 128, (uint64_t)D.units * D.Qu, 64, 128))
        return cudaErrorInvalidValue;
    AttnArgs A;
    A.n = D.n;
    A.Qu = D.Qu;
    A.nq = D.nq;
    A.w = D.w;
    A.sink = D.sink;
    A.window_causal = D.window_causal;
    A.nsplit = D.nsplit;
    A.split_len = D.split_len;
    const int qt = D.at_qt == 1 ? 1 : 2;
    A.nqp = (D.Qu + 128 * qt - 1) / (128 * qt);
    A.k1 = kLog2e / sqrtf((float)D.d);
    A.part_ml = reinterpret_cast<float2 *>(b + W.part_ml);
    A.part_o = reinterpret_cast<float *>(b + W.part_o);
    A.part_mx = reinterpret_cast<float *>(b + W.part_mx);
    A.err = err;
    auto kern = qt == 1 ? attention_tc_kernel<1> : attention_tc_kernel<2>;
    const size_t smem = qt == 1 ? AtLayout<1>::SMEM : AtLayout<2>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<D.units * A.nqp * D.nsplit, qt == 1 ? at_threads<1>() : at_threads<2>(), smem, st>>>(
        tk, tv, tq, A);
    return cudaGetLastError();
}

cudaError_t launch_scores_tc(const LorekvDims &D, const void *K, const void *V, const float *Lf,
                             void *ws, const LorekvWorkspace &W, float *scores, unsigned *err,
                             cudaStream_t st) {
    char *b = static_cast<char *>(ws);
    __nv_bfloat16 *lt16 = reinterpret_cast<__nv_bfloat16 *>(b + W.lt16);
    const int npairs = (D.g + SC_HPC - 1) / SC_HPC;
    pack_lt_kernel<<<dim3(D.L * D.Hkv * npairs, 8), 256, 0, st>>>(Lf, lt16, D.Hq, D.Hkv, D.g,
                                                                  npairs);
    const long rows_q = (long)D.units * D.Qu;
    pack_qconst_kernel<<<(unsigned)((rows_q + 255) / 256), 256, 0, st>>>(
        reinterpret_cast<const float *>(b + W.lse2), reinterpret_cast<const float *>(b + W.cq),
        reinterpret_cast<const float *>(b + W.wq), reinterpret_cast<const float *>(b + W.amax),
        rows_q, reinterpret_cast<float4 *>(b + W.qconst));
    CUtensorMap tk, tv, tq, tu, tl;
    const uint64_t rows = (uint64_t)D.units * D.n;
    if (!make_tmap_bf16_2d(&tk, K, 128, rows, 64, 128) ||
        !make_tmap_bf16_2d(&tv, V, 128, rows, 64, 128) ||
        !make_tmap_bf16_2d(&tq, b + W.q16, 128, (uint64_t)rows_q, 64, 64) ||
        !make_tmap_bf16_2d(&tu, b + W.u16, 128, (uint64_t)rows_q, 64, 64) ||
        !make_tmap_bf16_2d(&tl, lt16, 128, (uint64_t)D.L * D.Hkv * npairs * 256, 64, 64))
        return cudaErrorInvalidValue;
    ScoresArgs A;
    A.n = D.n;
    A.g = D.g;
    A.Hkv = D.Hkv;
    A.L = D.L;
    A.Hq = D.Hq;
    A.nq = D.nq;
    A.Qu = D.Qu;
    A.sink = D.sink;
    A.w = D.w;
    A.ntiles = (D.n + 127) / 128;
    A.nranges = balance_parts((long)D.units * npairs, A.ntiles, 64, kScSetupTiles);
    A.tpr = (A.ntiles + A.nranges - 1) / A.nranges;
    A.nranges = (A.ntiles + A.tpr - 1) / A.tpr;
    A.eps = D.eps;
    A.k1 = kLog2e / sqrtf((float)D.d);
    A.qconst = reinterpret_cast<const float4 *>(b + W.qconst);
    A.part_s = reinterpret_cast<float *>(b + W.part_s);
    A.pk_cnt = reinterpret_cast<int *>(b + W.pk_cnt);
    A.pk_tok = reinterpret_cast<int *>(b + W.pk_tok);
    A.err = err;
    // the window / trajectory layout of the configured workloads gets compile-time query sets
    const bool fixed_sets = D.w == kSetW && D.M == kSetM && D.T == kSetT;
    auto kern = fixed_sets ? scores_tc_kernel<true> : scores_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SC_SMEM);
    if (e != cudaSuccess) return e;
    kern<<<D.units * A.nranges * npairs, kScThreads, SC_SMEM, st>>>(tk, tv, tq, tu, tl, A);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    reduce_heads_kernel<<<dim3((D.n + 255) / 256, D.units), 256, 0, st>>>(
        A.part_s, D.g, D.n, D.sink, D.w, scores);
    return cudaGetLastError();
}

}  // namespace kve

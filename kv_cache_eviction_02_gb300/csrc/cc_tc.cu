// Counter-causal attention on the tensor cores (review of "Back from the Future: KV Cache Management
// by Counter-Causal Surprise", Section 3.2 step 1: fresh queries over the cached keys and values
// with a strictly upper-triangular mask, so token i attends to the tokens j > i).
//
// cc_attn_tc_kernel: bf16, d_head = 128. The g * ceil(n/128) query tiles of one (sequence, KV
// head) -- 128 positions of one query head each, ordered by position block and then by query head
// -- are taken two at a time by one CTA (both read the same K/V tiles, as the heads of a GQA group
// share them). The CTA streams the 128-token K/V tiles from the first tile's diagonal block to the
// end of the sequence:
//   warp 0       TMA: both Q tiles once, then K_i, V_i through a 5-slot ring of 32 KB;
//   warp 1       one thread issues S_t = Q_t K_i^T (M = N = 128, K = 128) into TMEM, then, once the
//                softmax group has written P_t, O_t += P_t V_i with P read from TMEM (kind::f16);
//   warps 4-11   two softmax groups (one per query tile, one TMEM lane = one query row): mask to
//                i < j < n, online softmax in the log2 domain with the rescale of O deferred until
//                the row maximum grew by more than 2^8, P as bf16 pairs into TMEM; at the end
//                o = O / l is written as fp32, or as bf16 when the tensor-core projection below
//                consumes it.
// Every wait is bounded (tc::mbar_wait), a warp gives up as a whole before warp-collective TMEM
// instructions, and roles drain their copies and products in flight before TMEM is freed.
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace kve {

namespace {

constexpr int kCaThreads = 384;  // TMA, MMA issuer, 2 idle, 2 softmax groups
constexpr int CA_SLOTS = 5;
constexpr uint32_t CA_Q = 0, CA_RING = 65536;  // Q_0, Q_1 | 5 x 32 KB ring (K_0, V_0, K_1, ...)
constexpr uint32_t CA_BAR = CA_RING + CA_SLOTS * 32768;
constexpr size_t CA_SMEM = CA_BAR + 256 + 1024;
constexpr float kCaRescaleLog2 = 8.f;  // rescale O only when a row maximum grows by > 2^8
constexpr float kCaNoMax = -1e30f;     // running maximum before any visible token

struct CcAttnArgs {
    int n, ld, hq, hkv, g, nblk, units;  // units = batch * hkv; ld = token row stride
    float k1;                        // log2(e) / sqrt(d)
    float *O;                        // [batch][n][hq * 128] fp32, or
    __nv_bfloat16 *Ob;               // the same in bf16 (the tensor-core projection's operand)
    unsigned *err;
};

// Query tile t (0, 1) of CTA pair p: position block and query head within the group. The second
// tile of an odd count repeats the first (its rows are computed and discarded).
struct CaTile {
    int blk, hh;
    bool valid;
};
__device__ __forceinline__ CaTile ca_tile(int pair, int t, int g, int nblk) {
    const int q = 2 * pair + t;
    const bool valid = q < g * nblk;
    const int qq = valid ? q : 2 * pair;
    return CaTile{qq / g, qq % g, valid};
}

// S_t = Q_t K_i^T into TMEM columns [128 t, 128 t + 128). Issued after P_t(i-1) V_(i-1) by the same
// thread: MMAs run in issue order, so that product has read P_t (in these columns) first.
__device__ __forceinline__ bool ca_issue_s(uint32_t base, uint32_t tmem, int t, int i,
                                           uint64_t *rfull, uint64_t *rempty, uint64_t *s_full,
                                           volatile int *abort_flag, unsigned *err) {
    constexpr uint32_t id_s = tc::idesc_bf16(128, 128, 0);
    const int c = 2 * i, slot = c % CA_SLOTS;
    if (t == 0 && !tc::mbar_wait(&rfull[slot], (c / CA_SLOTS) & 1, abort_flag, err)) return false;
    tc::fence_after_sync();
    const uint32_t q_addr = base + CA_Q + t * 32768;
    const uint32_t k_addr = base + CA_RING + slot * 32768;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
        tc::mma_bf16(tmem + t * 128, tc::sdesc_sw128(q_addr + o, 16, 1024),
                     tc::sdesc_sw128(k_addr + o, 16, 1024), id_s, k > 0);
    }
    tc::mma_commit(&s_full[t]);
    if (t == 1) tc::mma_commit(&rempty[slot]);  // K_i is done once both tiles used it
    return true;
}

// O_t += P_t V_i: P_t from TMEM (bf16 pairs in the first 64 columns of S_t, 8 columns per 16
// tokens), V_i (ring item 2i+1) as the MN-major B operand.
__device__ __forceinline__ bool ca_issue_pv(uint32_t base, uint32_t tmem, int t, int i,
                                            uint64_t *rfull, uint64_t *rempty, uint64_t *p_full,
                                            uint64_t *o_done, volatile int *abort_flag,
                                            unsigned *err) {
    constexpr uint32_t id_pv = tc::idesc_bf16(128, 128, 1);
    const int c = 2 * i + 1, slot = c % CA_SLOTS;
    if (t == 0 && !tc::mbar_wait(&rfull[slot], (c / CA_SLOTS) & 1, abort_flag, err)) return false;
    if (!tc::mbar_wait(&p_full[t], i & 1, abort_flag, err)) return false;
    tc::fence_after_sync();
    const uint32_t v_addr = base + CA_RING + slot * 32768;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        tc::mma_bf16_ts(tmem + 256 + t * 128, tmem + t * 128 + 8 * k,
                        tc::sdesc_sw128(v_addr + k * 2048, 16384, 1024), id_pv,
                        (i > 0 || k > 0) ? 1u : 0u);
    tc::mma_commit(&o_done[t]);
    if (t == 1) tc::mma_commit(&rempty[slot]);  // V_i is done once both tiles used it
    return true;
}

__global__ void __launch_bounds__(kCaThreads, 1)
    cc_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, CcAttnArgs A) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // pairs with the most key tiles (early position blocks) come first in launch order
    const int unit = blockIdx.x % A.units;  // sequence * hkv + KV head
    const int pair = blockIdx.x / A.units;
    const int b = unit / A.hkv, kh = unit % A.hkv;
    const int kstart = ca_tile(pair, 0, A.g, A.nblk).blk;
    const int ntl = A.nblk - kstart;

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + CA_BAR);
    uint64_t *q_full = bars + 0, *rfull = bars + 1, *rempty = bars + 1 + CA_SLOTS,
             *s_full = bars + 1 + 2 * CA_SLOTS, *p_full = bars + 3 + 2 * CA_SLOTS,
             *o_done = bars + 5 + 2 * CA_SLOTS, *drain = bars + 7 + 2 * CA_SLOTS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 8 + 2 * CA_SLOTS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 9 + 2 * CA_SLOTS);

    if (threadIdx.x == 0) {
        tc::mbar_init(q_full, 1);
        for (int s = 0; s < CA_SLOTS; ++s) {
            tc::mbar_init(&rfull[s], 1);
            tc::mbar_init(&rempty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            tc::mbar_init(&s_full[t], 1);
            tc::mbar_init(&p_full[t], 128);
            tc::mbar_init(&o_done[t], 1);
        }
        tc::mbar_init(drain, 1);
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
        if (lane == 0) {  // ---- TMA producer: Q_0, Q_1 once, then K_i, V_i through the ring ----
            tc::mbar_expect_tx(q_full, 65536);
            for (int t = 0; t < 2; ++t) {
                const CaTile qt = ca_tile(pair, t, A.g, A.nblk);
                const int qrow = (b * A.hq + kh * A.g + qt.hh) * A.ld + qt.blk * 128;
                tc::tma_load_2d(sm + CA_Q + t * 32768, &tm_q, 0, qrow, q_full);
                tc::tma_load_2d(sm + CA_Q + t * 32768 + 16384, &tm_q, 64, qrow, q_full);
            }
            int issued = 0;
            for (int c = 0; c < 2 * ntl; ++c) {
                const int slot = c % CA_SLOTS;
                const uint32_t ph = (c / CA_SLOTS) & 1;
                if (!tc::mbar_wait(&rempty[slot], ph ^ 1, abort_flag, A.err)) break;
                tc::mbar_expect_tx(&rfull[slot], 32768);
                const int row = unit * A.ld + (kstart + (c >> 1)) * 128;
                const CUtensorMap *map = (c & 1) ? &tm_v : &tm_k;
                uint8_t *dst = sm + CA_RING + slot * 32768;
                tc::tma_load_2d(dst, map, 0, row, &rfull[slot]);
                tc::tma_load_2d(dst + 16384, map, 64, row, &rfull[slot]);
                issued = c + 1;
            }
            // copies still in flight land before the CTA exits (immediate on the normal path)
            tc::mbar_drain(q_full, 0);
            for (int c = issued - CA_SLOTS < 0 ? 0 : issued - CA_SLOTS; c < issued; ++c)
                tc::mbar_drain(&rfull[c % CA_SLOTS], (c / CA_SLOTS) & 1);
        }
    } else if (warp == 1) {
        // ---- MMA issuer: per K/V tile [P_0 V, S_0 next] then [P_1 V, S_1 next], so the two
        // softmax groups alternate with the tensor pipe
        if (lane == 0 && tc::mbar_wait(q_full, 0, abort_flag, A.err)) {
            const uint32_t base = tc::smem_u32(sm);
            bool ok = ca_issue_s(base, tmem, 0, 0, rfull, rempty, s_full, abort_flag, A.err) &&
                      ca_issue_s(base, tmem, 1, 0, rfull, rempty, s_full, abort_flag, A.err);
            for (int i = 0; ok && i < ntl; ++i) {
                for (int t = 0; ok && t < 2; ++t) {
                    ok = ca_issue_pv(base, tmem, t, i, rfull, rempty, p_full, o_done, abort_flag,
                                     A.err);
                    if (ok && i + 1 < ntl)
                        ok = ca_issue_s(base, tmem, t, i + 1, rfull, rempty, s_full, abort_flag,
                                        A.err);
                }
            }
        }
        if (lane == 0) {  // every product issued has completed before the tensor memory is freed
            tc::mma_commit(drain);
            tc::mbar_drain(drain, 0);
        }
    } else if (warp >= 4) {  // ---- softmax groups: warps 4-7 own query tile 0, 8-11 tile 1 ----
        const int t = (warp - 4) >> 2, lg = warp & 3;
        const CaTile qt = ca_tile(pair, t, A.g, A.nblk);
        const int r = lg * 32 + lane;
        const int i = qt.blk * 128 + r;  // this row's position
        const bool valid_row = qt.valid && i < A.n;
        const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
        const uint32_t s_col = tmem + lane_off + t * 128;
        const uint32_t o_col = tmem + lane_off + 256 + t * 128;
        float m_used = kCaNoMax, l = 0.f;  // finite sentinel: exp2(x - kCaNoMax) = 0
        bool ok = true;
        for (int it = 0; it < ntl; ++it) {
            if (!tc::mbar_wait_warp(&s_full[t], it & 1, abort_flag, A.err)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            float s[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tc::tmem_ld32(s_col + c * 32, s[c]);
            tc::tmem_wait_ld();
            // visible columns of this tile: jb + col in (i, n)
            const int jb = (kstart + it) * 128;
            const int lo = i - jb, hi = A.n - jb;
            if (lo >= 0 || hi < 128) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (c * 32 + e <= lo || c * 32 + e >= hi) s[c][e] = -INFINITY;
            }
            float mt;
            {
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) m4[c] = tc::max3(m4[c], s[c][e], s[c][e + 1]);
                mt = tc::max3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
            }
            const float m_new = fmaxf(m_used, mt * A.k1);
            const bool rescale = m_new > m_used + kCaRescaleLog2;
            const float f = (rescale && it > 0) ? tc::ex2_approx(m_used - m_new) : 1.f;
            if (rescale) m_used = m_new;
            const float neg_m = -m_used;
            const uint64_t k1_2 = tc::pk2(A.k1, A.k1), negm_2 = tc::pk2(neg_m, neg_m);
            uint64_t lsum2[4] = {0, 0, 0, 0};
            float pk[2][32];
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                float x0, x1;
                tc::upk2(tc::fma2(tc::pk2(s[j >> 4][(2 * j) & 31], s[j >> 4][(2 * j + 1) & 31]),
                                  k1_2, negm_2),
                         x0, x1);
                const float p0 = tc::ex2_approx(x0), p1 = tc::ex2_approx(x1);
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
            // warp-collective TMEM access: the whole warp rescales when any row needs it
            if (__any_sync(0xffffffffu, f != 1.f)) {
                if (!tc::mbar_wait_warp(&o_done[t], (it - 1) & 1, abort_flag, A.err)) {
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
            tc::tmem_st32(s_col, pk[0]);
            tc::tmem_st32(s_col + 32, pk[1]);
            tc::tmem_wait_st();
            tc::fence_before_sync();
            tc::mbar_arrive(&p_full[t]);
        }
        if (__all_sync(0xffffffffu,
                       ok && tc::mbar_wait(&o_done[t], (ntl - 1) & 1, abort_flag, A.err))) {
            tc::fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;  // the last token sees no key: o = 0
            const size_t off = ((size_t)(b * A.ld + i) * A.hq + kh * A.g + qt.hh) * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tc::tmem_ld32(o_col + c * 32, o);
                tc::tmem_wait_ld();
                if (valid_row && A.Ob) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(A.Ob + off + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const __nv_bfloat162 h2 = __floats2bfloat162_rn(
                                o[8 * e + 2 * k] * inv, o[8 * e + 2 * k + 1] * inv);
                            w[k] = *reinterpret_cast<const uint32_t *>(&h2);
                        }
                        d4[e] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else if (valid_row) {
                    float4 *d4 = reinterpret_cast<float4 *>(A.O + off + c * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        d4[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv,
                                            o[4 * e + 2] * inv, o[4 * e + 3] * inv);
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ---- r = h + W_O o and the true token's logit, on the tensor cores -------------------------------
//
// cc_logits_tc_kernel: CTA tile of 128 tokens x 256 output columns m of d_model; the K loop runs
// over o's H_q * 128 entries in steps of 64 (one 128-byte-swizzled TMA box of each operand per
// step, 4-stage ring), one thread issues D += O W_O^T (M = 128, N = 256, K = 16 per instruction)
// into 256 TMEM columns. The logit is linear in r, so the K loop may be split over CTAs: each split
// contributes sum_m W_U[x_t][m] (its part of W_O o)_m, the first one also adds h. Epilogue: warps
// 2-9, one TMEM lane (token) and 128 columns each, write one partial logit per (column tile,
// split, column half); a fixed-order sum of the partials gives the logit.
constexpr int kLgThreads = 320;  // TMA, MMA issuer, 8 epilogue warps
constexpr int LG_STAGES = 4;
constexpr uint32_t LG_A = 16384, LG_STAGE = LG_A + 32768;  // O: 128 x 64, W_O: 256 x 64 (bf16)
constexpr uint32_t LG_BAR = LG_STAGES * LG_STAGE;
constexpr size_t LG_SMEM = LG_BAR + 256 + 1024;

struct CcLogitsArgs {
    int n, ld, dm, vocab, mtiles, ntiles, ksplit, ksteps, ksteps_per;
    const __nv_bfloat16 *H, *W_U;
    const int32_t *X;
    float *part;  // [batch][ntiles * ksplit * 2][n]
    unsigned *err;
};

__global__ void __launch_bounds__(kLgThreads, 1)
    cc_logits_tc_kernel(const __grid_constant__ CUtensorMap tm_o,
                        const __grid_constant__ CUtensorMap tm_w, CcLogitsArgs A) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int bx = blockIdx.x;
    const int ks = bx % A.ksplit;
    bx /= A.ksplit;
    const int mt = bx % A.mtiles;
    bx /= A.mtiles;
    const int nt = bx % A.ntiles;
    const int b = bx / A.ntiles;
    const int kb = ks * A.ksteps_per;
    const int nk = min(A.ksteps, kb + A.ksteps_per) - kb;  // >= 1 (host sizes the splits)
    const int m0 = mt * 128, n0 = nt * 256;

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + LG_BAR);
    uint64_t *full = bars, *empty = bars + LG_STAGES, *acc_full = bars + 2 * LG_STAGES,
             *drain = bars + 2 * LG_STAGES + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * LG_STAGES + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * LG_STAGES + 3);
    if (threadIdx.x == 0) {
        for (int s = 0; s < LG_STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(acc_full, 1);
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 256);
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer ----
            int issued = 0;
            for (int s = 0; s < nk; ++s) {
                const int slot = s % LG_STAGES;
                if (!tc::mbar_wait(&empty[slot], ((s / LG_STAGES) & 1) ^ 1, abort_flag, A.err))
                    break;
                tc::mbar_expect_tx(&full[slot], LG_STAGE);
                uint8_t *dst = sm + slot * LG_STAGE;
                const int x = (kb + s) * 64;
                tc::tma_load_2d(dst, &tm_o, x, b * A.ld + m0, &full[slot]);
                tc::tma_load_2d(dst + LG_A, &tm_w, x, n0, &full[slot]);
                issued = s + 1;
            }
            for (int s = issued - LG_STAGES < 0 ? 0 : issued - LG_STAGES; s < issued; ++s)
                tc::mbar_drain(&full[s % LG_STAGES], (s / LG_STAGES) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---- MMA issuer ----
            constexpr uint32_t id = tc::idesc_bf16(128, 256, 0);
            const uint32_t base = tc::smem_u32(sm);
            bool ok = true;
            for (int s = 0; s < nk; ++s) {
                const int slot = s % LG_STAGES;
                if (!tc::mbar_wait(&full[slot], (s / LG_STAGES) & 1, abort_flag, A.err)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a = base + slot * LG_STAGE, w = a + LG_A;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tc::mma_bf16(tmem, tc::sdesc_sw128(a + k * 32, 16, 1024),
                                 tc::sdesc_sw128(w + k * 32, 16, 1024), id, (s > 0 || k > 0));
                tc::mma_commit(&empty[slot]);
            }
            if (ok) tc::mma_commit(acc_full);
            tc::mma_commit(drain);  // every product issued has completed before TMEM is freed
            tc::mbar_drain(drain, 0);
        }
    } else {  // ---- epilogue: warps 2-9 ----
        const int lg = warp & 3, half = (warp - 2) >> 2;
        const int t = m0 + lg * 32 + lane;
        const bool valid = t < A.n;
        int x = 0;
        if (valid) {
            x = A.X[(size_t)b * A.ld + t];
            if (x < 0 || x >= A.vocab) {  // reported, and the row read as token 0
                if (A.err) atomicOr(A.err, KVE_DEVERR_BADINDEX);
                x = 0;
            }
        }
        if (tc::mbar_wait_warp(acc_full, 0, abort_flag, A.err)) {
            tc::fence_after_sync();
            const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
            const __nv_bfloat16 *wu = A.W_U + (size_t)x * A.dm;
            const __nv_bfloat16 *hr = A.H + ((size_t)b * A.ld + (valid ? t : 0)) * A.dm;
            float z = 0.f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                const int col = half * 128 + c * 32;
                float acc[32];
                tc::tmem_ld32(tmem + lane_off + col, acc);
                tc::tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        const int m = n0 + col + e;
                        if (m < A.dm) {  // d_model is a multiple of 8
                            const uint4 wv = *reinterpret_cast<const uint4 *>(wu + m);
                            uint4 hv = make_uint4(0u, 0u, 0u, 0u);
                            if (ks == 0) hv = *reinterpret_cast<const uint4 *>(hr + m);
                            const __nv_bfloat162 *w2 = reinterpret_cast<const __nv_bfloat162 *>(&wv);
                            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&hv);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float2 wf = __bfloat1622float2(w2[k]);
                                const float2 hf = __bfloat1622float2(h2[k]);
                                z = fmaf(wf.x, acc[e + 2 * k] + hf.x, z);
                                z = fmaf(wf.y, acc[e + 2 * k + 1] + hf.y, z);
                            }
                        }
                    }
                }
            }
            if (valid)
                A.part[((size_t)b * (A.ntiles * A.ksplit * 2) + (nt * A.ksplit + ks) * 2 + half) *
                           A.ld + t] = z;
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 256);
    }
}

}  // namespace

int cc_logits_tc_split(const CcDims &D) {
    const long ctas = (long)D.batch * ((D.n + 127) / 128) * ((D.dm + 255) / 256);
    const int ksteps = D.hq * D.d / 64;
    int best = 1;
    long best_cost = -1;
    for (int p = 1; p <= kCcMaxKSplit && p <= ksteps; ++p) {
        const int per = (ksteps + p - 1) / p;
        const int used = (ksteps + per - 1) / per;  // splits that get at least one step
        const long cost = ((ctas * used + 151) / 152) * per;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = used;
        }
    }
    return best;
}

bool cc_logits_tc_supported(const CcDims &D) {
    return cc_attention_tc_supported(D) && D.dm % 8 == 0;
}

cudaError_t launch_cc_logits_tc(const CcDims &D, const __nv_bfloat16 *Ob, const void *H,
                                const void *W_O, const void *W_U, const int32_t *X, float *part,
                                int ksplit, unsigned *err, cudaStream_t st) {
    const int kdim = D.hq * D.d;
    CUtensorMap to, tw;
    if (!make_tmap_bf16_2d(&to, Ob, kdim, (uint64_t)D.batch * D.ld, 64, 128) ||
        !make_tmap_bf16_2d(&tw, W_O, kdim, D.dm, 64, 256))
        return cudaErrorInvalidValue;
    CcLogitsArgs A;
    A.n = D.n;
    A.ld = D.ld;
    A.dm = D.dm;
    A.vocab = D.vocab;
    A.mtiles = (D.n + 127) / 128;
    A.ntiles = (D.dm + 255) / 256;
    A.ksteps = kdim / 64;
    A.ksteps_per = (A.ksteps + ksplit - 1) / ksplit;
    A.ksplit = (A.ksteps + A.ksteps_per - 1) / A.ksteps_per;
    A.H = static_cast<const __nv_bfloat16 *>(H);
    A.W_U = static_cast<const __nv_bfloat16 *>(W_U);
    A.X = X;
    A.part = part;
    A.err = err;
    const long grid = (long)D.batch * A.mtiles * A.ntiles * A.ksplit;
    if (grid > 0x7fffffffL) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(cc_logits_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LG_SMEM);
    if (e != cudaSuccess) return e;
    cc_logits_tc_kernel<<<(unsigned)grid, kLgThreads, LG_SMEM, st>>>(to, tw, A);
    return cudaGetLastError();
}

bool cc_attention_tc_supported(const CcDims &D) {
    return D.dtype == KVE_BF16 && D.d == 128 && (long)D.batch * D.hkv * D.ld >= 128;
}

cudaError_t launch_cc_attention_tc(const CcDims &D, const void *K, const void *V, const void *Q,
                                   float *O, __nv_bfloat16 *Ob, unsigned *err, cudaStream_t st) {
    CUtensorMap tk, tv, tq;
    const uint64_t kv_rows = (uint64_t)D.batch * D.hkv * D.ld;
    const uint64_t q_rows = (uint64_t)D.batch * D.hq * D.ld;
    if (!make_tmap_bf16_2d(&tk, K, 128, kv_rows, 64, 128) ||
        !make_tmap_bf16_2d(&tv, V, 128, kv_rows, 64, 128) ||
        !make_tmap_bf16_2d(&tq, Q, 128, q_rows, 64, 128))
        return cudaErrorInvalidValue;
    CcAttnArgs A;
    A.n = D.n;
    A.ld = D.ld;
    A.hq = D.hq;
    A.hkv = D.hkv;
    A.g = D.hq / D.hkv;
    A.nblk = (D.n + 127) / 128;
    A.units = D.batch * D.hkv;
    A.k1 = kLog2e / sqrtf(128.f);
    A.O = O;
    A.Ob = Ob;
    A.err = err;
    const long pairs = ((long)A.g * A.nblk + 1) / 2;
    const long grid = pairs * A.units;
    if (grid > 0x7fffffffL) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(cc_attn_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CA_SMEM);
    if (e != cudaSuccess) return e;
    cc_attn_tc_kernel<<<(unsigned)grid, kCaThreads, CA_SMEM, st>>>(tk, tv, tq, A);
    return cudaGetLastError();
}

}  // namespace kve

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
//                o = O / l is written as fp32.
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
    int n, hq, hkv, g, nblk, units;  // units = batch * hkv
    float k1;                        // log2(e) / sqrt(d)
    float *O;                        // [batch][n][hq * 128] fp32
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
                const int qrow = (b * A.hq + kh * A.g + qt.hh) * A.n + qt.blk * 128;
                tc::tma_load_2d(sm + CA_Q + t * 32768, &tm_q, 0, qrow, q_full);
                tc::tma_load_2d(sm + CA_Q + t * 32768 + 16384, &tm_q, 64, qrow, q_full);
            }
            int issued = 0;
            for (int c = 0; c < 2 * ntl; ++c) {
                const int slot = c % CA_SLOTS;
                const uint32_t ph = (c / CA_SLOTS) & 1;
                if (!tc::mbar_wait(&rempty[slot], ph ^ 1, abort_flag, A.err)) break;
                tc::mbar_expect_tx(&rfull[slot], 32768);
                const int row = unit * A.n + (kstart + (c >> 1)) * 128;
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
            float *dst = A.O + ((size_t)(b * A.n + i) * A.hq + kh * A.g + qt.hh) * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tc::tmem_ld32(o_col + c * 32, o);
                tc::tmem_wait_ld();
                if (valid_row) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
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

}  // namespace

bool cc_attention_tc_supported(const CcDims &D) {
    return D.dtype == KVE_BF16 && D.d == 128 && (long)D.batch * D.hkv * D.n >= 128;
}

cudaError_t launch_cc_attention_tc(const CcDims &D, const void *K, const void *V, const void *Q,
                                   float *O, unsigned *err, cudaStream_t st) {
    CUtensorMap tk, tv, tq;
    const uint64_t kv_rows = (uint64_t)D.batch * D.hkv * D.n;
    const uint64_t q_rows = (uint64_t)D.batch * D.hq * D.n;
    if (!make_tmap_bf16_2d(&tk, K, 128, kv_rows, 64, 128) ||
        !make_tmap_bf16_2d(&tv, V, 128, kv_rows, 64, 128) ||
        !make_tmap_bf16_2d(&tq, Q, 128, q_rows, 64, 128))
        return cudaErrorInvalidValue;
    CcAttnArgs A;
    A.n = D.n;
    A.hq = D.hq;
    A.hkv = D.hkv;
    A.g = D.hq / D.hkv;
    A.nblk = (D.n + 127) / 128;
    A.units = D.batch * D.hkv;
    A.k1 = kLog2e / sqrtf(128.f);
    A.O = O;
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

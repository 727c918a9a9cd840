// H2O prefill scores on the 5th-generation tensor cores (tcgen05, sm_103a): f16 or bf16 inputs,
// fp32 TMEM accumulators, TMA-staged 128-byte-swizzled tiles.
//
// H2O summary, Section 4.1 (the prompt handled as one block): for every (batch, layer, head)
// unit, acc_j = sum over prompt queries i >= j of softmax_i(q_i . K_{<=i} / sqrt d)_j. The prompt
// is cut into 128-token tiles; query tile r is processed in two phases that share its Q tile:
//   1. S = Q_r K_b^T for the key tiles b <= r, queries on TMEM lanes: the thread of query q keeps
//      an online maximum and normaliser over its row, giving lse2_q (the log2 of the softmax
//      denominator of q, in units of s log2e / sqrt d).
//   2. S^T = K_b Q_r^T for the same key tiles, keys on TMEM lanes: the thread of key j adds
//      exp2(s log2e / sqrt d - lse2_q) over the tile's queries q >= j.
// The unit's K tiles stay in shared memory while its query tiles run in descending order, so key
// tile r is last used by query tile r and the next unit's K tiles stream into the slots as they
// are released; Q tiles are double-buffered. One persistent CTA per SM walks the units.
// Roles: warp 0 TMA producer, warp 1 MMA issuer (one thread), warps 2-9 the lane owners: warp w
// reads TMEM lanes 32 (w % 4) .. +31, warps 2-5 columns 0-63 and warps 6-9 columns 64-127 of every
// block (the two halves' row statistics are merged between the phases). Causal and prompt masks
// are decided per warp and 32-column half (every column visible, none, or per element). TMEM:
// four 128-column slots, one 128 x 128 block each.
#include "tc_common.cuh"

namespace kve {

namespace {

constexpr int kHpThreads = 320;
constexpr int HP_KSLOTS = 5, HP_QSLOTS = 2, HP_TSLOTS = 4;
constexpr int kHpMaxTiles = HP_KSLOTS;  // a unit's K tiles must fit in the ring at once
constexpr uint32_t HP_K = 0;
constexpr uint32_t HP_Q = HP_K + HP_KSLOTS * 32768;
constexpr uint32_t HP_ML = HP_Q + HP_QSLOTS * 32768;   // [128] float2: (m, l) of column half 1
constexpr uint32_t HP_LSE = HP_ML + 128 * 8;           // [128] f32: -lse2 of the tile's queries
constexpr uint32_t HP_BAR = HP_LSE + 128 * 4;
constexpr size_t HP_SMEM = HP_BAR + 256 + 1024;
constexpr float kNoMax = -1e30f;

struct ColsumArgs {
    int units, P, nt;
    int ab_bf16;
    float k1;  // log2(e) / sqrt(d)
    float *acc;
    unsigned *err;
};

// 64 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void load_half(uint32_t taddr, float (&v)[64]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float t[32];
        tc::tmem_ld32(taddr + 32 * h, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * h + i] = t[i];
    }
    tc::tmem_wait_ld();
}

// How the 32 columns of one half of a lane owner's 64-column block slice are treated, decided
// per warp from the causal and prompt limits of its 32 rows: every column visible to every row,
// visibility decided per element, or no column visible to any row.
enum : int { kColAll = 0, kColMask = 1, kColNone = 2 };

// Phase 1 on one block: the row's running maximum m and sum l (log2 domain) take the visible
// key columns c <= lim of v; H0 and H1 are the modes of columns 0-31 and 32-63. Every mode
// gives the values of the per-element test (skipped columns add the maximum's identity and +0).
template <int H0, int H1>
__device__ __forceinline__ void p1_block(const float (&v)[64], int lim, float k1, uint64_t k1_2,
                                         float &m, float &l) {
    float m4[4] = {kNoMax, kNoMax, kNoMax, kNoMax};
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
        const int mode = c < 32 ? H0 : H1;
        if (mode == kColNone) continue;
        const float a = (mode == kColAll || c <= lim) ? v[c] : kNoMax;
        const float b = (mode == kColAll || c + 1 <= lim) ? v[c + 1] : kNoMax;
        m4[(c >> 1) & 3] = tc::max3(m4[(c >> 1) & 3], a, b);
    }
    const float mx = tc::max3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
    const float mn = fmaxf(m, mx);
    const float nmk = -mn * k1;
    const uint64_t nmk_2 = tc::pk2(nmk, nmk);
    uint64_t s2[4] = {0, 0, 0, 0};  // bit pattern 0 = (0.f, 0.f)
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
        const int mode = c < 32 ? H0 : H1;
        if (mode == kColNone) continue;
        float ta, tb;
        tc::upk2(tc::fma2(tc::pk2(v[c], v[c + 1]), k1_2, nmk_2), ta, tb);
        float ea = tc::ex2_approx(ta), eb = tc::ex2_approx(tb);
        if (mode == kColMask) {
            ea = c <= lim ? ea : 0.f;
            eb = c + 1 <= lim ? eb : 0.f;
        }
        s2[(c >> 1) & 3] = tc::add2(s2[(c >> 1) & 3], tc::pk2(ea, eb));
    }
    float bs = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float a, bb;
        tc::upk2(s2[k], a, bb);
        bs += a + bb;
    }
    // a half may see no valid column yet (m stays kNoMax, l 0): the merge of the halves
    // weights it by 2^(-huge) = 0
    l = l * tc::ex2_approx((m - mn) * k1) + bs;
    m = mn;
}

// Phase 2 on one block: the key row's sum of 2^(s k1 - lse2) over the visible query columns
// lo <= c <= qmax of v (-lse2 of column c in nlse4); H0, H1 as in p1_block.
template <int H0, int H1>
__device__ __forceinline__ float p2_block(const float (&v)[64], const float4 *nlse4, int lo,
                                          int qmax, uint64_t k1_2) {
    uint64_t s2[4] = {0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
        const int mode = c < 32 ? H0 : H1;
        if (mode == kColNone) continue;
        const float4 nl = nlse4[c >> 2];
        float ta, tb, tc_, td;
        tc::upk2(tc::fma2(tc::pk2(v[c], v[c + 1]), k1_2, tc::pk2(nl.x, nl.y)), ta, tb);
        tc::upk2(tc::fma2(tc::pk2(v[c + 2], v[c + 3]), k1_2, tc::pk2(nl.z, nl.w)), tc_, td);
        float ea = tc::ex2_approx(ta), eb = tc::ex2_approx(tb);
        float ec = tc::ex2_approx(tc_), ed = tc::ex2_approx(td);
        if (mode == kColMask) {
            ea = (c >= lo && c <= qmax) ? ea : 0.f;
            eb = (c + 1 >= lo && c + 1 <= qmax) ? eb : 0.f;
            ec = (c + 2 >= lo && c + 2 <= qmax) ? ec : 0.f;
            ed = (c + 3 >= lo && c + 3 <= qmax) ? ed : 0.f;
        }
        s2[(c >> 2) & 1] = tc::add2(s2[(c >> 2) & 1], tc::pk2(ea, eb));
        s2[2 + ((c >> 2) & 1)] = tc::add2(s2[2 + ((c >> 2) & 1)], tc::pk2(ec, ed));
    }
    float bs = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float a, bb;
        tc::upk2(s2[k], a, bb);
        bs += a + bb;
    }
    return bs;
}

__global__ void __launch_bounds__(kHpThreads, 1)
    h2o_colsum_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_q, ColsumArgs A) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt = A.nt;

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + HP_BAR);
    uint64_t *kfull = bars, *kempty = bars + HP_KSLOTS;
    uint64_t *qfull = bars + 2 * HP_KSLOTS, *qempty = qfull + HP_QSLOTS;
    uint64_t *tfull = qempty + HP_QSLOTS, *tempty = tfull + HP_TSLOTS;
    uint64_t *lsef = tempty + HP_TSLOTS, *lsef2 = lsef + 1, *drain = lsef + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(lsef + 3);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(lsef + 4);
    float2 *ml_s = reinterpret_cast<float2 *>(sm + HP_ML);
    float *lse_s = reinterpret_cast<float *>(sm + HP_LSE);

    if (threadIdx.x == 0) {
        for (int i = 0; i < HP_KSLOTS; ++i) {
            tc::mbar_init(&kfull[i], 1);
            tc::mbar_init(&kempty[i], 1);
        }
        for (int i = 0; i < HP_QSLOTS; ++i) {
            tc::mbar_init(&qfull[i], 1);
            tc::mbar_init(&qempty[i], 1);
        }
        for (int i = 0; i < HP_TSLOTS; ++i) {
            tc::mbar_init(&tfull[i], 1);
            tc::mbar_init(&tempty[i], 8);  // one arrival per lane-owner warp
        }
        tc::mbar_init(lsef, 8);
        tc::mbar_init(lsef2, 8);
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
        if (lane == 0) {  // ---- TMA producer: per unit Q_{nt-1}, K_{nt-1..0}, Q_{nt-2}, ..., Q_0 ----
            tc::tma_prefetch_desc(&tm_k);
            tc::tma_prefetch_desc(&tm_q);
            int kc = 0, qc = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < A.units && ok; unit += gridDim.x) {
                const int row0 = unit * A.P;
                for (int r = nt - 1; r >= 0 && ok; --r) {
                    {
                        const int sl = qc % HP_QSLOTS;
                        if (!tc::mbar_wait(&qempty[sl], ((qc / HP_QSLOTS) & 1) ^ 1, abort_flag,
                                           A.err)) {
                            ok = false;
                            break;
                        }
                        tc::mbar_expect_tx(&qfull[sl], 32768);
                        uint8_t *dst = sm + HP_Q + sl * 32768;
                        tc::tma_load_2d(dst, &tm_q, 0, row0 + 128 * r, &qfull[sl]);
                        tc::tma_load_2d(dst + 16384, &tm_q, 64, row0 + 128 * r, &qfull[sl]);
                        ++qc;
                    }
                    if (r == nt - 1) {
                        for (int b = nt - 1; b >= 0; --b) {
                            const int sl = kc % HP_KSLOTS;
                            if (!tc::mbar_wait(&kempty[sl], ((kc / HP_KSLOTS) & 1) ^ 1,
                                               abort_flag, A.err)) {
                                ok = false;
                                break;
                            }
                            tc::mbar_expect_tx(&kfull[sl], 32768);
                            uint8_t *dst = sm + HP_K + sl * 32768;
                            tc::tma_load_2d(dst, &tm_k, 0, row0 + 128 * b, &kfull[sl]);
                            tc::tma_load_2d(dst + 16384, &tm_k, 64, row0 + 128 * b, &kfull[sl]);
                            ++kc;
                        }
                    }
                }
            }
            // copies still in flight land before the CTA exits (immediate on the normal path)
            for (int c = kc - HP_KSLOTS < 0 ? 0 : kc - HP_KSLOTS; c < kc; ++c)
                tc::mbar_drain(&kfull[c % HP_KSLOTS], (c / HP_KSLOTS) & 1);
            for (int c = qc - HP_QSLOTS < 0 ? 0 : qc - HP_QSLOTS; c < qc; ++c)
                tc::mbar_drain(&qfull[c % HP_QSLOTS], (c / HP_QSLOTS) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---- MMA issuer ----
            const uint32_t k_base = tc::smem_u32(sm + HP_K), q_base = tc::smem_u32(sm + HP_Q);
            const uint32_t idesc = tc::idesc_f16kind(128, 128, 0, A.ab_bf16);
            int kc = 0, qc = 0, tcn = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < A.units && ok; unit += gridDim.x) {
                const int kbase = kc;  // K_b of this unit is ring item kbase + (nt - 1 - b)
                kc += nt;
                for (int r = nt - 1; r >= 0 && ok; --r) {
                    const int qs = qc % HP_QSLOTS;
                    if (!tc::mbar_wait(&qfull[qs], (qc / HP_QSLOTS) & 1, abort_flag, A.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t q_addr = q_base + qs * 32768;
                    for (int ph = 0; ph < 2 && ok; ++ph) {
                        for (int b = r; b >= 0; --b) {
                            const int kidx = kbase + (nt - 1 - b);
                            const int ks = kidx % HP_KSLOTS;
                            if (ph == 0 && r == nt - 1 &&
                                !tc::mbar_wait(&kfull[ks], (kidx / HP_KSLOTS) & 1, abort_flag,
                                               A.err)) {
                                ok = false;
                                break;
                            }
                            const int ts = tcn % HP_TSLOTS;
                            if (!tc::mbar_wait(&tempty[ts], ((tcn / HP_TSLOTS) & 1) ^ 1,
                                               abort_flag, A.err)) {
                                ok = false;
                                break;
                            }
                            tc::fence_after_sync();
                            const uint32_t k_addr = k_base + ks * 32768;
                            // phase 0: D[query][key] = Q_r K_b^T; phase 1: D[key][query] = K_b Q_r^T
                            const uint32_t a_addr = ph == 0 ? q_addr : k_addr;
                            const uint32_t b_addr = ph == 0 ? k_addr : q_addr;
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const uint32_t o = (k >> 2) * 16384 + (k & 3) * 32;
                                tc::mma_bf16(tmem + ts * 128, tc::sdesc_sw128(a_addr + o, 16, 1024),
                                             tc::sdesc_sw128(b_addr + o, 16, 1024), idesc, k > 0);
                            }
                            tc::mma_commit(&tfull[ts]);
                            ++tcn;
                            if (ph == 1 && b == r) tc::mma_commit(&kempty[ks]);  // K_r done
                        }
                    }
                    if (!ok) break;
                    tc::mma_commit(&qempty[qs]);
                    ++qc;
                }
            }
        }
        if (lane == 0) {  // every product issued has completed before the tensor memory is freed
            tc::mma_commit(drain);
            tc::mbar_drain(drain, 0);
        }
    } else {
        // ---- lane owners: warp w reads TMEM lanes 32 (w % 4) .. +31, columns 64 hf .. +63 of
        // every block (hf = 0 for warps 2-5, 1 for warps 6-9) ----
        const int row = (warp & 3) * 32 + lane;
        const int hf = (warp - 2) >> 2;
        const uint32_t tcol = (uint32_t)(64 * hf) + ((uint32_t)((warp & 3) * 32) << 16);
        const float k1 = A.k1;
        const uint64_t k1_2 = tc::pk2(k1, k1);
        int tcn = 0, lcn = 0;
        bool ok = true;
        for (int unit = blockIdx.x; unit < A.units && ok; unit += gridDim.x) {
            float *accu = A.acc + ((size_t)unit * 2 + hf) * A.P;  // this half's partial sums
            float accb[kHpMaxTiles];  // running sums of key rows 128 b + row
#pragma unroll
            for (int b = 0; b < kHpMaxTiles; ++b) accb[b] = 0.f;
            for (int r = nt - 1; r >= 0 && ok; --r) {
                // phase 1: online softmax statistics of query row q = 128 r + row over this
                // half's key columns
                const int q = 128 * r + row;
                float m = kNoMax, l = 0.f;
                for (int b = r; b >= 0; --b) {
                    const int ts = tcn % HP_TSLOTS;
                    if (!tc::mbar_wait_warp(&tfull[ts], (tcn / HP_TSLOTS) & 1, abort_flag, A.err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    // key column c of this half valid iff c <= lim; the warp's rows 32 lg .. +31
                    // span lim_lo .. lim_hi (warp-uniform)
                    const int lim = min(q - 128 * b, A.P - 1 - 128 * b) - 64 * hf;
                    const int qb = 128 * (r - b) + (warp & 3) * 32, plim = A.P - 1 - 128 * b;
                    const int lim_lo = min(qb, plim) - 64 * hf, lim_hi = min(qb + 31, plim) - 64 * hf;
                    if (lim_hi < 0) {  // no column of this half is visible to the warp's rows
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&tempty[ts]);
                        ++tcn;
                        continue;
                    }
                    float v[64];
                    load_half(tmem + tcol + ts * 128, v);
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&tempty[ts]);
                    ++tcn;
                    if (lim_lo >= 63)
                        p1_block<kColAll, kColAll>(v, lim, k1, k1_2, m, l);
                    else if (lim_lo == 0 && lim_hi == 31)
                        p1_block<kColMask, kColNone>(v, lim, k1, k1_2, m, l);
                    else if (lim_lo == 32 && lim_hi == 63)
                        p1_block<kColAll, kColMask>(v, lim, k1, k1_2, m, l);
                    else
                        p1_block<kColMask, kColMask>(v, lim, k1, k1_2, m, l);
                }
                if (!ok) break;
                // merge the halves: half 1 hands (m, l) over, half 0 writes lse2 of the row
                if (hf == 1) ml_s[row] = make_float2(m, l);
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(lsef);
                if (!tc::mbar_wait_warp(lsef, lcn & 1, abort_flag, A.err)) {
                    ok = false;
                    break;
                }
                if (hf == 0) {
                    const float2 o = ml_s[row];
                    const float mm = fmaxf(m, o.x);
                    const float ll = l * tc::ex2_approx((m - mm) * k1) +
                                     o.y * tc::ex2_approx((o.x - mm) * k1);
                    lse_s[row] = -(mm * k1 + __log2f(ll));  // -lse2 of query row q
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(lsef2);
                if (!tc::mbar_wait_warp(lsef2, lcn & 1, abort_flag, A.err)) {
                    ok = false;
                    break;
                }
                ++lcn;
                const float4 *nlse4 = reinterpret_cast<const float4 *>(lse_s + 64 * hf);
                // phase 2: key row j = 128 b + row adds its probabilities under this half's
                // query columns of the tile; key tile b is complete after query tile r = b
                const int qmax = A.P - 1 - 128 * r - 64 * hf;  // query column c valid iff c <= qmax
#pragma unroll
                for (int b = kHpMaxTiles - 1; b >= 0; --b) {
                    if (b > r || !ok) continue;
                    const int ts = tcn % HP_TSLOTS;
                    if (!tc::mbar_wait_warp(&tfull[ts], (tcn / HP_TSLOTS) & 1, abort_flag, A.err)) {
                        ok = false;
                        continue;
                    }
                    tc::fence_after_sync();
                    const int j = 128 * b + row;
                    const int lo = j - 128 * r - 64 * hf;  // query column c valid iff c >= lo
                    // the warp's rows span lo_lo .. lo_lo + 31 (warp-uniform)
                    const int lo_lo = 128 * (b - r) + (warp & 3) * 32 - 64 * hf;
                    float bs = 0.f;
                    if (qmax < 0 || lo_lo > min(63, qmax)) {  // no column visible to the warp
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&tempty[ts]);
                        ++tcn;
                    } else {
                        float v[64];
                        load_half(tmem + tcol + ts * 128, v);
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&tempty[ts]);
                        ++tcn;
                        if (lo_lo + 31 <= 0 && qmax >= 63)
                            bs = p2_block<kColAll, kColAll>(v, nlse4, lo, qmax, k1_2);
                        else if (lo_lo == 0 && qmax >= 63)
                            bs = p2_block<kColMask, kColAll>(v, nlse4, lo, qmax, k1_2);
                        else if (lo_lo == 32 && qmax >= 63)
                            bs = p2_block<kColNone, kColMask>(v, nlse4, lo, qmax, k1_2);
                        else
                            bs = p2_block<kColMask, kColMask>(v, nlse4, lo, qmax, k1_2);
                    }
                    accb[b] = (r == nt - 1 ? 0.f : accb[b]) + bs;
                    if (b == r && j < A.P) accu[j] = accb[b];
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

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 1;
    return n;
}

}  // namespace

bool h2o_colsum_tc_supported(int d, int P, int dtype) {
    return d == 128 && P >= 1 && (P + 127) / 128 <= kHpMaxTiles &&
           (dtype == KVE_F16 || dtype == KVE_BF16);
}

cudaError_t launch_h2o_colsum_tc(int units, int P, const void *K, const void *Q, int dtype,
                                 float *acc_out, cudaStream_t st) {
    if (units <= 0) return cudaSuccess;
    const bool f16 = dtype == KVE_F16;
    const uint64_t rows = (uint64_t)units * (uint64_t)P;
    CUtensorMap tk, tq;
    if (!make_tmap_bf16_2d(&tk, K, 128, rows, 64, 128, f16) ||
        !make_tmap_bf16_2d(&tq, Q, 128, rows, 64, 128, f16))
        return cudaErrorInvalidValue;
    ColsumArgs A;
    A.units = units;
    A.P = P;
    A.nt = (P + 127) / 128;
    A.ab_bf16 = f16 ? 0 : 1;
    A.k1 = kLog2e / sqrtf(128.f);
    A.acc = acc_out;
    A.err = device_error_word();
    cudaError_t e = cudaFuncSetAttribute(h2o_colsum_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)HP_SMEM);
    if (e != cudaSuccess) return e;
    const int grid = units < sm_count() ? units : sm_count();
    h2o_colsum_tc_kernel<<<grid, kHpThreads, HP_SMEM, st>>>(tk, tq, A);
    return cudaGetLastError();
}

}  // namespace kve

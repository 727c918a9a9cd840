// Per-model preparation of the output-projection norm (LORE-KV page, Method, Eqs. 5-7:
// e = ||W_O Delta o||). For each layer and query head h, G = W_O^h^T W_O^h and its Cholesky
// factor L (double), so that ||W_O^h x||^2 = x^T G x = ||L^T x||^2. This runs once per model
// (the weights are static); it is not part of the per-request eviction pass. bf16 weights with
// d_head 128 form G on the tensor cores; other shapes accumulate it in double on the CUDA cores.
#include "tc_common.cuh"

namespace kve {

namespace {

constexpr int kGramRows = 16;  // rows of W staged in shared memory per step

// grid (Hq, L), block 256; d <= 128. Thread (ty, tx) of a 16x16 grid owns the (d/16)x(d/16)
// block of G at rows ty*(d/16).., columns tx*(d/16)..
template <typename T>
__global__ void __launch_bounds__(256) gram_kernel(const T *__restrict__ W, int Hq, int d,
                                                   int d_model, double *__restrict__ Gd) {
    extern __shared__ double wsm[];  // [kGramRows][d]
    const int h = blockIdx.x, l = blockIdx.y;
    const int ncols = Hq * d;
    const T *Wl = W + (size_t)l * d_model * ncols + (size_t)h * d;
    const int per = d / 16;  // <= 8
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    double acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0;
    for (int r0 = 0; r0 < d_model; r0 += kGramRows) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kGramRows * d; idx += blockDim.x) {
            const int rr = idx / d, k = idx % d;
            wsm[idx] = (r0 + rr < d_model) ? (double)to_f(Wl[(size_t)(r0 + rr) * ncols + k]) : 0.0;
        }
        __syncthreads();
        for (int rr = 0; rr < kGramRows; ++rr) {
            double a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                a[i] = (i < per) ? wsm[rr * d + ty * per + i] : 0.0;
                b[i] = (i < per) ? wsm[rr * d + tx * per + i] : 0.0;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
        }
    }
    double *G = Gd + ((size_t)l * Hq + h) * d * d;
    for (int i = 0; i < per; ++i)
        for (int j = 0; j < per; ++j) G[(size_t)(ty * per + i) * d + tx * per + j] = acc[i][j];
}

// grid (Hq, L), block d (<= 128). Right-looking Cholesky of one d x d matrix in shared memory.
__global__ void cholesky_kernel(const double *__restrict__ Gd, int Hq, int d,
                                float *__restrict__ L_out, float *__restrict__ G_out,
                                int *__restrict__ notpd) {
    extern __shared__ double A[];  // [d][d]
    const int h = blockIdx.x, l = blockIdx.y, i = threadIdx.x;
    const size_t off = ((size_t)l * Hq + h) * d * d;
    for (int idx = threadIdx.x; idx < d * d; idx += blockDim.x) {
        A[idx] = Gd[off + idx];
        G_out[off + idx] = (float)Gd[off + idx];
    }
    __syncthreads();
    __shared__ int bad;
    if (i == 0) bad = 0;
    __syncthreads();
    for (int j = 0; j < d; ++j) {
        // pivot (all threads read the same value after the barrier)
        const double piv2 = A[j * d + j];
        if (!(piv2 > 0.0)) {
            if (i == 0) bad = 1;
            break;
        }
        const double piv = sqrt(piv2);
        __syncthreads();
        if (i >= j) A[i * d + j] = (i == j) ? piv : A[i * d + j] / piv;
        __syncthreads();
        if (i > j) {
            const double lij = A[i * d + j];
            for (int k = j + 1; k <= i; ++k) A[i * d + k] -= lij * A[k * d + j];
        }
        __syncthreads();
    }
    __syncthreads();
    if (bad) {
        if (i == 0) atomicExch(notpd, 1);
        return;
    }
    for (int idx = threadIdx.x; idx < d * d; idx += blockDim.x) {
        const int r = idx / d, c = idx % d;
        L_out[off + idx] = (c <= r) ? (float)A[idx] : 0.f;
    }
}

// ---- G on the tensor cores (bf16 W, d = 128, d_model a multiple of 128) --------------------------
// G = W^T W for W = W_O^h (d_model x 128): both MMA operands are the same 128-row chunk of W in
// shared memory, read MN-major (the output dimensions i, j along M and N, the d_model rows along
// K). The bf16 products are exact in fp32. Each 32-row slice of the sum goes to a TMEM buffer of
// its own (four per chunk) and is added, right after its MMAs, into a compensated fp32 pair
// (hi, lo) per element, so the roundings left are the tensor pipe's within a 32-row slice and the
// final hi + lo in double: about 1e-8 of |G| at d_model 4096.
// One CTA per (head, layer), 16 warps: warp w owns TMEM lanes 32 (w % 4) .. +31 (rows i of G) and
// columns 32 (w / 4) .. +31 of every buffer; thread 0 also issues the copies and the MMAs. A chunk
// is copied two ahead into a 2-slot ring; its MMAs start once every thread has read the previous
// chunk's buffers.
constexpr int kGtThreads = 512;
constexpr uint32_t GT_SLOT = 32768;      // one 128 x 128 bf16 chunk: two 64-column TMA boxes
constexpr uint32_t GT_BAR = 2 * GT_SLOT;
constexpr size_t GT_SMEM = 120 * 1024;   // also keeps a second CTA (and its TMEM) off the SM

__device__ __forceinline__ void two_sum_add(float &hi, float &lo, float v) {
    const float s = hi + v;
    const float bp = s - hi;
    lo += (hi - (s - bp)) + (v - bp);  // the exact rounding error of hi + v
    hi = s;
}

__global__ void __launch_bounds__(kGtThreads, 1)
    gram_tc_kernel(const __grid_constant__ CUtensorMap tm_w, int d_model, int Hq,
                   double *__restrict__ Gd, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const int h = blockIdx.x, l = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + GT_BAR);  // [2]: chunk copied
    uint64_t *mdone = full + 2, *drain = full + 3;                // chunk's MMAs complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(full + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + 5);
    if (threadIdx.x == 0) {
        tc::mbar_init(&full[0], 1);
        tc::mbar_init(&full[1], 1);
        tc::mbar_init(mdone, 1);
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int nch = d_model / 128;
    const int row0 = l * d_model, col0 = h * 128;
    auto load = [&](int c) {  // chunk c into slot c % 2
        uint8_t *dst = sm + (c & 1) * GT_SLOT;
        tc::mbar_expect_tx(&full[c & 1], GT_SLOT);
        tc::tma_load_2d(dst, &tm_w, col0, row0 + 128 * c, &full[c & 1]);
        tc::tma_load_2d(dst + 16384, &tm_w, col0 + 64, row0 + 128 * c, &full[c & 1]);
    };
    int issued = 0;  // chunks whose copy thread 0 has started
    if (threadIdx.x == 0)
        for (; issued < 2 && issued < nch; ++issued) load(issued);
    constexpr uint32_t idesc = tc::idesc_f16kind(128, 128, 1, 1, 1);
    const uint32_t tb = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 32u * (warp >> 2);
    float hi[32], lo[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) hi[e] = lo[e] = 0.f;
    bool ok = true;
    int used = 0;  // chunks whose MMAs thread 0 has issued
    for (int c = 0; c < nch; ++c) {
        if (threadIdx.x == 0) {
            ok = tc::mbar_wait(&full[c & 1], (c >> 1) & 1, abort_flag, err);
            if (ok) {
                tc::fence_after_sync();
                const uint32_t a = tc::smem_u32(sm + (c & 1) * GT_SLOT);
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // K step k (16 rows) into buffer k / 2
                    const uint64_t desc = tc::sdesc_sw128(a + k * 2048, 16384, 1024);
                    tc::mma_bf16(tmem + 128 * (k >> 1), desc, desc, idesc, k & 1);
                }
                tc::mma_commit(mdone);
                used = c + 1;
            }
        }
        // a wait that gave up sets the abort flag, which ends the other waits early
        const bool got = tc::mbar_wait_warp(mdone, c & 1, abort_flag, err);
        if (got) {
            tc::fence_after_sync();
#pragma unroll
            for (int b = 0; b < 8; ++b) {  // buffer b / 2, columns 16 (b % 2) ..
                float v[16];
                tc::tmem_ld16(tb + 128 * (b >> 1) + 16 * (b & 1), v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    two_sum_add(hi[16 * (b & 1) + e], lo[16 * (b & 1) + e], v[e]);
            }
            tc::fence_before_sync();
            // the chunk's MMAs have read its slot: refill it with chunk c + 2
            if (threadIdx.x == 0 && c + 2 < nch) load(issued++);
        }
        // every thread has read the buffers before the next chunk's MMAs overwrite them
        if (!__syncthreads_and(ok && got)) {
            ok = false;
            break;
        }
    }
    if (ok) {
        const int i = (warp & 3) * 32 + lane;
        double *G = Gd + (((size_t)l * Hq + h) * 128 + i) * 128 + 32 * (warp >> 2);
#pragma unroll
        for (int e = 0; e < 32; ++e) G[e] = (double)hi[e] + (double)lo[e];
    } else if (threadIdx.x == 0) {
        // leave nothing in flight: the copies started and not consumed, and the MMAs issued
        for (int c = used; c < issued; ++c) tc::mbar_drain(&full[c & 1], (c >> 1) & 1);
        tc::mma_commit(drain);
        tc::mbar_drain(drain, 0);
    }
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_prepare_wo(int L, int Hq, int d, int d_model, int dtype, const void *W_O,
                              float *L_out, float *G_out, int *notpd_flag, cudaStream_t st) {
    double *Gd = nullptr;
    cudaError_t e = cudaMallocAsync(&Gd, sizeof(double) * (size_t)L * Hq * d * d, st);
    if (e != cudaSuccess) return e;
    const size_t smem_g = sizeof(double) * kGramRows * d;
    CUtensorMap tw;
    if (dtype == KVE_BF16 && d == 128 && d_model % 128 == 0 &&
        make_tmap_bf16_2d(&tw, W_O, (uint64_t)Hq * 128, (uint64_t)L * d_model, 64, 128)) {
        e = cudaFuncSetAttribute(gram_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)GT_SMEM);
        if (e != cudaSuccess) {
            cudaFreeAsync(Gd, st);
            return e;
        }
        gram_tc_kernel<<<dim3(Hq, L), kGtThreads, GT_SMEM, st>>>(tw, d_model, Hq, Gd,
                                                                 device_error_word());
    } else if (dtype == KVE_F32)
        gram_kernel<float><<<dim3(Hq, L), 256, smem_g, st>>>(static_cast<const float *>(W_O), Hq,
                                                            d, d_model, Gd);
    else
        gram_kernel<__nv_bfloat16><<<dim3(Hq, L), 256, smem_g, st>>>(
            static_cast<const __nv_bfloat16 *>(W_O), Hq, d, d_model, Gd);
    const size_t smem_c = sizeof(double) * d * d;
    e = cudaFuncSetAttribute(cholesky_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_c);
    if (e != cudaSuccess) return e;
    cholesky_kernel<<<dim3(Hq, L), d, smem_c, st>>>(Gd, Hq, d, L_out, G_out, notpd_flag);
    e = cudaGetLastError();
    cudaFreeAsync(Gd, st);
    return e;
}

}  // namespace kve

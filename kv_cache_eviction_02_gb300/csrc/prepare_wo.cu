// Per-model preparation of the output-projection norm (LORE-KV page, Method, Eqs. 5-7:
// e = ||W_O Delta o||). For each layer and query head h, G = W_O^h^T W_O^h (double accumulation)
// and its Cholesky factor L (double), so that ||W_O^h x||^2 = x^T G x = ||L^T x||^2. This runs
// once per model (the weights are static); it is not part of the per-request eviction pass.
#include "kve_internal.cuh"

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

}  // namespace

cudaError_t launch_prepare_wo(int L, int Hq, int d, int d_model, int dtype, const void *W_O,
                              float *L_out, float *G_out, int *notpd_flag, cudaStream_t st) {
    double *Gd = nullptr;
    cudaError_t e = cudaMallocAsync(&Gd, sizeof(double) * (size_t)L * Hq * d * d, st);
    if (e != cudaSuccess) return e;
    const size_t smem_g = sizeof(double) * kGramRows * d;
    if (dtype == KVE_F32)
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

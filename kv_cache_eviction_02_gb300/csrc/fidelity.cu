// Attention-output fidelity of a compressed cache (LORE-KV page, analyses, "Attention-output
// fidelity": the retained cache reproduces full-cache attention outputs). Reading: the fidelity of
// one query is the cosine similarity between its attention output over the compressed cache and
// over the full cache; the diagnostic reports every query's cosine and their mean.
//
//   cosine_kernel: one warp per row, 16-byte loads, fp32 dot product and norms;
//   mean_kernel:   one CTA, strided per-thread sums and a fixed-order tree, so the mean is
//                  deterministic.
#include "kve_internal.cuh"

namespace kve {

namespace {

__global__ void cosine_kernel(const float *__restrict__ a, const float *__restrict__ b, int rows,
                              int d, float *__restrict__ cos_out) {
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *x = a + (size_t)row * d;
    const float *y = b + (size_t)row * d;
    float xy = 0.f, xx = 0.f, yy = 0.f;
    if ((d & 3) == 0) {
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
        const float4 *y4 = reinterpret_cast<const float4 *>(y);
        for (int k = lane; k < (d >> 2); k += 32) {
            const float4 p = x4[k], q = y4[k];
            xy = fmaf(p.x, q.x, fmaf(p.y, q.y, fmaf(p.z, q.z, fmaf(p.w, q.w, xy))));
            xx = fmaf(p.x, p.x, fmaf(p.y, p.y, fmaf(p.z, p.z, fmaf(p.w, p.w, xx))));
            yy = fmaf(q.x, q.x, fmaf(q.y, q.y, fmaf(q.z, q.z, fmaf(q.w, q.w, yy))));
        }
    } else {
        for (int k = lane; k < d; k += 32) {
            xy = fmaf(x[k], y[k], xy);
            xx = fmaf(x[k], x[k], xx);
            yy = fmaf(y[k], y[k], yy);
        }
    }
    xy = warp_sum(xy);
    xx = warp_sum(xx);
    yy = warp_sum(yy);
    if (lane == 0) {
        const float den = sqrtf(xx) * sqrtf(yy);
        cos_out[row] = den > 0.f ? xy / den : 0.f;
    }
}

constexpr int kMeanThreads = 1024;

__global__ void __launch_bounds__(kMeanThreads) mean_kernel(const float *__restrict__ v, int rows,
                                                            float *__restrict__ mean_out) {
    __shared__ double part[kMeanThreads];
    double s = 0.0;
    for (int i = threadIdx.x; i < rows; i += kMeanThreads) s += (double)v[i];
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = kMeanThreads / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) mean_out[0] = (float)(part[0] / (double)rows);
}

}  // namespace

cudaError_t launch_output_fidelity(const float *o_full, const float *o_comp, int rows, int d,
                                   float *cos_out, float *mean_out, cudaStream_t st) {
    constexpr int kWarps = 8;
    cosine_kernel<<<(rows + kWarps - 1) / kWarps, kWarps * 32, 0, st>>>(o_full, o_comp, rows, d,
                                                                        cos_out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !mean_out) return e;
    mean_kernel<<<1, kMeanThreads, 0, st>>>(cos_out, rows, mean_out);
    return cudaGetLastError();
}

}  // namespace kve

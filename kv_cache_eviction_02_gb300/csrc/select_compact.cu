// Chunked top-B selection and gather-compaction (LORE-KV page, "Evict and decode", Eq. 8;
// "Hyperparameters": adjacent-token chunks of 4). One CTA per unit:
//   1. chunk scores C_c = mean of S over [sink + c*chunk, sink + (c+1)*chunk), as order-preserving
//      32-bit keys, computed once into shared memory (recomputed from S when they do not fit);
//   2. MSB-first radix select (4 passes of 8 bits, shared-memory histograms, one warp finds the
//      bin) gives the key tau of the (B/chunk)-th largest chunk; every chunk above tau is kept, and
//      among the chunks equal to tau the lowest indices fill the remainder;
//   3. each thread owns a contiguous run of chunks: two block-wide prefix sums (chunks equal to tau,
//      then kept chunks) give every thread its first output slot, and the kept positions are
//      written in ascending order (sink, kept chunks, window);
//   4. the CTA gathers the kept K and V rows with 16-byte vector copies.
#include "kve_internal.cuh"

namespace kve {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelSmemKeys = 53248;  // chunk keys held in shared memory (208 KB)

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t chunk_key(const float *__restrict__ S, int sink, int chunk,
                                              int c) {
    const float *p = S + sink + (size_t)c * chunk;
    float acc = 0.f;
    for (int j = 0; j < chunk; ++j) acc += p[j];
    return order_key(acc / (float)chunk);
}

// Exclusive block-wide scan of one value per thread; returns the exclusive prefix, *total = sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int t = (lane < nw) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) warp_tot[lane] = t;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const int before = (warp > 0) ? warp_tot[warp - 1] : 0;
    *total = warp_tot[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before + x - v;
}

template <typename VecT>
__global__ void __launch_bounds__(kSelThreads) select_compact_kernel(
    LorekvDims D, const float *__restrict__ scores, const VecT *__restrict__ K,
    const VecT *__restrict__ V, int32_t *__restrict__ kept_idx, int32_t *__restrict__ kept_len,
    VecT *__restrict__ K_out, VecT *__restrict__ V_out, int cap, int vec_per_row) {
    extern __shared__ uint32_t keys_s[];  // [nch] when they fit
    __shared__ uint32_t hist[256];
    __shared__ int warp_tot[32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_krem;
    const int unit = blockIdx.x;
    const float *S = scores + (size_t)unit * D.n;
    int32_t *idx = kept_idx + (size_t)unit * cap;
    const int nch = (D.n - D.sink - D.w) / D.chunk;
    const int keepc = D.B / D.chunk;
    const bool in_smem = nch <= kSelSmemKeys;
    if (nch <= keepc) {
        for (int i = threadIdx.x; i < D.n; i += blockDim.x) idx[i] = i;
    } else {
        if (in_smem)
            for (int c = threadIdx.x; c < nch; c += blockDim.x)
                keys_s[c] = chunk_key(S, D.sink, D.chunk, c);
        // ---- radix select of the keepc-th largest chunk key ----
        if (threadIdx.x == 0) {
            s_prefix = 0u;
            s_krem = keepc;
        }
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            const uint32_t mask = (pass == 0) ? 0u : (0xffffffffu << (shift + 8));
            for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
            __syncthreads();
            const uint32_t prefix = s_prefix;
            for (int c = threadIdx.x; c < nch; c += blockDim.x) {
                const uint32_t key = in_smem ? keys_s[c] : chunk_key(S, D.sink, D.chunk, c);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (threadIdx.x < 32) {  // warp 0 finds the bin of the krem-th largest key
                const int lane = threadIdx.x;
                uint32_t cnt[8];
                int sum = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    cnt[k] = hist[255 - 8 * lane - k];
                    sum += (int)cnt[k];
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
                    for (int k = 0; k < 8; ++k) {
                        if ((int)cnt[k] >= kr) {
                            bsel = 255 - 8 * lane - k;
                            break;
                        }
                        kr -= (int)cnt[k];
                    }
                    s_krem = kr;
                    s_prefix = prefix | ((uint32_t)bsel << shift);
                }
            }
            __syncthreads();
        }
        const uint32_t tau = s_prefix;
        const int take_eq = s_krem;  // chunks equal to tau to keep, lowest indices first
        // ---- ordered write-out: thread t owns chunks [c0, c1) ----
        // an odd run length puts the 32 threads of a warp on 32 different shared-memory banks
        const int seg = ((nch + blockDim.x - 1) / blockDim.x) | 1;
        const int c0 = min(nch, (int)threadIdx.x * seg), c1 = min(nch, c0 + seg);
        int n_gt = 0, n_eq = 0;
        for (int c = c0; c < c1; ++c) {
            const uint32_t key = in_smem ? keys_s[c] : chunk_key(S, D.sink, D.chunk, c);
            n_gt += key > tau;
            n_eq += key == tau;
        }
        int tot;
        const int eq_before = block_exclusive_scan(n_eq, warp_tot, &tot);
        const int take_here = max(0, min(n_eq, take_eq - eq_before));
        int pos = block_exclusive_scan(n_gt + take_here, warp_tot, &tot);
        int eq_seen = 0;
        for (int c = c0; c < c1; ++c) {
            const uint32_t key = in_smem ? keys_s[c] : chunk_key(S, D.sink, D.chunk, c);
            bool sel = key > tau;
            if (key == tau) sel = eq_seen++ < take_here;
            if (sel) {
                for (int j = 0; j < D.chunk; ++j)
                    idx[D.sink + pos * D.chunk + j] = D.sink + c * D.chunk + j;
                ++pos;
            }
        }
        for (int i = threadIdx.x; i < D.sink; i += blockDim.x) idx[i] = i;
        for (int i = threadIdx.x; i < D.w; i += blockDim.x)
            idx[D.sink + keepc * D.chunk + i] = D.n - D.w + i;
    }
    if (threadIdx.x == 0) kept_len[unit] = cap;
    __syncthreads();
    // ---- gather-compaction ----
    const VecT *Ku = K + (size_t)unit * D.n * vec_per_row;
    const VecT *Vu = V + (size_t)unit * D.n * vec_per_row;
    VecT *Ko = K_out + (size_t)unit * cap * vec_per_row;
    VecT *Vo = V_out + (size_t)unit * cap * vec_per_row;
    const int total = cap * vec_per_row;
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
        const int r = e / vec_per_row, c = e % vec_per_row;
        const int src = idx[r];
        Ko[e] = Ku[(size_t)src * vec_per_row + c];
        Vo[e] = Vu[(size_t)src * vec_per_row + c];
    }
}

}  // namespace

cudaError_t launch_select_compact(const LorekvDims &D, const float *scores, const void *K,
                                  const void *V, int32_t *kept_idx, int32_t *kept_len,
                                  void *K_out, void *V_out, int cap, cudaStream_t st) {
    const size_t row_bytes = (size_t)D.d * dtype_size(D.dtype);
    if (row_bytes % 16 != 0) return cudaErrorInvalidValue;
    const int vpr = (int)(row_bytes / 16);
    const int nch = (D.n - D.sink - D.w) / D.chunk;
    const size_t smem = nch <= kSelSmemKeys ? (size_t)nch * sizeof(uint32_t) : 0;
    cudaError_t e = cudaFuncSetAttribute(select_compact_kernel<uint4>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSelSmemKeys * (int)sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    select_compact_kernel<uint4><<<D.units, kSelThreads, smem, st>>>(
        D, scores, (const uint4 *)K, (const uint4 *)V, kept_idx, kept_len, (uint4 *)K_out,
        (uint4 *)V_out, cap, vpr);
    return cudaGetLastError();
}

}  // namespace kve

// Counter-causal surprise refresh, fast single-layer variant (counter-causal page, "Back from the
// Future: KV Cache Management by Counter-Causal Surprise": Section 3.2 steps 1-5, Section 3.3,
// Algorithm 3, design choice 4).
//
//   cc_attn_kernel      o_i^h = sum_{j>i} softmax_j(q_i^h . k_j / sqrt d) v_j over the cached K/V
//                       (strictly upper-triangular mask, fresh queries); one warp per query, K tiles
//                       of 32 keys staged in padded shared memory (lane l scores key l), online
//                       softmax, lanes hold d/32 output columns each. Used for fp32 and for head
//                       sizes other than 128; bf16 with d_head 128 runs on the tensor cores
//                       (cc_tc.cu).
//   cc_proj_kernel      r_i = h_i + W_O o_i (o_i = the heads' outputs concatenated) as a tiled FP32
//                       product, fused with the true token's unembedding row: each CTA writes the
//                       partial logit sum_m W_U[x_i][m] r_i[m] over its 64 columns m.
//   cc_finish_kernel    surprise_i = -(sum of the partial logits, fixed order); +inf for the sink
//                       slots and the last token.
//   cc_select_kernel    keep the J highest surprises (equal: the lower position), ascending order:
//                       MSB-first radix select over shared-memory histograms, an ordered scan,
//                       kept positions and token ids (one CTA per sequence);
//   cc_gather_kernel    16-byte copies of the kept K and V rows over the whole GPU.
#include <algorithm>

#include "kve_internal.cuh"

namespace kve {

namespace {

constexpr int kCcQueriesPerCta = 8;  // one warp per query
constexpr int kCcKeys = 32;          // keys per staged tile

template <typename T>
__global__ void __launch_bounds__(kCcQueriesPerCta * 32) cc_attn_kernel(
    const T *__restrict__ K, const T *__restrict__ V, const T *__restrict__ Q, int n, int ld,
    int hq, int hkv, int d, float scale, float *__restrict__ O) {
    __shared__ float ks[kCcKeys][129];  // padded: lane l reads row l column c conflict-free
    __shared__ float vs[kCcKeys][128];
    __shared__ float qs[kCcQueriesPerCta][128];
    const int b = blockIdx.z, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = blockIdx.x * kCcQueriesPerCta;
    const int i = i0 + warp;
    const int kh = h / (hq / hkv);
    const T *Kb = K + ((size_t)b * hkv + kh) * ld * d;
    const T *Vb = V + ((size_t)b * hkv + kh) * ld * d;
    const T *Qb = Q + ((size_t)b * hq + h) * ld * d;
    for (int e = threadIdx.x; e < kCcQueriesPerCta * d; e += blockDim.x) {
        const int r = e / d, c = e % d;
        qs[r][c] = (i0 + r < n) ? to_f(Qb[(size_t)(i0 + r) * d + c]) * scale : 0.f;
    }
    const int per = d >> 5;  // output columns per lane (d = 32, 64 or 128): lane + 32 e
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    float m = -INFINITY, l = 0.f;
    for (int j0 = i0 + 1; j0 < n; j0 += kCcKeys) {
        __syncthreads();
        for (int e = threadIdx.x; e < kCcKeys * d; e += blockDim.x) {
            const int r = e / d, c = e % d;
            const bool in = j0 + r < n;
            ks[r][c] = in ? to_f(Kb[(size_t)(j0 + r) * d + c]) : 0.f;
            vs[r][c] = in ? to_f(Vb[(size_t)(j0 + r) * d + c]) : 0.f;
        }
        __syncthreads();
        if (i >= n) continue;
        const int j = j0 + lane;
        float s = 0.f;
        for (int c = 0; c < d; ++c) s = fmaf(qs[warp][c], ks[lane][c], s);
        const bool valid = j > i && j < n;
        const float sv = valid ? s : -INFINITY;
        const float mt = warp_max(sv);
        if (mt == -INFINITY) continue;  // no visible key in this tile (warp-uniform)
        const float mn = fmaxf(m, mt);
        const float corr = __expf(m - mn);  // exp(-inf) = 0 on the first visible tile
        const float p = valid ? __expf(s - mn) : 0.f;
        l = l * corr + warp_sum(p);
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] *= corr;
        for (int r = 0; r < kCcKeys; ++r) {
            const float pr = __shfl_sync(0xffffffffu, p, r);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < per) o[e] = fmaf(pr, vs[r][lane + 32 * e], o[e]);
        }
        m = mn;
    }
    if (i < n) {
        const float inv = l > 0.f ? 1.f / l : 0.f;  // the last token sees no key: o = 0
        float *dst = O + ((size_t)b * ld + i) * hq * d + (size_t)h * d + lane;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e < per) dst[32 * e] = o[e] * inv;
    }
}

// r = h + W_O o and the partial logits; CTA tile 64 tokens x 64 columns m, K chunks of 32.
constexpr int kPT = 64, kPM = 64, kPK = 32;

template <typename T>
__global__ void __launch_bounds__(256) cc_proj_kernel(
    const float *__restrict__ O, const T *__restrict__ Hres, const T *__restrict__ W_O,
    const T *__restrict__ W_U, const int32_t *__restrict__ X, int n, int ld, int kdim, int dm,
    int vocab, float *__restrict__ part, unsigned *err) {
    __shared__ float as[kPT][kPK + 1];
    __shared__ float bs[kPM][kPK + 1];
    const int b = blockIdx.z;
    const int t0 = blockIdx.x * kPT, m0 = blockIdx.y * kPM;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;  // 16 x 16 threads, 4 x 4 outputs
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
    const float *Ob = O + (size_t)b * ld * kdim;
    for (int k0 = 0; k0 < kdim; k0 += kPK) {
        __syncthreads();
        for (int e = threadIdx.x; e < kPT * kPK; e += 256) {
            const int r = e / kPK, c = e % kPK;
            const int t = t0 + r, k = k0 + c;
            as[r][c] = (t < n && k < kdim) ? Ob[(size_t)t * kdim + k] : 0.f;
            const int mm = m0 + r;
            bs[r][c] = (mm < dm && k < kdim) ? to_f(W_O[(size_t)mm * kdim + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int c = 0; c < kPK; ++c) {
            float av[4], bv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) av[a] = as[ty * 4 + a][c];
#pragma unroll
            for (int q = 0; q < 4; ++q) bv[q] = bs[tx * 4 + q][c];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(av[a], bv[q], acc[a][q]);
        }
    }
    // epilogue: r = acc + h, partial logit over this CTA's columns for each of the 4 tokens
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int t = t0 + ty * 4 + a;
        float z = 0.f;
        if (t < n) {
            int x = X[(size_t)b * ld + t];
            if (x < 0 || x >= vocab) {  // reported, and the row treated as token 0
                if (err) atomicOr(err, KVE_DEVERR_BADINDEX);
                x = 0;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int mm = m0 + tx * 4 + q;
                if (mm < dm) {
                    const float r = acc[a][q] + to_f(Hres[((size_t)b * ld + t) * dm + mm]);
                    z = fmaf(to_f(W_U[(size_t)x * dm + mm]), r, z);
                }
            }
        }
        // sum over the 16 threads (tx) that share these tokens: lanes 0-15 / 16-31 of a warp
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        if (tx == 0 && t < n) part[((size_t)b * gridDim.y + blockIdx.y) * ld + t] = z;
    }
}

__global__ void cc_finish_kernel(const float *__restrict__ part, int n, int ld, int parts,
                                 int sink, float *__restrict__ surprise) {
    const int b = blockIdx.y;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n) return;
    float z = 0.f;
    for (int k = 0; k < parts; ++k) z += part[((size_t)b * parts + k) * ld + t];
    surprise[(size_t)b * ld + t] = (t < sink || t == n - 1) ? INFINITY : -z;
}

__device__ __forceinline__ uint32_t cc_key(float f) {  // order-preserving (+inf largest)
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kSelT = 1024;

// Exclusive block-wide scan of one value per thread; *total = the block's sum. All threads call.
__device__ __forceinline__ int cc_scan(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int before = 0, tot = 0;
    for (int w = 0; w < kSelT / 32; ++w) {
        const int t = warp_tot[w];
        before += w < warp ? t : 0;
        tot += t;
    }
    __syncthreads();
    *total = tot;
    return before + x - v;
}

// surprise, X, pos: [batch][ld] (first n used); kept [batch][J]; X_out, pos_out: [batch][ldo].
// pos and pos_out may be null.
__global__ void __launch_bounds__(kSelT) cc_select_kernel(
    const float *__restrict__ surprise, const int32_t *__restrict__ X,
    const int32_t *__restrict__ pos, int n, int ld, int J, int32_t *__restrict__ kept,
    int32_t *__restrict__ X_out, int32_t *__restrict__ pos_out, int ldo) {
    __shared__ uint32_t hist[256];
    __shared__ int warp_tot[32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_krem;
    const int b = blockIdx.x;
    const float *S = surprise + (size_t)b * ld;
    int32_t *kb = kept + (size_t)b * J;
    if (threadIdx.x == 0) {
        s_prefix = 0u;
        s_krem = J;
    }
    __syncthreads();
    if (J < n) {
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            const uint32_t mask = pass == 0 ? 0u : (0xffffffffu << (shift + 8));
            for (int i = threadIdx.x; i < 256; i += kSelT) hist[i] = 0u;
            __syncthreads();
            const uint32_t prefix = s_prefix;
            for (int i = threadIdx.x; i < n; i += kSelT) {
                const uint32_t key = cc_key(S[i]);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (threadIdx.x < 32) {  // warp 0 finds the bin of the krem-th largest key
                const int lane = threadIdx.x;
                uint32_t c[8];
                int sum = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    c[k] = hist[255 - 8 * lane - k];
                    sum += (int)c[k];
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
                        if ((int)c[k] >= kr) {
                            bsel = 255 - 8 * lane - k;
                            break;
                        }
                        kr -= (int)c[k];
                    }
                    s_krem = kr;
                    s_prefix = prefix | ((uint32_t)bsel << shift);
                }
            }
            __syncthreads();
        }
    }
    const uint32_t tau = s_prefix;
    const int take_eq = s_krem;  // keys equal to tau that stay, lower positions first
    int run_eq = 0, run = 0;
    for (int base = 0; base < n; base += kSelT) {
        const int i = base + threadIdx.x;
        uint32_t key = 0u;
        if (i < n) key = cc_key(S[i]);
        const int eq = (J < n && i < n && key == tau) ? 1 : 0;
        int tot_eq;
        const int rank_eq = run_eq + cc_scan(eq, warp_tot, &tot_eq);
        const int sel = (i < n && (J >= n || key > tau || (eq && rank_eq < take_eq))) ? 1 : 0;
        int tot;
        const int slot = run + cc_scan(sel, warp_tot, &tot);
        if (sel) kb[slot] = i;
        run_eq += tot_eq;
        run += tot;
    }
    __syncthreads();
    for (int r = threadIdx.x; r < J; r += kSelT) {
        X_out[(size_t)b * ldo + r] = X[(size_t)b * ld + kb[r]];
        if (pos_out) pos_out[(size_t)b * ldo + r] = pos[(size_t)b * ld + kb[r]];
    }
}

// Kept rows of up to four row-major tensors [batch][heads][ld][row] (16-byte words): dst row
// (b, h, r) = src row (b, h, kept[b][r]); one grid-stride loop over all words of all tensors.
__global__ void cc_gather_kernel(CcGatherSet G, const int32_t *__restrict__ kept, int J,
                                 int ld_in, int ld_out) {
    for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < G.start[G.count];
         e += (long)gridDim.x * blockDim.x) {
        int k = 0;
        while (k + 1 < G.count && e >= G.start[k + 1]) ++k;
        const long local = e - G.start[k];
        const int vpr = G.vpr[k];
        const int c = (int)(local % vpr);
        const long row = local / vpr;  // (b * heads + h) * J + r
        const int r = (int)(row % J);
        const long bh = row / J;
        const long b = bh / G.heads[k];
        const size_t src = ((size_t)bh * ld_in + kept[(size_t)b * J + r]) * vpr + c;
        const size_t dst = ((size_t)bh * ld_out + r) * vpr + c;
        G.dst[k][dst] = G.src[k][src];
    }
}

template <typename T>
cudaError_t cc_attention_t(const CcDims &D, const void *K, const void *V, const void *Q, float *O,
                           cudaStream_t st) {
    cc_attn_kernel<T><<<dim3((D.n + kCcQueriesPerCta - 1) / kCcQueriesPerCta, D.hq, D.batch),
                        kCcQueriesPerCta * 32, 0, st>>>(
        (const T *)K, (const T *)V, (const T *)Q, D.n, D.ld, D.hq, D.hkv, D.d,
        1.f / sqrtf((float)D.d), O);
    return cudaGetLastError();
}

template <typename T>
cudaError_t cc_logits_t(const CcDims &D, const float *O, const void *H, const void *W_O,
                        const void *W_U, const int32_t *X, float *part, float *surprise,
                        unsigned *err, cudaStream_t st) {
    const int mtiles = (D.dm + kPM - 1) / kPM;
    cc_proj_kernel<T><<<dim3((D.n + kPT - 1) / kPT, mtiles, D.batch), 256, 0, st>>>(
        O, (const T *)H, (const T *)W_O, (const T *)W_U, X, D.n, D.ld, D.hq * D.d, D.dm, D.vocab,
        part, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cc_finish_kernel<<<dim3((D.n + 255) / 256, D.batch), 256, 0, st>>>(part, D.n, D.ld, mtiles,
                                                                      D.sink, surprise);
    return cudaGetLastError();
}

}  // namespace

size_t cc_o_bytes(const CcDims &D) {
    return ((size_t)D.batch * D.ld * D.hq * D.d * sizeof(float) + 255) & ~size_t(255);
}

size_t cc_workspace_bytes(const CcDims &D) {
    // partial logits: ceil(d_model/64) column tiles (CUDA cores) or ceil(d_model/256) column
    // tiles x K splits x 2 column halves (tensor cores)
    const size_t parts = std::max<size_t>((D.dm + kPM - 1) / kPM,
                                          (size_t)((D.dm + 255) / 256) * kCcMaxKSplit * 2);
    return cc_o_bytes(D) + (((size_t)D.batch * parts * D.ld * sizeof(float) + 255) & ~size_t(255));
}

cudaError_t launch_cc_attention(const CcDims &D, const void *K, const void *V, const void *Q,
                                void *ws, unsigned *err, cudaStream_t st) {
    float *O = static_cast<float *>(ws);
    if (cc_attention_tc_supported(D))
        return launch_cc_attention_tc(
            D, K, V, Q, O, cc_logits_tc_supported(D) ? static_cast<__nv_bfloat16 *>(ws) : nullptr,
            err, st);
    if (D.dtype == KVE_F32) return cc_attention_t<float>(D, K, V, Q, O, st);
    return cc_attention_t<__nv_bfloat16>(D, K, V, Q, O, st);
}

cudaError_t launch_cc_logits(const CcDims &D, const void *H, const void *W_O, const void *W_U,
                             const int32_t *X, float *surprise, void *ws, unsigned *err,
                             cudaStream_t st) {
    const float *O = static_cast<const float *>(ws);
    float *part = reinterpret_cast<float *>(static_cast<char *>(ws) + cc_o_bytes(D));
    if (cc_logits_tc_supported(D)) {
        const int ksplit = cc_logits_tc_split(D);
        cudaError_t e = launch_cc_logits_tc(D, static_cast<const __nv_bfloat16 *>(ws), H, W_O,
                                            W_U, X, part, ksplit, err, st);
        if (e != cudaSuccess) return e;
        const int ksteps = D.hq * D.d / 64, per = (ksteps + ksplit - 1) / ksplit;
        const int parts = ((D.dm + 255) / 256) * ((ksteps + per - 1) / per) * 2;
        cc_finish_kernel<<<dim3((D.n + 255) / 256, D.batch), 256, 0, st>>>(part, D.n, D.ld,
                                                                          parts, D.sink, surprise);
        return cudaGetLastError();
    }
    if (D.dtype == KVE_F32)
        return cc_logits_t<float>(D, O, H, W_O, W_U, X, part, surprise, err, st);
    return cc_logits_t<__nv_bfloat16>(D, O, H, W_O, W_U, X, part, surprise, err, st);
}

cudaError_t launch_cc_select_idx(const CcDims &D, const float *surprise, const int32_t *X,
                                 const int32_t *pos, int32_t *kept, int32_t *X_out,
                                 int32_t *pos_out, int ldo, cudaStream_t st) {
    cc_select_kernel<<<D.batch, kSelT, 0, st>>>(surprise, X, pos, D.n, D.ld, D.J, kept, X_out,
                                                 pos_out, ldo);
    return cudaGetLastError();
}

cudaError_t launch_cc_gather(const CcGatherSet &G, const int32_t *kept, int J, int ld_in,
                             int ld_out, cudaStream_t st) {
    const long total = G.start[G.count];
    if (total <= 0) return cudaSuccess;
    const long blocks = std::min<long>((total + 255) / 256, 152L * 8);
    cc_gather_kernel<<<(unsigned)blocks, 256, 0, st>>>(G, kept, J, ld_in, ld_out);
    return cudaGetLastError();
}

void cc_gather_add(CcGatherSet *G, const void *src, void *dst, int batch, int heads,
                   size_t row_bytes, int J) {
    const int k = G->count;
    G->src[k] = static_cast<const uint4 *>(src);
    G->dst[k] = static_cast<uint4 *>(dst);
    G->heads[k] = heads;
    G->vpr[k] = (int)(row_bytes / 16);
    G->start[k + 1] = G->start[k] + (long)batch * heads * J * G->vpr[k];
    G->count = k + 1;
}

namespace {
// Appends count rows to tensors [batch][heads][ld][row] at row `at` from [batch][heads][count][row]
// sources (16-byte words; the same four-tensor table as the gather), plus the ids and positions.
__global__ void cc_append_kernel(CcGatherSet G, int count, int at, int ld,
                                 const int32_t *__restrict__ x_new, int32_t *__restrict__ X,
                                 int32_t *__restrict__ pos, int batch, int first) {
    const long total = G.start[G.count];
    for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < total + (long)batch * count;
         e += (long)gridDim.x * blockDim.x) {
        if (e >= total) {  // ids and positions
            const int k = (int)(e - total), b = k / count, r = k % count;
            X[(size_t)b * ld + at + r] = x_new[k];
            pos[(size_t)b * ld + at + r] = first + r;
            continue;
        }
        int k = 0;
        while (k + 1 < G.count && e >= G.start[k + 1]) ++k;
        const long local = e - G.start[k];
        const int vpr = G.vpr[k];
        const int c = (int)(local % vpr);
        const long row = local / vpr;  // (b * heads + h) * count + r
        const int r = (int)(row % count);
        const long bh = row / count;
        G.dst[k][((size_t)bh * ld + at + r) * vpr + c] = G.src[k][local];
    }
}

}  // namespace

cudaError_t launch_cc_append(const CcGatherSet &G, int count, int at, int ld,
                             const int32_t *x_new, int32_t *X, int32_t *pos, int batch, int first,
                             cudaStream_t st) {
    const long total = G.start[G.count] + (long)batch * count;
    const long blocks = std::min<long>((total + 255) / 256, 152L * 8);
    cc_append_kernel<<<(unsigned)blocks, 256, 0, st>>>(G, count, at, ld, x_new, X, pos, batch,
                                                       first);
    return cudaGetLastError();
}

cudaError_t launch_cc_select(const CcDims &D, const float *surprise, const void *K, const void *V,
                             const int32_t *X, int32_t *kept, void *K_out, void *V_out,
                             int32_t *X_out, cudaStream_t st) {
    const size_t row = (size_t)D.d * dtype_size(D.dtype);
    if (row % 16 != 0) return cudaErrorInvalidValue;
    cudaError_t e = launch_cc_select_idx(D, surprise, X, nullptr, kept, X_out, nullptr, D.J, st);
    if (e != cudaSuccess) return e;
    CcGatherSet G{};
    cc_gather_add(&G, K, K_out, D.batch, D.hkv, row, D.J);
    cc_gather_add(&G, V, V_out, D.batch, D.hkv, row, D.J);
    return launch_cc_gather(G, kept, D.J, D.ld, D.J, st);
}

}  // namespace kve

// lorekv_score_noalloc: the scoring pass of lorekv_score with its scratch memory in a fixed
// device array that belongs to the library, for callers that must not allocate device memory at
// all (no cudaMalloc, no allocator of a framework). Examples: code running under a memory
// manager that owns every device allocation, inside a pre-reserved memory budget, or in a host
// process whose allocator is not available at the call site.
//
// The array lives in this file's device image. In host code `g_noalloc_scratch` names a host-side
// stand-in, not a device address, so its device address is looked up with cudaGetSymbolAddress,
// once per CUDA context (on the first call made while that context is current; cached by the
// driver's context id, so the primary context of each device, a context made current with the
// driver API and a context re-created after cudaDeviceReset each get their own), and that
// address is what the kernels get.
#include "kve_internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 20;  // 64 MiB on every device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

kve::SymbolCache g_noalloc_cache;  // device address of the array, per context

}  // namespace

extern "C" int lorekv_score_noalloc(const KveShape *shape, const KveLorekvParams *params,
                                    const void *K, const void *V, const void *Q_W,
                                    const void *Q_look, const float *L, const float *G,
                                    const float *logits, const int32_t *sampled,
                                    float *scores_out, float *omega_out, void *stream) {
    const size_t need = lorekv_workspace_size(shape, params);
    if (need == 0)  // invalid shape or parameters: let the regular entry point report why
        return lorekv_score(shape, params, K, V, Q_W, Q_look, L, G, logits, sampled, scores_out,
                            omega_out, nullptr, 0, stream);
    if (need > kNoallocScratchBytes)
        return kve::report_error(KVE_EWORKSPACE,
                                 "lorekv_score_noalloc: this shape needs %zu bytes of scratch; "
                                 "the fixed array holds %zu (use lorekv_score with a workspace)",
                                 need, kNoallocScratchBytes);
    void *scratch = kve::context_symbol_address(
        reinterpret_cast<const void *>(&g_noalloc_scratch), g_noalloc_cache);
    if (!scratch)
        return kve::report_error(KVE_ECUDA, "lorekv_score_noalloc: scratch address lookup failed (%s)",
                                 cudaGetErrorString(cudaGetLastError()));
    return lorekv_score(shape, params, K, V, Q_W, Q_look, L, G, logits, sampled, scores_out,
                        omega_out, scratch, kNoallocScratchBytes, stream);
}

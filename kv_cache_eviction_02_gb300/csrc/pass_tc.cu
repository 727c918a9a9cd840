// Tensor-core (tcgen05) kernels of the LORE-KV scoring pass. Not enabled yet: tc_supported()
// reports false and the CUDA-core kernels run for every shape.
#include "kve_internal.cuh"

namespace kve {

bool tc_supported(const LorekvDims &) { return false; }

cudaError_t launch_pack_queries(const LorekvDims &, const void *, const void *, void *,
                                const LorekvWorkspace &, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t launch_attention_tc(const LorekvDims &, const void *, const void *, void *,
                                const LorekvWorkspace &, unsigned *, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t launch_scores_tc(const LorekvDims &, const void *, const void *, const float *,
                             void *, const LorekvWorkspace &, float *, unsigned *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace kve

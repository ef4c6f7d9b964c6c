// draft_d256.cu -- keys-as-M draft kernel instantiations for head_dim 256 (one
// translation unit per head dim so that the library builds in parallel): the
// plain draft attention and the fused draft step, each with the products on
// the tensor cores (mma.sync) or on the CUDA cores (FMA).
#include "draft_kernel.cuh"

namespace wm {

cudaError_t launch_draft_d256(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                            const CUtensorMap &mv, const AttnParams &p, bool step, bool fma, cudaStream_t stream) {
    if (fma)
        return step ? launch_draft_kernel<256, true, true>(k, v, mk, mv, p, stream)
                    : launch_draft_kernel<256, false, true>(k, v, mk, mv, p, stream);
    return step ? launch_draft_kernel<256, true, false>(k, v, mk, mv, p, stream)
                : launch_draft_kernel<256, false, false>(k, v, mk, mv, p, stream);
}

int draft_blocks_per_sm_d256(bool step, bool fma) {
    if (fma) return step ? draft_blocks_per_sm_t<256, true, true>() : draft_blocks_per_sm_t<256, false, true>();
    return step ? draft_blocks_per_sm_t<256, true, false>() : draft_blocks_per_sm_t<256, false, false>();
}

}  // namespace wm

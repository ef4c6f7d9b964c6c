// draft_d64.cu -- keys-as-M draft kernel instantiations for head_dim 64 (one
// translation unit per head dim so that the library builds in parallel): the
// plain draft attention and the fused draft step.
#include "draft_kernel.cuh"

namespace wm {

cudaError_t launch_draft_d64(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                            const CUtensorMap &mv, const AttnParams &p, bool step, cudaStream_t stream) {
    return step ? launch_draft_kernel<64, true>(k, v, mk, mv, p, stream)
                : launch_draft_kernel<64, false>(k, v, mk, mv, p, stream);
}

int draft_blocks_per_sm_d64(bool step) {
    return step ? draft_blocks_per_sm_t<64, true>() : draft_blocks_per_sm_t<64, false>();
}

}  // namespace wm

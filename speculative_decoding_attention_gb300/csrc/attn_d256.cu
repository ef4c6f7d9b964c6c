// attn_d256.cu -- attention kernel instantiations for head_dim 256 (one translation
// unit per head dim so that the library builds in parallel): split-KV attention
// and the fused draft step.
#include "attn_kernel.cuh"

namespace wm {

cudaError_t launch_attn_d256(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                            const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream) {
    return launch_attn<256>(k, v, mk, mv, p, m_tiles, stream);
}

cudaError_t launch_step_d256(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                            const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream) {
    return launch_step<256>(k, v, mk, mv, p, m_tiles, stream);
}

int attn_blocks_per_sm_d256(int m_tiles, bool step) { return blocks_per_sm<256>(m_tiles, step); }

}  // namespace wm

// attn_d64.cu -- attention kernel instantiations for head_dim 64 (one translation
// unit per head dim so that the library builds in parallel): split-KV attention
// and the fused draft step.
#include "attn_kernel.cuh"

namespace wm {

cudaError_t launch_attn_d64(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                            const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream) {
    return launch_attn<64>(k, v, mk, mv, p, m_tiles, stream);
}

cudaError_t launch_step_d64(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                            const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream) {
    return launch_step<64>(k, v, mk, mv, p, m_tiles, stream);
}

int attn_blocks_per_sm_d64(int m_tiles, bool step) { return blocks_per_sm<64>(m_tiles, step); }

}  // namespace wm

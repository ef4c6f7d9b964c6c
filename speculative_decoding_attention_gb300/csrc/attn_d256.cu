// attn_d256.cu -- attention kernel instantiations for head_dim 256 (one translation
// unit per head dim so that the library builds in parallel).
#include "attn_kernel.cuh"

namespace wm {

cudaError_t launch_attn_d256(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p,
                            int m_tiles, cudaStream_t stream) {
    return launch_attn<256>(k, v, p, m_tiles, stream);
}

}  // namespace wm

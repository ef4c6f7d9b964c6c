// attn_d64.cu -- attention kernel instantiations for head_dim 64 (one translation
// unit per head dim so that the library builds in parallel).
#include "attn_kernel.cuh"

namespace wm {

cudaError_t launch_attn_d64(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p,
                            int m_tiles, cudaStream_t stream) {
    return launch_attn<64>(k, v, p, m_tiles, stream);
}

}  // namespace wm

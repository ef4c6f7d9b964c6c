// attn_tc_d128.cu -- tensor-core attention kernel instantiations for head_dim 128.
#include "attn_tc.cuh"

namespace wm {

cudaError_t launch_attn_tc_d128(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p, int n_rows16,
                               cudaStream_t stream) {
    return launch_attn_tc<128>(k, v, p, n_rows16, stream);
}

int attn_tc_blocks_per_sm_d128(int n_rows16) { return tc_blocks_per_sm<128>(n_rows16); }

}  // namespace wm

// attn_tcp_d128.cu -- persistent tensor-core verify instantiations for head_dim 128.
#include "attn_tcp.cuh"

namespace wm {

cudaError_t launch_attn_tcp_d128(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p, int n_rows16,
                                 int n_cta, cudaStream_t stream) {
    switch (n_rows16) {
        case 16: return launch_attn_tcp_nr<128, 16>(k, v, p, n_cta, stream);
        case 32: return launch_attn_tcp_nr<128, 32>(k, v, p, n_cta, stream);
        case 48: return launch_attn_tcp_nr<128, 48>(k, v, p, n_cta, stream);
        case 64: return launch_attn_tcp_nr<128, 64>(k, v, p, n_cta, stream);
        default: return cudaErrorInvalidValue;
    }
}

int attn_tcp_blocks_per_sm_d128(int n_rows16) {
    switch (n_rows16) {
        case 16: return tcp_blocks_per_sm_nr<128, 16>();
        case 32: return tcp_blocks_per_sm_nr<128, 32>();
        case 48: return tcp_blocks_per_sm_nr<128, 48>();
        case 64: return tcp_blocks_per_sm_nr<128, 64>();
        default: return 0;
    }
}

}  // namespace wm

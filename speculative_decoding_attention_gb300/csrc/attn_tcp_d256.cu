// attn_tcp_d256.cu -- persistent tensor-core verify instantiations for head_dim 256
// (up to 32 rows per KV head; more rows stage V in half tiles, which the
// persistent kernel does not).
#include "attn_tcp.cuh"

namespace wm {

cudaError_t launch_attn_tcp_d256(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p, int n_rows16,
                                 int n_cta, cudaStream_t stream) {
    switch (n_rows16) {
        case 16: return launch_attn_tcp_nr<256, 16>(k, v, p, n_cta, stream);
        case 32: return launch_attn_tcp_nr<256, 32>(k, v, p, n_cta, stream);
        default: return cudaErrorInvalidValue;
    }
}

int attn_tcp_blocks_per_sm_d256(int n_rows16) {
    switch (n_rows16) {
        case 16: return tcp_blocks_per_sm_nr<256, 16>();
        case 32: return tcp_blocks_per_sm_nr<256, 32>();
        default: return 0;
    }
}

}  // namespace wm

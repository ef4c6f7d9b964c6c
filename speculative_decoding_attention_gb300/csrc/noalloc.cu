// noalloc.cu -- draft attention with library-owned scratch, for callers that
// cannot allocate device memory (see wm_draft_attn_static in wm_api.h).
//
// The split partials of wm_draft_attn normally go to a caller-provided
// workspace.  Here they go to `g_static_scratch`, a fixed-size array that
// every device holds for the life of the process.  In host code the array's
// name is only a host-side stand-in, so the device address is looked up with
// cudaGetSymbolAddress once per device and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/wm_api.h"
#include "wm_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[WM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device, or nullptr.
void *static_scratch_ptr() {
    static void *ptrs[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return nullptr;
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

}  // namespace

extern "C" wm_status wm_draft_attn_static(const wm_ring *ring, const void *q, int32_t n_q_heads,
                                          float scale, int32_t n_split, void *out, float *lse,
                                          void *stream) {
    // The same host-side checks as wm_draft_attn, first: a bad argument is
    // reported as such, never as a scratch-size problem.
    const int32_t args = wm::draft_args_status(ring, q, n_q_heads, scale, n_split, out, lse);
    if (args != WM_OK) return static_cast<wm_status>(args);
    const size_t need = wm_workspace_size(WM_OP_DRAFT, ring->batch, ring->n_kv_heads, n_q_heads, 1,
                                          ring->head_dim, (int64_t)ring->sink + ring->window, n_split);
    if (need == (size_t)-1) return WM_ERR_INVALID_ARG;
    if (need > WM_STATIC_SCRATCH_BYTES) return WM_ERR_WORKSPACE;
    void *scratch = static_scratch_ptr();
    if (!scratch) return WM_ERR_CUDA;
    return wm_draft_attn(ring, q, n_q_heads, scale, n_split, out, lse, scratch, WM_STATIC_SCRATCH_BYTES,
                         stream);
}

// mem.cu -- the memory-slot store of a memory-augmented sliding-window draft
// ("Strong Drafts Need Compact Memories: Long-Context Speculative Decoding
// with Compressed KV Cache", 4.2-4.3): at every r-token
// boundary the draft's adaptor materializes one compressed memory slot, which
// stays after the raw tokens it summarizes leave the window; on rejection the
// slots materialized after the accepted prefix are discarded.
//
// Layout (per sequence b): K, V [Hkv][capacity][D] bf16, count int64 (slots
// materialized so far).  Slot i lives at index i.
#include "launch.h"
#include "ptx.cuh"
#include "wm_internal.h"
#include "../../include/wm_api.h"

namespace wm {

namespace {

__device__ __forceinline__ void report(int32_t *err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// One CTA per sequence: slot count[b] <- (k_new[b], v_new[b]) for every KV
// head, then count[b] + 1.  A full store (or a negative count) is recorded as
// a data error and left unchanged.
__global__ void mem_append_kernel(uint4 *mk, uint4 *mv, int64_t *count, int64_t capacity, int n_kv_heads,
                                  int head_dim, const uint4 *kn, const uint4 *vn, int32_t *err) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int64_t c = count[b];
    if (c < 0 || c >= capacity) {
        if (threadIdx.x == 0) report(err, WM_DEVERR_BAD_LENGTH);
        return;
    }
    const int vpr = head_dim / 8;
    for (int idx = threadIdx.x; idx < n_kv_heads * vpr; idx += blockDim.x) {
        const int h = idx / vpr, v = idx - (idx / vpr) * vpr;
        const int64_t dst = (((int64_t)b * n_kv_heads + h) * capacity + c) * vpr + v;
        const int64_t src = ((int64_t)b * n_kv_heads + h) * vpr + v;
        mk[dst] = kn[src];
        mv[dst] = vn[src];
    }
    __syncthreads();  // every thread has read count[b] before it changes
    if (threadIdx.x == 0) count[b] = c + 1;
}

// count[b] = min(count[b], new_count[b]) for each sequence (one thread each).
__global__ void mem_rollback_kernel(int64_t *count, int batch, const int64_t *new_count, int32_t *err) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int64_t nc = new_count[b];
    if (nc < 0) {
        report(err, WM_DEVERR_BAD_LENGTH);
        return;
    }
    const int64_t c = count[b];
    count[b] = c < nc ? c : nc;
}

}  // namespace

cudaError_t launch_mem_append(void *mk, void *mv, int64_t *count, int64_t capacity, int batch, int n_kv_heads,
                              int head_dim, const void *k_new, const void *v_new, int32_t *err,
                              cudaStream_t stream) {
    return launch_pdl(mem_append_kernel, dim3(batch), dim3(128), 0, stream, static_cast<uint4 *>(mk),
                      static_cast<uint4 *>(mv), count, capacity, n_kv_heads, head_dim,
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), err);
}

cudaError_t launch_mem_rollback(int64_t *count, int batch, const int64_t *new_count, int32_t *err,
                                cudaStream_t stream) {
    return launch_pdl(mem_rollback_kernel, dim3((batch + 127) / 128), dim3(128), 0, stream, count, batch,
                      new_count, err);
}

}  // namespace wm

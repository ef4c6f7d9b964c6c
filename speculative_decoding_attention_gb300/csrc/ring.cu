// ring.cu -- the draft's compact ring buffer: append, bulk fill, rollback.
//
// Layout (per sequence b): K, V [Hkv][S + W][D] bf16, pos_tag [S + W] int32,
// n_seen int64.  Position p lives in slot p if p < S, else in slot
// S + (p - S) mod W, so the ring always holds the attention sinks and the W
// most recent positions ("Windowed-MTP: Removing the Full-Context Draft-KV Tax
// at Million-Token Context", Abstract: the unread draft KV is reclaimed via a
// compact ring buffer).
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"
#include "wm_internal.h"
#include "../../include/wm_api.h"

namespace wm {

namespace {

__device__ __forceinline__ void report(int32_t *err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ int64_t slot_of(int64_t p, int sink, int window) {
    return p < sink ? p : sink + (p - sink) % window;
}

// Latest position among 0..n-1 whose slot is s, or -1 if no such position.
__device__ __forceinline__ int64_t latest_in_slot(int64_t s, int64_t n, int sink, int window) {
    if (s < sink) return s < n ? s : -1;
    const int64_t w = s - sink;
    if (n - 1 < sink + w) return -1;
    return sink + w + ((n - 1 - sink - w) / window) * window;
}

__global__ void ring_append_kernel(uint4 *rk, uint4 *rv, int32_t *tag, int64_t *n_seen, int n_kv_heads,
                                   int head_dim, int sink, int window, const uint4 *kn,
                                   const uint4 *vn, int32_t *err) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int n_slots = sink + window;
    const int64_t p = n_seen[b];
    if (p < 0 || p >= INT32_MAX) {  // tags are int32: the last position a ring can hold is INT32_MAX - 1
        if (threadIdx.x == 0) report(err, WM_DEVERR_BAD_LENGTH);
        return;
    }
    const int64_t slot = slot_of(p, sink, window);
    const int vpr = head_dim / 8;  // 16-byte vectors per row
    for (int idx = threadIdx.x; idx < n_kv_heads * vpr; idx += blockDim.x) {
        const int h = idx / vpr, v = idx - (idx / vpr) * vpr;
        const int64_t dst = (((int64_t)b * n_kv_heads + h) * n_slots + slot) * vpr + v;
        const int64_t src = ((int64_t)b * n_kv_heads + h) * vpr + v;
        rk[dst] = kn[src];
        rv[dst] = vn[src];
    }
    __syncthreads();  // every thread has read n_seen[b] before it changes
    if (threadIdx.x == 0) {
        tag[(int64_t)b * n_slots + slot] = (int32_t)p;
        n_seen[b] = p + 1;
    }
}

constexpr int kFillSlots = 32;  // slots per block in the bulk fill

__global__ void ring_fill_kernel(uint4 *rk, uint4 *rv, int32_t *tag, int64_t *n_seen, int n_kv_heads,
                                 int head_dim, int sink, int window, HistSource hist, int32_t *err) {
    pdl_wait();
    pdl_launch_dependents();
    const int unit = blockIdx.y;
    const int b = unit / n_kv_heads, h = unit - (unit / n_kv_heads) * n_kv_heads;
    const int n_slots = sink + window;
    const int vpr = head_dim / 8;
    const int64_t cap = hist.block_table ? (int64_t)hist.max_pages * hist.page_size : hist.n_cap;
    int64_t n = hist.lens[b];
    if (n < 0 || n > cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) report(err, WM_DEVERR_BAD_LENGTH);
        n = n < 0 ? 0 : cap;
    }
    const uint4 *hk = static_cast<const uint4 *>(hist.k);
    const uint4 *hv = static_cast<const uint4 *>(hist.v);
    const int s0 = blockIdx.x * kFillSlots;
    for (int idx = threadIdx.x; idx < kFillSlots * vpr; idx += blockDim.x) {
        const int s = s0 + idx / vpr, v = idx - (idx / vpr) * vpr;
        if (s >= n_slots) continue;
        const int64_t pos = latest_in_slot(s, n, sink, window);
        if (pos < 0) continue;
        int64_t src;
        if (hist.block_table) {
            const int32_t page = hist.block_table[(int64_t)b * hist.max_pages + pos / hist.page_size];
            if (page < 0 || page >= hist.n_pages) {
                report(err, WM_DEVERR_BAD_PAGE);
                continue;
            }
            src = (((int64_t)page * n_kv_heads + h) * hist.page_size + pos % hist.page_size) * vpr + v;
        } else {
            src = (((int64_t)b * n_kv_heads + h) * hist.n_cap + pos) * vpr + v;
        }
        const int64_t dst = (((int64_t)b * n_kv_heads + h) * n_slots + s) * vpr + v;
        rk[dst] = hk[src];
        rv[dst] = hv[src];
    }
    if (h == 0) {
        for (int i = threadIdx.x; i < kFillSlots; i += blockDim.x) {
            const int s = s0 + i;
            if (s < n_slots) tag[(int64_t)b * n_slots + s] = (int32_t)latest_in_slot(s, n, sink, window);
        }
        if (blockIdx.x == 0 && threadIdx.x == 0) n_seen[b] = n;
    }
}

constexpr int kRollbackThreads = 256;

// One thread per slot; block (0, b) also lowers n_seen[b].  No block reads
// n_seen, so the update cannot race with the tag clearing.
__global__ void ring_rollback_kernel(int32_t *tag, int64_t *n_seen, int n_slots, const int64_t *new_len,
                                     int32_t *err) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.y;
    const int64_t nl = new_len[b];
    if (nl < 0) {
        if (threadIdx.x == 0 && blockIdx.x == 0) report(err, WM_DEVERR_BAD_LENGTH);
        return;
    }
    const int s = blockIdx.x * kRollbackThreads + threadIdx.x;
    if (s < n_slots) {
        int32_t *t = tag + (int64_t)b * n_slots + s;
        if (*t >= nl) *t = -1;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int64_t seen = n_seen[b];
        n_seen[b] = seen < nl ? seen : nl;
    }
}

}  // namespace

cudaError_t launch_ring_append(void *rk, void *rv, int32_t *tag, int64_t *n_seen, int batch,
                               int n_kv_heads, int head_dim, int sink, int window, const void *k_new,
                               const void *v_new, int32_t *err, cudaStream_t stream) {
    return launch_pdl(ring_append_kernel, dim3(batch), dim3(128), 0, stream, static_cast<uint4 *>(rk),
                      static_cast<uint4 *>(rv), tag, n_seen, n_kv_heads, head_dim, sink, window,
                      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), err);
}

cudaError_t launch_ring_fill(void *rk, void *rv, int32_t *tag, int64_t *n_seen, int batch,
                             int n_kv_heads, int head_dim, int sink, int window, const HistSource &hist,
                             int32_t *err, cudaStream_t stream) {
    const int n_slots = sink + window;
    const dim3 grid((n_slots + kFillSlots - 1) / kFillSlots, batch * n_kv_heads);
    return launch_pdl(ring_fill_kernel, grid, dim3(256), 0, stream, static_cast<uint4 *>(rk),
                      static_cast<uint4 *>(rv), tag, n_seen, n_kv_heads, head_dim, sink, window, hist, err);
}

cudaError_t launch_ring_rollback(int32_t *tag, int64_t *n_seen, int batch, int n_slots,
                                 const int64_t *new_len, int32_t *err, cudaStream_t stream) {
    const dim3 grid((n_slots + kRollbackThreads - 1) / kRollbackThreads, batch);
    return launch_pdl(ring_rollback_kernel, grid, dim3(kRollbackThreads), 0, stream, tag, n_seen, n_slots,
                      new_len, err);
}

}  // namespace wm

// merge.cu -- log-sum-exp merge of split-KV partial attention results.
//
// Per row r with parts s = 0..n-1 (each part normalised by its own softmax sum):
//   M = max_s lse_s,  lse = M + ln sum_s exp(lse_s - M),  o = sum_s exp(lse_s - lse) o_s.
// A part with lse = -inf holds no key; it gets weight 0 and its o is not read.
//
// One CTA per (row, 32-column block).  Its 128 threads are 8 column threads
// (one float4 each) x 16 part groups, so the loads of different parts are
// independent and in flight together; the 16 group sums meet in shared
// memory.  Every CTA of a row recomputes the row's lse (n_parts floats).
//
// After a fused draft step the merge also commits the append: the first CTA
// of each sequence's rows advances n_seen[b] by one.  The attention grid has
// completed by then (this kernel waits for it), so no CTA of it can have
// read the new count.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"
#include "wm_internal.h"

namespace wm {

namespace {

constexpr int kColThreads = 8;     // float4 columns per CTA -> 32 columns
constexpr int kPartGroups = 16;
constexpr int kMergeThreads = kColThreads * kPartGroups;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__global__ void __launch_bounds__(kMergeThreads)
    lse_merge_kernel(const float *__restrict__ o_parts, const float *__restrict__ lse_parts, int n_parts,
                     int head_dim, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out,
                     int64_t *__restrict__ commit_n_seen, int rows_per_seq) {
    __shared__ float red[kMergeThreads / 32];
    __shared__ float4 acc_s[kPartGroups][kColThreads];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t r = blockIdx.x;
    const float *ls = lse_parts + r * n_parts;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (commit_n_seen && blockIdx.y == 0 && tid == 0 && r % rows_per_seq == 0) {
        const int64_t b = r / rows_per_seq;
        const int64_t seen = commit_n_seen[b];
        if (seen >= 0) commit_n_seen[b] = seen + 1;  // a negative count was reported, nothing appended
    }

    float mx = -CUDART_INF_F;
    for (int s = tid; s < n_parts; s += kMergeThreads) mx = fmaxf(mx, ls[s]);
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) mx = fmaxf(mx, red[w]);
    __syncthreads();
    float z = 0.f;
    if (mx != -CUDART_INF_F)
        for (int s = tid; s < n_parts; s += kMergeThreads) z += ex2((ls[s] - mx) * kLog2e);
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane == 0) red[warp] = z;
    __syncthreads();
    float zt = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) zt += red[w];
    const float lse = zt > 0.f ? mx + lg2(zt) * kLn2 : -CUDART_INF_F;

    const int ct = tid % kColThreads, pg = tid / kColThreads;
    const int col = (blockIdx.y * kColThreads + ct) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < head_dim && lse != -CUDART_INF_F) {
        const float *op = o_parts + r * (int64_t)n_parts * head_dim + col;
#pragma unroll 4
        for (int s = pg; s < n_parts; s += kPartGroups) {
            const float w = ex2((ls[s] - lse) * kLog2e);
            if (w == 0.f) continue;  // empty part (lse -inf): its o is never read
            const float4 v = __ldg(reinterpret_cast<const float4 *>(op + (int64_t)s * head_dim));
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
    }
    acc_s[pg][ct] = acc;
    __syncthreads();
    if (pg == 0 && col < head_dim) {
        float4 t = acc_s[0][ct];
#pragma unroll
        for (int g = 1; g < kPartGroups; ++g) {
            const float4 u = acc_s[g][ct];
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(t.x, t.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(t.z, t.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t *>(&lo);
        pk.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(out + r * head_dim + col) = pk;
    }
    if (blockIdx.y == 0 && tid == 0 && lse_out) lse_out[r] = lse;
}

}  // namespace

cudaError_t launch_lse_merge(const float *o_parts, const float *lse_parts, int n_parts, int64_t rows,
                             int head_dim, void *out, float *lse_out, int64_t *commit_n_seen, int rows_per_seq,
                             cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const dim3 grid((unsigned)rows, (unsigned)((head_dim + 4 * kColThreads - 1) / (4 * kColThreads)));
    return launch_pdl(lse_merge_kernel, grid, dim3(kMergeThreads), 0, stream, o_parts, lse_parts, n_parts,
                      head_dim, static_cast<__nv_bfloat16 *>(out), lse_out, commit_n_seen,
                      rows_per_seq > 0 ? rows_per_seq : 1);
}

}  // namespace wm

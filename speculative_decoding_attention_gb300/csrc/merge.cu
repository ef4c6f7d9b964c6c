// merge.cu -- log-sum-exp merge of split-KV partial attention results.
//
// Per row r with parts s = 0..n-1 (each part normalised by its own softmax sum):
//   M = max_s lse_s,  lse = M + ln sum_s exp(lse_s - M),  o = sum_s exp(lse_s - lse) o_s.
// A part with lse = -inf holds no key; it gets weight 0 (its o is loaded, not used).
//
// One CTA per (row, 32-column block).  Its 128 threads are 8 column threads
// (one float4 each) x 16 part groups.  Each thread folds its parts (every
// 16th) in batches of 8 with a running maximum -- a batch's lse and o loads
// do not depend on each other or on earlier parts, so they are all in flight
// together -- and the 16 group states (max, sum of weights, weighted o) meet
// in shared memory.
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
constexpr int kBatch = 8;         // parts per thread whose loads are in flight together
constexpr int kMergeThreads = kColThreads * kPartGroups;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__global__ void __launch_bounds__(kMergeThreads)
    lse_merge_kernel(const float *__restrict__ o_parts, const float *__restrict__ lse_parts, int n_parts,
                     int head_dim, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out,
                     int64_t *__restrict__ commit_n_seen, int rows_per_seq) {
    __shared__ float m_s[kPartGroups][kColThreads], z_s[kPartGroups][kColThreads];
    __shared__ float4 acc_s[kPartGroups][kColThreads];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x;
    if (commit_n_seen && blockIdx.y == 0 && tid == 0 && r % rows_per_seq == 0) {
        const int64_t b = r / rows_per_seq;
        const int64_t seen = commit_n_seen[b];
        // a count the attention kernel reported (negative, or past an int32 tag) appended nothing
        if (seen >= 0 && seen < INT32_MAX) commit_n_seen[b] = seen + 1;
    }
    const float *ls = lse_parts + r * n_parts;
    const int ct = tid % kColThreads, pg = tid / kColThreads;
    const int col = (blockIdx.y * kColThreads + ct) * 4;
    const bool in_cols = col < head_dim;
    const float *op = o_parts + r * (int64_t)n_parts * head_dim + (in_cols ? col : 0);

    // this group's parts, in log2 units: m = max lse, z = sum 2^(lse - m), acc = sum 2^(lse - m) o.
    // Parts are folded kBatch at a time: all of a batch's loads are issued
    // before any is used, so up to kBatch * kPartGroups parts cost one round
    // trip to L2.
    float m = -CUDART_INF_F, z = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = pg; s0 < n_parts; s0 += kBatch * kPartGroups) {
        float l[kBatch];
        float4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int s = s0 + j * kPartGroups;
            l[j] = s < n_parts ? __ldg(ls + s) * kLog2e : -CUDART_INF_F;
            v[j] = s < n_parts && in_cols ? __ldg(reinterpret_cast<const float4 *>(op + (int64_t)s * head_dim))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mb = m;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) mb = fmaxf(mb, l[j]);
        if (mb == -CUDART_INF_F) continue;  // no part with a key yet
        const float c = ex2(m - mb);         // 0 while m is -inf
        z *= c;
        acc.x *= c;
        acc.y *= c;
        acc.z *= c;
        acc.w *= c;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (l[j] == -CUDART_INF_F) continue;  // an empty part: its o was never written
            const float w = ex2(l[j] - mb);
            z += w;
            acc.x += w * v[j].x;
            acc.y += w * v[j].y;
            acc.z += w * v[j].z;
            acc.w += w * v[j].w;
        }
        m = mb;
    }
    m_s[pg][ct] = m;
    z_s[pg][ct] = z;
    acc_s[pg][ct] = acc;
    __syncthreads();
    if (pg != 0) return;
    float mt = -CUDART_INF_F;
#pragma unroll
    for (int g = 0; g < kPartGroups; ++g) mt = fmaxf(mt, m_s[g][ct]);
    float zt = 0.f;
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mt != -CUDART_INF_F) {
#pragma unroll
        for (int g = 0; g < kPartGroups; ++g) {
            const float c = ex2(m_s[g][ct] - mt);  // 0 for a group without a part
            const float4 u = acc_s[g][ct];
            zt += c * z_s[g][ct];
            t.x += c * u.x;
            t.y += c * u.y;
            t.z += c * u.z;
            t.w += c * u.w;
        }
    }
    const float inv = zt > 0.f ? 1.f / zt : 0.f;
    if (in_cols) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(t.x * inv, t.y * inv);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(t.z * inv, t.w * inv);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t *>(&lo);
        pk.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(out + r * head_dim + col) = pk;
    }
    if (blockIdx.y == 0 && ct == 0 && lse_out) lse_out[r] = zt > 0.f ? (mt + lg2(zt)) * kLn2 : -CUDART_INF_F;
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

// verify_sched.cu -- device-side work schedule of the verify attention over a
// batch of sequences, and the merge of its partials.
//
// The host sees only the largest sequence length, so a split plan made there
// covers every sequence as if it had that length: a short sequence leaves
// most of its splits empty, and how evenly the block scheduler pairs the long
// and short splits on the SMs decides the time.  Here the actual lengths are
// read once on the device.  The batch's key tiles are laid end to end -- unit
// u = b * n_kv_heads + kvh holds tiles_b = ceil(seq_len[b] / 128) tiles, unit
// after unit -- and the persistent verify grid of n_cta CTAs (every one
// resident at once) gives CTA c the run of `chunk` tiles starting at c *
// chunk, chunk = ceil(total / n_cta).  Every CTA then streams the same number
// of bytes, whatever the length mix.
//
// A run that crosses unit boundaries is cut into segments, one per unit it
// touches, and each segment leaves one partial (its rows' normalised output
// and log-sum-exp).  The segment of CTA c in unit u gets index c + u: along
// the concatenated tiles, each next segment starts at a new chunk (c + 1), a
// new unit (u + 1), or both, so the indices increase along the tiles, no two
// segments share one, and all stay below n_cta + units - 1.  The partials of
// unit u are those of the CTAs c0(u) .. c1(u) whose runs touch it -- c0 =
// first tile / chunk, c1 = last tile / chunk -- at indices c0 + u .. c1 + u.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"
#include "wm_internal.h"
#include "../../include/wm_api.h"

namespace wm {

namespace {

constexpr int kSchedThreads = 1024;

// Block-wide inclusive prefix sum of one int64 per thread; also returns the
// block's total.  Every thread of the block must call it.
__device__ int64_t block_inclusive_scan(int64_t v, int64_t *s_warp, int64_t &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int64_t r = (warp > 0 ? s_warp[warp - 1] : 0) + x;
    total = s_warp[31];
    __syncthreads();  // s_warp is reused by the next call
    return r;
}

// Batches up to this many sequences keep the prefix in shared memory for the
// CTAs' searches (larger ones read it back from global memory).
constexpr int kSchedSmemBatch = 2048;

// One CTA: tile prefix per sequence, the chunk, and each CTA's first tile.
//   sched[0] = chunk (tiles per CTA), sched[1] = total tiles,
//   sched[2 + b] = tiles of one KV head of the sequences before b (b = 0..batch).
//   cta_start[c] = (sequence, KV head, tile within that unit, tiles of the run);
//   a run of 0 tiles (total < n_cta * chunk) means no work.
__global__ void __launch_bounds__(kSchedThreads)
    verify_sched_kernel(const int64_t *__restrict__ seq_lens, int batch, int n_kv_heads, int64_t capacity, int n_cta,
                        int64_t *__restrict__ sched, int4 *__restrict__ cta_start, int32_t *__restrict__ err) {
    __shared__ int64_t s_warp[32];
    __shared__ int64_t s_prefix[kSchedSmemBatch + 1];
    pdl_wait();  // the lengths may come from the previous kernel
    pdl_launch_dependents();
    int64_t *prefix = sched + 2;
    const bool in_smem = batch <= kSchedSmemBatch;
    int64_t carry = 0;
    for (int base = 0; base < batch; base += kSchedThreads) {
        const int b = base + (int)threadIdx.x;
        int64_t nt = 0;
        if (b < batch) {
            int64_t len = seq_lens[b];
            if (len < 0 || len > capacity) {
                if (err) atomicCAS(err, 0, WM_DEVERR_BAD_LENGTH);
                len = len < 0 ? 0 : capacity;  // the same clamp as the verify kernel's
            }
            nt = (len + kTcTile - 1) / kTcTile;
        }
        int64_t block_total = 0;
        const int64_t incl = block_inclusive_scan(nt, s_warp, block_total);
        if (b < batch) {
            prefix[b] = carry + incl - nt;
            if (in_smem) s_prefix[b] = carry + incl - nt;
        }
        carry += block_total;
    }
    const int64_t total = carry * n_kv_heads;
    const int64_t chunk = total > 0 ? (total + n_cta - 1) / n_cta : 1;
    if (threadIdx.x == 0) {
        prefix[batch] = carry;
        if (in_smem) s_prefix[batch] = carry;
        sched[0] = chunk;
        sched[1] = total;
    }
    __syncthreads();  // every prefix entry visible to the whole CTA
    const int64_t *pf = in_smem ? s_prefix : prefix;
    for (int c = threadIdx.x; c < n_cta; c += kSchedThreads) {
        const int64_t t0 = (int64_t)c * chunk;
        int4 v = make_int4(0, 0, 0, 0);
        if (t0 < total) {
            // the first sequence b with n_kv_heads * prefix[b + 1] > t0 (it has tiles)
            int lo = 0, hi = batch - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if ((int64_t)n_kv_heads * pf[mid + 1] > t0)
                    hi = mid;
                else
                    lo = mid + 1;
            }
            const int64_t nt = pf[lo + 1] - pf[lo];
            const int64_t within = t0 - (int64_t)n_kv_heads * pf[lo];
            const int64_t kvh = within / nt;
            v = make_int4(lo, (int)kvh, (int)(within - kvh * nt), (int)min(chunk, total - t0));
        }
        cta_start[c] = v;
    }
}

// Merge of the segment partials: one warp per output row, lane l holding
// columns 4l .. 4l + 3 of every 128 (head_dim 128 or 256), eight rows per CTA.
// A row has few parts (the CTAs whose runs touch its unit), so its lse and o
// loads are issued kSegBatch parts at a time and folded with a running maximum.
constexpr int kSegRows = 8;
constexpr int kSegBatch = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int NV>  // float4 columns per lane: head_dim / 128
__global__ void __launch_bounds__(32 * kSegRows)
    seg_merge_kernel(const float *__restrict__ o_seg, const float *__restrict__ lse_seg,
                     const int64_t *__restrict__ sched, int n_kv_heads, int n_q, int n_q_heads, int group, int rows_u,
                     int64_t rows, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out) {
    constexpr int D = 128 * NV;
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kSegRows + (threadIdx.x >> 5);
    if (r >= rows) return;
    // output row r = (b * n_q + qi) * n_q_heads + head; its unit and its row in the unit
    const int64_t per_b = (int64_t)n_q * n_q_heads;
    const int b = (int)(r / per_b);
    const int rem = (int)(r - (int64_t)b * per_b);
    const int qi = rem / n_q_heads, head = rem - qi * n_q_heads;
    const int kvh = head / group, hh = head - kvh * group;
    const int ru = qi * group + hh;
    const int64_t u = (int64_t)b * n_kv_heads + kvh;
    const int64_t chunk = sched[0];
    const int64_t nt = sched[2 + b + 1] - sched[2 + b];
    int64_t s_first = 0;
    int n_parts = 0;
    if (nt > 0) {
        const int64_t start = (int64_t)n_kv_heads * sched[2 + b] + kvh * nt;
        const int64_t c0 = start / chunk, c1 = (start + nt - 1) / chunk;
        n_parts = (int)(c1 - c0 + 1);
        s_first = c0 + u;
    }
    const float *ls = lse_seg + s_first * rows_u + ru;
    const float *op = o_seg + (s_first * rows_u + ru) * D + 4 * lane;
    const int64_t o_stride = (int64_t)rows_u * D;

    float m = -CUDART_INF_F, z = 0.f;
    float4 acc[NV];
#pragma unroll
    for (int c = 0; c < NV; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < n_parts; j0 += kSegBatch) {
        float l[kSegBatch];
        float4 v[kSegBatch][NV];
#pragma unroll
        for (int j = 0; j < kSegBatch; ++j) {
            const bool in = j0 + j < n_parts;
            l[j] = in ? __ldg(ls + (int64_t)(j0 + j) * rows_u) * kLog2e : -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < NV; ++c)
                v[j][c] = in ? __ldg(reinterpret_cast<const float4 *>(op + (j0 + j) * o_stride + 128 * c))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mb = m;
#pragma unroll
        for (int j = 0; j < kSegBatch; ++j) mb = fmaxf(mb, l[j]);
        if (mb == -CUDART_INF_F) continue;  // no part with a key yet
        const float cs = ex2(m - mb);       // 0 while m is -inf
        z *= cs;
#pragma unroll
        for (int c = 0; c < NV; ++c) {
            acc[c].x *= cs;
            acc[c].y *= cs;
            acc[c].z *= cs;
            acc[c].w *= cs;
        }
#pragma unroll
        for (int j = 0; j < kSegBatch; ++j) {
            if (l[j] == -CUDART_INF_F) continue;  // a segment none of whose keys this row sees
            const float w = ex2(l[j] - mb);
            z += w;
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                acc[c].x += w * v[j][c].x;
                acc[c].y += w * v[j][c].y;
                acc[c].z += w * v[j][c].z;
                acc[c].w += w * v[j][c].w;
            }
        }
        m = mb;
    }
    const float inv = z > 0.f ? 1.f / z : 0.f;
#pragma unroll
    for (int c = 0; c < NV; ++c) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[c].x * inv, acc[c].y * inv);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[c].z * inv, acc[c].w * inv);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t *>(&lo);
        pk.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(out + r * D + 128 * c + 4 * lane) = pk;
    }
    if (lane == 0 && lse_out) lse_out[r] = z > 0.f ? (m + lg2(z)) * kLn2 : -CUDART_INF_F;
}

}  // namespace

cudaError_t launch_verify_sched(const int64_t *seq_lens, int batch, int n_kv_heads, int64_t capacity, int n_cta,
                                int64_t *sched, int4 *cta_start, int32_t *err, cudaStream_t stream) {
    return launch_pdl(verify_sched_kernel, dim3(1), dim3(kSchedThreads), 0, stream, seq_lens, batch, n_kv_heads,
                      capacity, n_cta, sched, cta_start, err);
}

cudaError_t launch_seg_merge(const float *o_seg, const float *lse_seg, const int64_t *sched, int batch,
                             int n_kv_heads, int n_q, int n_q_heads, int head_dim, void *out, float *lse_out,
                             cudaStream_t stream) {
    const int64_t rows = (int64_t)batch * n_q * n_q_heads;
    if (rows == 0) return cudaSuccess;
    const int group = n_q_heads / n_kv_heads;
    const dim3 grid((unsigned)((rows + kSegRows - 1) / kSegRows));
    auto *o = static_cast<__nv_bfloat16 *>(out);
    switch (head_dim) {
        case 128:
            return launch_pdl(seg_merge_kernel<1>, grid, dim3(32 * kSegRows), 0, stream, o_seg, lse_seg, sched,
                              n_kv_heads, n_q, n_q_heads, group, n_q * group, rows, o, lse_out);
        case 256:
            return launch_pdl(seg_merge_kernel<2>, grid, dim3(32 * kSegRows), 0, stream, o_seg, lse_seg, sched,
                              n_kv_heads, n_q, n_q_heads, group, n_q * group, rows, o, lse_out);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace wm

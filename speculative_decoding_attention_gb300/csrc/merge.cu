// merge.cu -- log-sum-exp merge of split-KV partial attention results.
//
// Per row r with parts s = 0..n-1 (each part normalised by its own softmax sum):
//   M = max_s lse_s,  lse = M + ln sum_s exp(lse_s - M),  o = sum_s exp(lse_s - lse) o_s.
// A part with lse = -inf holds no key and gets weight 0.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "ptx.cuh"
#include "wm_internal.h"

namespace wm {

namespace {

constexpr int kMergeThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__global__ void __launch_bounds__(kMergeThreads)
    lse_merge_kernel(const float *__restrict__ o_parts, const float *__restrict__ lse_parts, int n_parts,
                     int head_dim, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out) {
    extern __shared__ float weight[];  // [n_parts]
    __shared__ float red[kMergeThreads / 32];
    __shared__ float s_lse;
    const int64_t r = blockIdx.x;
    const float *ls = lse_parts + r * n_parts;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    float mx = -CUDART_INF_F;
    for (int s = threadIdx.x; s < n_parts; s += blockDim.x) mx = fmaxf(mx, ls[s]);
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
    for (int w = 1; w < kMergeThreads / 32; ++w) mx = fmaxf(mx, red[w]);
    __syncthreads();

    float z = 0.f;
    if (mx != -CUDART_INF_F)
        for (int s = threadIdx.x; s < n_parts; s += blockDim.x) z += ex2((ls[s] - mx) * kLog2e);
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane == 0) red[warp] = z;
    __syncthreads();
    if (threadIdx.x == 0) {
        float zt = 0.f;
        for (int w = 0; w < kMergeThreads / 32; ++w) zt += red[w];
        s_lse = zt > 0.f ? mx + lg2(zt) * kLn2 : -CUDART_INF_F;
    }
    __syncthreads();
    const float lse = s_lse;
    for (int s = threadIdx.x; s < n_parts; s += blockDim.x)
        weight[s] = lse == -CUDART_INF_F ? 0.f : ex2((ls[s] - lse) * kLog2e);
    __syncthreads();

    const float *op = o_parts + r * (int64_t)n_parts * head_dim;
    for (int d = threadIdx.x; d < head_dim; d += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < n_parts; ++s) {
            const float w = weight[s];
            if (w != 0.f) acc += w * op[(int64_t)s * head_dim + d];
        }
        out[r * head_dim + d] = __float2bfloat16_rn(acc);
    }
    if (threadIdx.x == 0 && lse_out) lse_out[r] = lse;
}

}  // namespace

cudaError_t launch_lse_merge(const float *o_parts, const float *lse_parts, int n_parts, int64_t rows,
                             int head_dim, void *out, float *lse_out, const int32_t *,
                             cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (size_t)n_parts;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(lse_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    lse_merge_kernel<<<(unsigned)rows, kMergeThreads, smem, stream>>>(
        o_parts, lse_parts, n_parts, head_dim, static_cast<__nv_bfloat16 *>(out), lse_out);
    return cudaGetLastError();
}

}  // namespace wm

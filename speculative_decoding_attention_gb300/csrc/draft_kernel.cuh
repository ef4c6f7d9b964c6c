// draft_kernel.cuh -- the windowed draft attention for up to 8 query rows per
// KV head, keys on the MMA's M dimension.
//
// One CTA handles one (sequence, KV head) pair and one contiguous range of the
// ring's slots (a split); its rows are the G <= 8 query heads that read this
// KV head (the draft has one query position).  With so few rows the
// row-major product S = Q K^T would spend half of every m16 tile on padding
// rows, so both products are taken transposed, the keys as M and the rows as
// the MMA's N = 8:
//     S^T[16 keys x 8 rows]  = K[16 keys x D] . Q^T[D x 8 rows]
//     O^T[D x 8 rows]       += V^T[D x 16 keys] . P^T[16 keys x 8 rows]
// (mma.sync m16n8k16, bf16 in, fp32 accumulate).  Q^T is the B operand of
// every S product, so it is loaded once into registers; P^T leaves the S
// accumulator as bf16 pairs and becomes the B operand of the P.V product
// after an in-register 8x8 transpose (movmatrix), without a trip through
// shared memory.
//
// Warp roles (5 warps):
//   warp 4 (producer)  : one lane streams 64-key K and V tiles of the ring (or
//                        of the memory-slot store) into a ring of shared-memory
//                        stages with TMA, one "full" mbarrier per stage.
//   warps 0-3 (compute): warp w owns keys 16w..16w+15 of every tile, end to
//                        end: its S^T block, the masks, its own online softmax
//                        (running row maximum raised only when a logit exceeds
//                        it by more than 2^8, so the O^T accumulators are
//                        rarely rescaled), and its own O^T accumulators over
//                        the whole head dim.  No barrier between the compute
//                        warps inside the tile loop: each hands a stage back
//                        with its own arrival on the stage's "empty" barrier.
// At the end the four warps' states meet once in shared memory (the staging
// area, free by then): row maxima, sums and O^T, combined in a fixed order.
// The split's normalised output and log-sum-exp go to the bf16 output (one
// split) or to fp32 partials that the merge kernel combines.  Splits are
// balanced: of T = q n + r key tiles, the first r of the n splits take q + 1
// tiles and the others q, so every planned count is realised with at most one
// tile of difference.
//
// P goes into the P.V product as two bf16 parts, hi = bf16(p) and
// lo = bf16(p - hi), so the weights keep ~2^-17 relative accuracy.
//
// Masks: a ring slot with tag t is a key of the query at position p iff
// 0 <= t <= p and (t < sink or t > p - window); memory slots (keys at or
// beyond mem_base, below mem_base + count) are always keys.  A key masked for
// every row has its V^T operand elements zeroed in registers, so stale or
// uninitialised ring bytes (even NaN patterns) cannot reach the output
// through 0 * NaN.
//
// Fused draft step (STEP): every CTA reads p = n_seen[b] and treats slot(p)
// as holding p.  The warp whose keys include slot(p) writes the new K and V
// rows over the stale ones in the staged tile before its S product, and
// after its last tile stores them (and the tag) into the ring.  The merge
// kernel then commits n_seen[b] = p + 1.
//
// Set-up that reads only kernel parameters and shared memory (the split's
// planned key range, the barriers, the tensor-map prefetches, the L2 policy)
// runs before griddepcontrol.wait, while the previous kernel drains.
//
// FMA = true (wm_set_draft_math): the same producer, stages, masks and combine
// with both products on the CUDA cores.  Lane (k, g) of a compute warp takes
// the logits of the warp's key k for rows 4g .. 4g + 3 (fp32 FMA over the head
// dim, Q held as fp32 in shared memory), the row maxima over the warp's 16
// keys come from warp shuffles, and for P.V each lane owns D/32 head-dim
// columns of all 8 rows and reads P back from a per-warp shared buffer.  It
// computes the same attention and is kept to measure the choice of tensor
// cores for the draft.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"
#include "wm_internal.h"
#include "../../include/wm_api.h"

namespace wm {

// Rows (query heads per KV head) the keys-as-M draft kernel serves: the N of its mma.
constexpr int kDraftRows = kDraftRowsMax;

// FMA = true: the same kernel with the products on the CUDA cores (fp32 FMA,
// warp-shuffle softmax) instead of mma.sync; kept to measure that choice.
template <int D, bool FMA = false>
struct DraftCfg {
    static constexpr int TK = kKeyTile;                 // keys per stage
    static constexpr int NW = kConsumerWarps;           // compute warps
    static constexpr int KW = TK / NW;                  // keys per warp per tile (the M of one mma)
    static constexpr int NCH = D / 64;                  // 128-byte chunks per key row
    static constexpr int KSTEPS = D / 16;               // k-steps of S^T, m-tiles of O^T
    static constexpr int TILE_BYTES = TK * D * 2;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K + V
    // 64 KB of staging at head_dim 64 and 128 (three CTAs per SM), 128 KB at 256
    static constexpr int STAGES = (D == 256 ? 128 * 1024 : 64 * 1024) / STAGE_BYTES;
    static constexpr int MIN_BLOCKS = D == 256 ? 1 : 3;
    // final combine: per warp, rows x (D + 4) fp32 (the pad spreads the rows over banks)
    static constexpr int OB_STRIDE = D + 4;  // 16-byte aligned rows
    static constexpr int OB_BYTES = NW * kDraftRows * OB_STRIDE * 4;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int FLAG_OFF = BAR_OFF + 2 * STAGES * 8;
    static constexpr int RED_OFF = FLAG_OFF + 16;       // m[NW][8], l[NW][8]
    static constexpr int Q32_OFF = RED_OFF + 2 * NW * kDraftRows * 4;       // FMA: Q as fp32 [8][D]
    static constexpr int PS_OFF = Q32_OFF + (FMA ? kDraftRows * D * 4 : 0);  // FMA: P [NW][16 keys][8 rows]
    static constexpr int TOTAL = PS_OFF + (FMA ? NW * KW * kDraftRows * 4 : 0) + 1024;  // + slack to 1024-align
    static constexpr int DL = D / 32;                   // FMA: head-dim columns per lane in P.V
    static_assert(KW == 16, "one m16 block of keys per warp");
    static_assert(OB_BYTES <= STAGES * STAGE_BYTES, "the combine reuses the staging area");
    static_assert(STAGES >= 2, "double buffering at least");
    static_assert(TOTAL <= 227 * 1024, "shared memory budget");
    static_assert(Q32_OFF % 16 == 0 && PS_OFF % 16 == 0, "16-byte vectors");
};

__device__ __forceinline__ void draft_report(int32_t *err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int D, bool STEP, bool FMA>
__global__ void __launch_bounds__(kThreads, DraftCfg<D, FMA>::MIN_BLOCKS)
    draft_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 const __grid_constant__ CUtensorMap tmk2, const __grid_constant__ CUtensorMap tmv2,
                 const AttnParams p) {
    using C = DraftCfg<D, FMA>;
    constexpr int TK = C::TK;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw);
    const uint32_t bar_full = sbase + C::BAR_OFF;
    const uint32_t bar_empty = bar_full + 8 * C::STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::FLAG_OFF);
    float *red_m = reinterpret_cast<float *>(gbase + C::RED_OFF);
    float *red_l = red_m + C::NW * kDraftRows;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int unit = blockIdx.y;
    const int b = unit / p.n_kv_heads;
    const int kvh = unit - b * p.n_kv_heads;
    const int split = blockIdx.x;

    // ---- set-up that reads only kernel parameters and this CTA's shared
    // memory runs before the wait on the previous kernel, while it drains:
    // the split's planned key range, the pipeline barriers, the tensor-map
    // prefetches and the L2 policy
    // balanced splits: T = q n + r tiles; the first r splits take q + 1 tiles, the rest q
    const int32_t tq = p.plan_tiles / p.n_split, tr = p.plan_tiles - tq * p.n_split;
    const int32_t t_first = split * tq + min(split, tr);
    const int64_t k_begin = (int64_t)t_first * TK;
    const int64_t k_end_plan = (int64_t)(t_first + tq + (split < tr ? 1 : 0)) * TK;
    const int64_t mem_lo = p.mem_count ? p.mem_base : INT64_MAX;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, C::NW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    uint64_t policy = 0;
    if (warp == C::NW && lane == 0) {
        if (k_begin < mem_lo) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        if (k_end_plan > mem_lo) {
            prefetch_tensormap(&tmk2);
            prefetch_tensormap(&tmv2);
        }
        policy = l2_policy_evict_normal();  // the next draft step reads the ring again: normal L2 priority
    }
    __syncthreads();

    pdl_wait();  // every global read below may depend on the previous kernel
    pdl_launch_dependents();

    // ---- keys of this split: the ring's slots, then (memory draft) the
    // materialized memory slots from mem_base on
    int64_t n_keys = p.n_slots;
    if (p.mem_count) {
        int64_t mc = p.mem_count[b];
        if (mc < 0 || mc > p.mem_cap) {
            if (threadIdx.x == 0) draft_report(p.err, WM_DEVERR_BAD_LENGTH);
            mc = mc < 0 ? 0 : p.mem_cap;
        }
        n_keys = p.mem_base + mc;
    }
    const int64_t k_end = min(k_end_plan, n_keys);
    const int n_tiles = k_end > k_begin ? (int)((k_end - k_begin + TK - 1) / TK) : 0;

    // =========================================================== producer warp
    if (warp == C::NW) {
        if (lane == 0 && n_tiles > 0) {
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                if (t == p.stall_tile) break;  // tests of the timeout path only
                const int s = t % C::STAGES;
                if (t >= C::STAGES &&
                    !mbar_wait_bounded(bar_empty + 8 * s, ((t / C::STAGES) & 1) ^ 1, p.wait_limit)) {
                    draft_report(p.err, WM_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const int64_t key0 = k_begin + (int64_t)t * TK;
                const bool mem = key0 >= mem_lo;  // a tile is all ring or all memory
                const int c_row = (int)(mem ? key0 - mem_lo : key0);
                const CUtensorMap *mk = mem ? &tmk2 : &tmk;
                const CUtensorMap *mv = mem ? &tmv2 : &tmv;
                const uint32_t sK = sbase + s * C::STAGE_BYTES;
                const uint32_t sV = sK + C::TILE_BYTES;
                mbar_arrive_expect_tx(bar_full + 8 * s, C::STAGE_BYTES);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_4d(sK + c * (TK * 128), mk, bar_full + 8 * s, c * 64, c_row, kvh, b, policy);
                    tma_load_4d(sV + c * (TK * 128), mv, bar_full + 8 * s, c * 64, c_row, kvh, b, policy);
                }
                issued = t + 1;
            }
            // never leave the CTA with bulk copies still landing in its shared memory
            for (int t = max(0, issued - C::STAGES); t < issued; ++t)
                mbar_wait_bounded(bar_full + 8 * (t % C::STAGES), (t / C::STAGES) & 1, p.wait_limit);
        }
        return;
    }

    // =========================================================== compute warps
    constexpr int NCT = C::NW * 32;
    const int g = lane >> 2, t4 = lane & 3;
    const int lm = lane >> 3, lr = lane & 7;  // ldmatrix: which 8x8 matrix this lane addresses, and its row

    // Prologue: every load first (n_seen, the first tile's tags, Q^T fragments,
    // the appended rows), then the stores, so their latencies overlap each
    // other and the first tile's copy.  Inside the split, key indices are
    // 32-bit offsets from k_begin (a split never exceeds the ring plus the
    // memory store, both bounded by INT32_MAX / 2).
    const int32_t klen = (int32_t)(k_end - k_begin);                                   // keys of the split
    const int32_t ring_rel = (int32_t)max((int64_t)0, min(k_end, (int64_t)p.n_slots) - k_begin);  // tagged keys
    const int32_t mem_rel = k_end > mem_lo ? (int32_t)(mem_lo - k_begin) : INT32_MAX;  // first memory key
    const int32_t *tags = p.pos_tag + (int64_t)b * p.n_slots + k_begin;
    int64_t seen = p.n_seen[b];
    // this thread's keys in a tile: key g and key g + 8 of its warp's 16
    const int32_t kw_lane = C::KW * warp + g;
    auto load_tags = [&](int t, int32_t &t0, int32_t &t1) {
        const int32_t ka = t * TK + kw_lane;
        t0 = ka < ring_rel ? __ldg(tags + ka) : -1;
        t1 = ka + 8 < ring_rel ? __ldg(tags + ka + 8) : -1;
    };
    int32_t tg0 = -1, tg1 = -1;
    if (n_tiles > 0) load_tags(0, tg0, tg1);
    // Q^T as the B operand of every S^T product: k-step kk holds
    // Q[row g][kk*16 + 2*t4 + {0,1}] and Q[row g][kk*16 + 8 + 2*t4 + {0,1}]
    uint32_t qf[C::KSTEPS][2];
    if constexpr (FMA) {
        // Q as fp32 in shared memory [8 rows][D] (zero rows past the real ones),
        // read by every lane of a row group at once
        float *q32 = reinterpret_cast<float *>(gbase + C::Q32_OFF);
        for (int i = threadIdx.x; i < kDraftRows * D / 8; i += NCT) {
            const int r = i / (D / 8), v = i - r * (D / 8);
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (r < p.rows)
                x = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.q) +
                                                           ((int64_t)b * p.n_q_heads + kvh * p.group + r) * D) + v);
            float4 *dst = reinterpret_cast<float4 *>(q32 + r * D + v * 8);
            dst[0] = make_float4(__uint_as_float(x.x << 16), __uint_as_float(x.x & 0xffff0000u),
                                 __uint_as_float(x.y << 16), __uint_as_float(x.y & 0xffff0000u));
            dst[1] = make_float4(__uint_as_float(x.z << 16), __uint_as_float(x.z & 0xffff0000u),
                                 __uint_as_float(x.w << 16), __uint_as_float(x.w & 0xffff0000u));
        }
    } else {
        const bool real = g < p.rows;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            static_cast<const __nv_bfloat16 *>(p.q) + ((int64_t)b * p.n_q_heads + kvh * p.group + (real ? g : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            qf[kk][0] = real ? __ldg(qrow + kk * 8 + t4) : 0u;
            qf[kk][1] = real ? __ldg(qrow + kk * 8 + 4 + t4) : 0u;
        }
    }
    // STEP: each compute warp holds the appended K and V rows (the warp that
    // owns slot(p) writes them into its staged tile)
    constexpr int NV = 2 * D / 8;                  // 16-byte vectors of the K row and the V row
    constexpr int VPL = (NV + 31) / 32;            // per lane
    uint4 new_v[VPL];
    if (STEP) {
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int i = lane + 32 * j;
            const uint4 *src = static_cast<const uint4 *>(i < D / 8 ? p.k_new : p.v_new);
            new_v[j] = i < NV ? __ldg(src + ((int64_t)b * p.n_kv_heads + kvh) * (D / 8) + i % (D / 8))
                              : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (seen < 0 || (STEP && seen >= INT32_MAX)) {  // STEP: p must fit an int32 tag
        if (threadIdx.x == 0) draft_report(p.err, WM_DEVERR_BAD_LENGTH);
        seen = STEP ? -1 : 0;  // STEP: nothing is appended, every key is masked
    }
    const int64_t qpos = STEP ? seen : seen - 1;  // the query's position
    const int64_t new_slot =
        (STEP && seen >= 0) ? (seen < p.sink ? seen : p.sink + (seen - p.sink) % p.window) : -1;
    const bool has_new = STEP && new_slot >= k_begin && new_slot < k_end;
    // The key set in 32-bit terms.  Tags are int32 (a ring never holds a
    // position >= INT32_MAX), so clamping the query position and the window's
    // lower edge into int32 keeps every comparison exact.
    const int32_t qp = (int32_t)min(qpos, (int64_t)INT32_MAX);
    const int32_t lo = (int32_t)max(min(qpos - p.window, (int64_t)INT32_MAX), (int64_t)INT32_MIN);
    const int32_t sink = p.sink;
    const int32_t new_rel = has_new ? (int32_t)(new_slot - k_begin) : -1;
    auto tag_ok = [&](int32_t t) { return t >= 0 && t <= qp && (t < sink || t > lo); };

    // running state: mma.sync path (rows 2*t4, 2*t4 + 1 of the S^T fragment)
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
    float l_run[2] = {0.f, 0.f};  // this thread's keys only
    float oacc[C::KSTEPS][4];
    // CUDA-core path: rows 4*rg .. 4*rg + 3 of this lane's key; O over 8 rows x DL columns
    float fm_run[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
    float fl_run[4] = {0.f, 0.f, 0.f, 0.f};
    float fo[kDraftRows][C::DL];
    const float kRaise = 8.f;  // log2 units: raise the running max only past 2^8

    if constexpr (!FMA) {
        // ldmatrix row addresses (this lane's row of its 8x8 matrix) within a
        // stage, for k-steps / head-dim blocks 0..3 of each 64-column chunk; the
        // chunk adds a constant TK * 128 bytes.  Rows are 16w + (0 or 8) + lr, so
        // a row's 128-byte swizzle phase is lr.
        uint32_t koff[4], voff[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int krow = C::KW * warp + (lm & 1) * 8 + lr;  // S^T: A = K[16 keys x 16 dims]
            koff[c] = krow * 128 + ((((2 * c + (lm >> 1)) & 7) ^ lr) << 4);
            const int vrow = C::KW * warp + (lm >> 1) * 8 + lr;  // O^T: A = V^T[16 dims x 16 keys] (transposed load)
            voff[c] = vrow * 128 + ((((2 * c + (lm & 1)) & 7) ^ lr) << 4);
        }

        float m_use[2] = {0.f, 0.f};                      // m_run, or 0 while it is -inf
#pragma unroll
        for (int i = 0; i < C::KSTEPS; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[i][e] = 0.f;

        for (int t = 0; t < n_tiles; ++t) {
            const int s = t % C::STAGES;
            int32_t nt0 = -1, nt1 = -1;
            if (t + 1 < n_tiles) load_tags(t + 1, nt0, nt1);
            bool live = !*abort_flag;
            if (live && !mbar_wait_bounded(bar_full + 8 * s, (t / C::STAGES) & 1, p.wait_limit)) {
                draft_report(p.err, WM_DEVERR_TIMEOUT);
                *abort_flag = 1;
                live = false;
            }
            const int32_t kt = t * TK;  // the tile's first key, relative to the split
            const uint32_t sK = sbase + s * C::STAGE_BYTES;
            const uint32_t sV = sK + C::TILE_BYTES;
            bool wrote_smem = false;
            if (live) {
                // ---- STEP: the appended rows replace the ring's stale row in the staged tile
                if (STEP && new_rel >= kt + C::KW * warp && new_rel < kt + C::KW * warp + C::KW) {
                    const int row = new_rel - kt;
#pragma unroll
                    for (int j = 0; j < VPL; ++j) {
                        const int i = lane + 32 * j;
                        if (i < NV) {
                            const int v = i % (D / 8);
                            st_shared_v4((i < D / 8 ? sK : sV) + (v >> 3) * (TK * 128) + swz128(row, v & 7), new_v[j]);
                        }
                    }
                    __syncwarp();
                    wrote_smem = true;
                }

                // ---- S^T = K Q^T for this warp's 16 keys (two accumulator chains)
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    uint32_t a[4];
                    ldsm_x4(sK + koff[kk & 3] + (kk >> 2) * (TK * 128), a[0], a[1], a[2], a[3]);
                    mma_bf16((kk & 1) ? sb : sa, a, qf[kk][0], qf[kk][1]);
                }
                // masks of this thread's two keys: memory tiles hold only keys; ring
                // keys are judged by their tags (the appended slot holds qpos)
                const int32_t k0 = kt + kw_lane, k1 = k0 + 8;
                bool ok0, ok1;
                if (kt >= mem_rel) {
                    ok0 = k0 < klen;
                    ok1 = k1 < klen;
                } else {
                    ok0 = k0 < klen && tag_ok(STEP && k0 == new_rel ? qp : tg0);
                    ok1 = k1 < klen && tag_ok(STEP && k1 == new_rel ? qp : tg1);
                }
                // sv[0], sv[1]: key g, rows 2t4 and 2t4+1; sv[2], sv[3]: key g + 8
                float sv[4];
                sv[0] = ok0 ? (sa[0] + sb[0]) * p.scale_log2 : -CUDART_INF_F;
                sv[1] = ok0 ? (sa[1] + sb[1]) * p.scale_log2 : -CUDART_INF_F;
                sv[2] = ok1 ? (sa[2] + sb[2]) * p.scale_log2 : -CUDART_INF_F;
                sv[3] = ok1 ? (sa[3] + sb[3]) * p.scale_log2 : -CUDART_INF_F;
                // ---- tile max per row over the warp's 16 keys
                float tmax[2] = {fmaxf(sv[0], sv[2]), fmaxf(sv[1], sv[3])};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 4));
                    tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 8));
                    tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 16));
                }
                // ---- raise the running max (rarely: only past 2^8), rescaling O^T and l
                const bool raise0 = tmax[0] > m_run[0] + kRaise, raise1 = tmax[1] > m_run[1] + kRaise;
                if (__any_sync(0xffffffffu, raise0 || raise1)) {
                    float alpha[2];
                    const bool rz[2] = {raise0, raise1};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float mn = rz[h] ? tmax[h] : m_run[h];
                        alpha[h] = rz[h] ? ex2(m_run[h] - mn) : 1.f;  // 0 when m_run was -inf
                        m_run[h] = mn;
                        m_use[h] = mn == -CUDART_INF_F ? 0.f : mn;
                        l_run[h] *= alpha[h];
                    }
#pragma unroll
                    for (int i = 0; i < C::KSTEPS; ++i) {
                        oacc[i][0] *= alpha[0];
                        oacc[i][1] *= alpha[1];
                        oacc[i][2] *= alpha[0];
                        oacc[i][3] *= alpha[1];
                    }
                }
                const float p0 = ex2(sv[0] - m_use[0]), p1 = ex2(sv[1] - m_use[1]);
                const float p2 = ex2(sv[2] - m_use[0]), p3 = ex2(sv[3] - m_use[1]);
                l_run[0] += p0 + p2;
                l_run[1] += p1 + p3;
                // ---- P^T as the B operand: hi and lo bf16 parts, transposed in registers
                const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
                const __nv_bfloat162 hb01 = *reinterpret_cast<const __nv_bfloat162 *>(&h01);
                const __nv_bfloat162 hb23 = *reinterpret_cast<const __nv_bfloat162 *>(&h23);
                const uint32_t l01 = pack_bf16(p0 - __low2float(hb01), p1 - __high2float(hb01));
                const uint32_t l23 = pack_bf16(p2 - __low2float(hb23), p3 - __high2float(hb23));
                const uint32_t bh0 = movmatrix_t(h01), bh1 = movmatrix_t(h23);
                const uint32_t bl0 = movmatrix_t(l01), bl1 = movmatrix_t(l23);
                // ---- keys masked for every row: their V^T operand elements are
                // zeroed (only on tiles that have such keys)
                const uint32_t okb0 = __ballot_sync(0xffffffffu, ok0), okb1 = __ballot_sync(0xffffffffu, ok1);
                if ((okb0 & okb1) == 0xffffffffu) {
#pragma unroll
                    for (int i = 0; i < C::KSTEPS; ++i) {
                        uint32_t a[4];
                        ldsm_x4_t(sV + voff[i & 3] + (i >> 2) * (TK * 128), a[0], a[1], a[2], a[3]);
                        mma_bf16(oacc[i], a, bh0, bh1);
                        mma_bf16(oacc[i], a, bl0, bl1);
                    }
                } else {
                    // this thread's V^T columns: keys 2t4, 2t4+1 (a0, a1) and 2t4+8, 2t4+9 (a2, a3)
                    const uint32_t mlo = (((okb0 >> (8 * t4)) & 1u) ? 0x0000ffffu : 0u) |
                                         (((okb0 >> (8 * t4 + 4)) & 1u) ? 0xffff0000u : 0u);
                    const uint32_t mhi = (((okb1 >> (8 * t4)) & 1u) ? 0x0000ffffu : 0u) |
                                         (((okb1 >> (8 * t4 + 4)) & 1u) ? 0xffff0000u : 0u);
#pragma unroll
                    for (int i = 0; i < C::KSTEPS; ++i) {
                        uint32_t a[4];
                        ldsm_x4_t(sV + voff[i & 3] + (i >> 2) * (TK * 128), a[0], a[1], a[2], a[3]);
                        a[0] &= mlo;
                        a[1] &= mlo;
                        a[2] &= mhi;
                        a[3] &= mhi;
                        mma_bf16(oacc[i], a, bh0, bh1);
                        mma_bf16(oacc[i], a, bl0, bl1);
                    }
                }
            }
            if (wrote_smem) fence_proxy_async_smem();  // the stage is refilled by TMA later
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
            tg0 = nt0;
            tg1 = nt1;
        }
    } else {
        // ================= CUDA-core products (fp32 FMA, warp-shuffle softmax)
        // Lane (kl, rg) = (lane & 15, lane >> 4) computes S for key 16w + kl and
        // rows 4rg .. 4rg + 3; for P.V the lane owns DL head-dim columns of all
        // 8 rows and reads P back from a per-warp shared buffer.
        const int kl = lane & 15, rg = lane >> 4;
        const int krow = C::KW * warp + kl;  // this lane's key row in a tile
        const float4 *q32 = reinterpret_cast<const float4 *>(gbase + C::Q32_OFF);
        float *ps = reinterpret_cast<float *>(gbase + C::PS_OFF) + warp * C::KW * kDraftRows;
        const int32_t *ftags = tags;
        auto load_tag = [&](int t) -> int32_t {
            const int32_t ka = t * TK + krow;
            return ka < ring_rel ? __ldg(ftags + ka) : -1;
        };
        int32_t ftg = n_tiles > 0 ? load_tag(0) : -1;
        float fm_use[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < kDraftRows; ++r)
#pragma unroll
            for (int j = 0; j < C::DL; ++j) fo[r][j] = 0.f;
        named_bar_sync(1, NCT);  // Q staged
        const int dcol = lane * C::DL;  // first head-dim column of this lane in P.V
        for (int t = 0; t < n_tiles; ++t) {
            const int s = t % C::STAGES;
            const int32_t nftg = t + 1 < n_tiles ? load_tag(t + 1) : -1;
            bool live = !*abort_flag;
            if (live && !mbar_wait_bounded(bar_full + 8 * s, (t / C::STAGES) & 1, p.wait_limit)) {
                draft_report(p.err, WM_DEVERR_TIMEOUT);
                *abort_flag = 1;
                live = false;
            }
            const int32_t kt = t * TK;
            const uint32_t sK = sbase + s * C::STAGE_BYTES;
            const uint32_t sV = sK + C::TILE_BYTES;
            const uint8_t *tK = gbase + (sK - sbase);
            const uint8_t *tV = tK + C::TILE_BYTES;
            bool wrote_smem = false;
            if (live) {
                if (STEP && new_rel >= kt + C::KW * warp && new_rel < kt + C::KW * warp + C::KW) {
                    const int row = new_rel - kt;
#pragma unroll
                    for (int j = 0; j < VPL; ++j) {
                        const int i = lane + 32 * j;
                        if (i < NV) {
                            const int v = i % (D / 8);
                            st_shared_v4((i < D / 8 ? sK : sV) + (v >> 3) * (TK * 128) + swz128(row, v & 7),
                                         new_v[j]);
                        }
                    }
                    __syncwarp();
                    wrote_smem = true;
                }
                // ---- S for this lane's key and four rows: dot products over D
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int c = 0; c < D / 8; ++c) {
                    const uint4 kv = *reinterpret_cast<const uint4 *>(tK + (c >> 3) * (TK * 128) + swz128(krow, c & 7));
                    const float k0 = __uint_as_float(kv.x << 16), k1 = __uint_as_float(kv.x & 0xffff0000u);
                    const float k2 = __uint_as_float(kv.y << 16), k3 = __uint_as_float(kv.y & 0xffff0000u);
                    const float k4 = __uint_as_float(kv.z << 16), k5 = __uint_as_float(kv.z & 0xffff0000u);
                    const float k6 = __uint_as_float(kv.w << 16), k7 = __uint_as_float(kv.w & 0xffff0000u);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 qa = q32[(4 * rg + i) * (D / 4) + 2 * c];
                        const float4 qb = q32[(4 * rg + i) * (D / 4) + 2 * c + 1];
                        float a = acc[i];
                        a = fmaf(qa.x, k0, a);
                        a = fmaf(qa.y, k1, a);
                        a = fmaf(qa.z, k2, a);
                        a = fmaf(qa.w, k3, a);
                        a = fmaf(qb.x, k4, a);
                        a = fmaf(qb.y, k5, a);
                        a = fmaf(qb.z, k6, a);
                        a = fmaf(qb.w, k7, a);
                        acc[i] = a;
                    }
                }
                const int32_t kk = kt + krow;
                const bool ok = kt >= mem_rel ? kk < klen : (kk < klen && tag_ok(STEP && kk == new_rel ? qp : ftg));
                float sv[4], tmax[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    sv[i] = ok ? acc[i] * p.scale_log2 : -CUDART_INF_F;
                    float m = sv[i];  // max over the warp's 16 keys (the 16 lanes of this row group)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    tmax[i] = m;
                }
                bool rz[4], any_rz = false;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    rz[i] = tmax[i] > fm_run[i] + kRaise;
                    any_rz |= rz[i];
                }
                if (__any_sync(0xffffffffu, any_rz)) {
                    float al[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float mn = rz[i] ? tmax[i] : fm_run[i];
                        al[i] = rz[i] ? ex2(fm_run[i] - mn) : 1.f;
                        fm_run[i] = mn;
                        fm_use[i] = mn == -CUDART_INF_F ? 0.f : mn;
                        fl_run[i] *= al[i];
                    }
                    // P.V rows: this group's four and, by exchange, the other group's
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float other = __shfl_xor_sync(0xffffffffu, al[i], 16);
                        const float a_lo = rg ? other : al[i], a_hi = rg ? al[i] : other;
#pragma unroll
                        for (int j = 0; j < C::DL; ++j) {
                            fo[i][j] *= a_lo;
                            fo[4 + i][j] *= a_hi;
                        }
                    }
                }
                float pr[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    pr[i] = ex2(sv[i] - fm_use[i]);
                    fl_run[i] += pr[i];
                }
                *reinterpret_cast<float4 *>(ps + kl * kDraftRows + 4 * rg) = make_float4(pr[0], pr[1], pr[2], pr[3]);
                const uint32_t vm = __ballot_sync(0xffffffffu, ok) & 0xffffu;  // keys of the warp with weight
                __syncwarp();
                // ---- O += P V over this lane's DL columns of the 8 rows
#pragma unroll 2
                for (int k = 0; k < C::KW; ++k) {
                    if (!((vm >> k) & 1u)) continue;  // masked for every row: its V bytes are never read
                    const int vrow = C::KW * warp + k;
                    const uint8_t *vp = tV + (dcol >> 6) * (TK * 128) + swz128(vrow, (dcol & 63) >> 3) + (dcol & 7) * 2;
                    float vf[C::DL];
                    if constexpr (C::DL == 8) {
                        const uint4 x = *reinterpret_cast<const uint4 *>(vp);
                        vf[0] = __uint_as_float(x.x << 16); vf[1] = __uint_as_float(x.x & 0xffff0000u);
                        vf[2] = __uint_as_float(x.y << 16); vf[3] = __uint_as_float(x.y & 0xffff0000u);
                        vf[4] = __uint_as_float(x.z << 16); vf[5] = __uint_as_float(x.z & 0xffff0000u);
                        vf[6] = __uint_as_float(x.w << 16); vf[7] = __uint_as_float(x.w & 0xffff0000u);
                    } else if constexpr (C::DL == 4) {
                        const uint2 x = *reinterpret_cast<const uint2 *>(vp);
                        vf[0] = __uint_as_float(x.x << 16); vf[1] = __uint_as_float(x.x & 0xffff0000u);
                        vf[2] = __uint_as_float(x.y << 16); vf[3] = __uint_as_float(x.y & 0xffff0000u);
                    } else {
                        const uint32_t x = *reinterpret_cast<const uint32_t *>(vp);
                        vf[0] = __uint_as_float(x << 16); vf[1] = __uint_as_float(x & 0xffff0000u);
                    }
                    const float4 pa = *reinterpret_cast<const float4 *>(ps + k * kDraftRows);
                    const float4 pb = *reinterpret_cast<const float4 *>(ps + k * kDraftRows + 4);
                    const float pk[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
                    for (int r = 0; r < kDraftRows; ++r)
#pragma unroll
                        for (int j = 0; j < C::DL; ++j) fo[r][j] = fmaf(pk[r], vf[j], fo[r][j]);
                }
            }
            if (wrote_smem) fence_proxy_async_smem();  // the stage is refilled by TMA later
            __syncwarp();  // every lane has read this tile's P before the next tile writes it
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
            ftg = nftg;
        }
    }

    // ---- STEP: store the appended entry into the ring (the owning warp; every
    // tile that staged its slot has been consumed)
    if (has_new) {
        const int64_t off = k_begin + (new_slot - k_begin) / TK * TK;  // first key of the slot's tile
        const int owner = (int)((new_slot - off) / C::KW);
        if (warp == owner) {
#pragma unroll
            for (int j = 0; j < VPL; ++j) {
                const int i = lane + 32 * j;
                if (i < NV) {
                    uint4 *dst = static_cast<uint4 *>(i < D / 8 ? p.ring_k : p.ring_v);
                    dst[(((int64_t)b * p.n_kv_heads + kvh) * p.n_slots + new_slot) * (D / 8) + i % (D / 8)] = new_v[j];
                }
            }
            if (kvh == 0 && lane == 0) p.tag_w[(int64_t)b * p.n_slots + new_slot] = (int32_t)qpos;
        }
    }

    // ---- combine the four warps: row maxima and sums, then O in a fixed order
    if constexpr (!FMA) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 4);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 8);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 16);
        }
        if (g == 0) {
            red_m[warp * kDraftRows + 2 * t4] = m_run[0];
            red_m[warp * kDraftRows + 2 * t4 + 1] = m_run[1];
            red_l[warp * kDraftRows + 2 * t4] = l_run[0];
            red_l[warp * kDraftRows + 2 * t4 + 1] = l_run[1];
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            fl_run[i] += __shfl_xor_sync(0xffffffffu, fl_run[i], 1);
            fl_run[i] += __shfl_xor_sync(0xffffffffu, fl_run[i], 2);
            fl_run[i] += __shfl_xor_sync(0xffffffffu, fl_run[i], 4);
            fl_run[i] += __shfl_xor_sync(0xffffffffu, fl_run[i], 8);
        }
        if ((lane & 15) == 0) {
            const int r0 = 4 * (lane >> 4);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                red_m[warp * kDraftRows + r0 + i] = fm_run[i];
                red_l[warp * kDraftRows + r0 + i] = fl_run[i];
            }
        }
    }
    // After an aborted pipeline, copies may still land in the staging area:
    // this CTA's result is then not written (the decision is the same in
    // every warp).
    const bool aborted = named_bar_sync_or(1, NCT, *abort_flag != 0);
    float *obuf = reinterpret_cast<float *>(gbase);  // the staging area: every copy has landed and been read
    if (!aborted) {
        float *ob = obuf + warp * kDraftRows * C::OB_STRIDE;
        if constexpr (!FMA) {
            float f[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = 2 * t4 + h;
                float mx = red_m[r];
#pragma unroll
                for (int w = 1; w < C::NW; ++w) mx = fmaxf(mx, red_m[w * kDraftRows + r]);
                f[h] = m_run[h] == -CUDART_INF_F ? 0.f : ex2(m_run[h] - mx);
            }
#pragma unroll
            for (int i = 0; i < C::KSTEPS; ++i) {
                const int d = i * 16 + g;
                ob[(2 * t4) * C::OB_STRIDE + d] = oacc[i][0] * f[0];
                ob[(2 * t4 + 1) * C::OB_STRIDE + d] = oacc[i][1] * f[1];
                ob[(2 * t4) * C::OB_STRIDE + d + 8] = oacc[i][2] * f[0];
                ob[(2 * t4 + 1) * C::OB_STRIDE + d + 8] = oacc[i][3] * f[1];
            }
        } else {
#pragma unroll
            for (int r = 0; r < kDraftRows; ++r) {
                const float mw = red_m[warp * kDraftRows + r];
                float mx = red_m[r];
#pragma unroll
                for (int w = 1; w < C::NW; ++w) mx = fmaxf(mx, red_m[w * kDraftRows + r]);
                const float f = mw == -CUDART_INF_F ? 0.f : ex2(mw - mx);
#pragma unroll
                for (int j = 0; j < C::DL; ++j) ob[r * C::OB_STRIDE + lane * C::DL + j] = fo[r][j] * f;
            }
        }
    }
    named_bar_sync(1, NCT);

    // ---- this split's result: 16 threads per row, float4 columns (c, c + 64, ...);
    // the final output when unsplit, else fp32 partials for the merge kernel
    if (aborted) return;
    const float kLn2 = 0.693147180559945309f;
    const int tid = threadIdx.x;
    const int r = tid >> 4;  // row 0..7
    const int cq = (tid & 15) * 4;
    if (r >= p.rows) return;
    float mx = red_m[r];
#pragma unroll
    for (int w = 1; w < C::NW; ++w) mx = fmaxf(mx, red_m[w * kDraftRows + r]);
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) {
        const float mw = red_m[w * kDraftRows + r];
        lt += (mw == -CUDART_INF_F ? 0.f : ex2(mw - mx)) * red_l[w * kDraftRows + r];
    }
    const bool has = lt > 0.f;
    const float inv = has ? 1.f / lt : 0.f;
    const float lse = has ? (mx + lg2(lt)) * kLn2 : -CUDART_INF_F;
    const int64_t orow = (int64_t)b * p.n_q_heads + kvh * p.group + r;
#pragma unroll
    for (int j = 0; j < D / 64; ++j) {
        const int col = j * 64 + cq;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < C::NW; ++w) {  // fixed order: the same bits every run
            const float4 u = *reinterpret_cast<const float4 *>(obuf + (w * kDraftRows + r) * C::OB_STRIDE + col);
            o.x += u.x;
            o.y += u.y;
            o.z += u.z;
            o.w += u.w;
        }
        o.x *= inv;
        o.y *= inv;
        o.z *= inv;
        o.w *= inv;
        if (p.o_part) {
            *reinterpret_cast<float4 *>(p.o_part + (orow * p.n_split + split) * D + col) = o;
        } else {
            uint2 pk;
            pk.x = pack_bf16(o.x, o.y);
            pk.y = pack_bf16(o.z, o.w);
            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.out) + orow * D + col) = pk;
        }
    }
    if ((tid & 15) == 0) {
        if (p.o_part)
            p.lse_part[orow * p.n_split + split] = lse;
        else if (p.lse)
            p.lse[orow] = lse;
    }
}

template <int D, bool STEP, bool FMA>
cudaError_t launch_draft_kernel(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                                const CUtensorMap &mv, const AttnParams &p, cudaStream_t stream) {
    constexpr int smem = DraftCfg<D, FMA>::TOTAL;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(draft_kernel<D, STEP, FMA>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const dim3 grid(p.n_split, p.batch * p.n_kv_heads);
    return launch_pdl(draft_kernel<D, STEP, FMA>, grid, dim3(kThreads), smem, stream, k, v, mk, mv, p);
}

template <int D, bool STEP, bool FMA>
int draft_blocks_per_sm_t() {
    constexpr int smem = DraftCfg<D, FMA>::TOTAL;
    if (cudaFuncSetAttribute(draft_kernel<D, STEP, FMA>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, draft_kernel<D, STEP, FMA>, kThreads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace wm

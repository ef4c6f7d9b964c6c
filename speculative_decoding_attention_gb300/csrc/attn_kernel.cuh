// attn_kernel.cuh -- split-KV decode attention for one KV head group.
//
// One CTA handles one (sequence, KV head) pair and one contiguous range of key
// positions (a split).  Its rows are every query that reads this KV head: for
// verification the n_q proposed positions x G grouped heads, for the draft the
// G grouped heads of the one query position.  So each KV byte is read from
// HBM once per group.
//
// Warp roles (5 warps):
//   warp 4 (producer)  : one lane streams 64-key K and V tiles into a ring of
//                        shared-memory stages with TMA (128-byte swizzle),
//                        signalling a "full" mbarrier per stage.
//   warps 0-3 (compute): S = Q K^T on tensor cores (each warp 16 keys of the
//                        tile, all rows), online softmax in base 2 with the
//                        running row max exchanged through shared memory,
//                        P to shared memory as two bf16 parts (hi = bf16(p),
//                        lo = bf16(p - hi)), then O += P_hi V + P_lo V (each
//                        warp a quarter of the head dim), and an "empty"
//                        arrival to hand the stage back.  The two-part P keeps
//                        the weights accurate to ~2^-17 relative: with only a
//                        few keys, or a peaked softmax, a single bf16 rounding
//                        of P (2^-9) would show up in the output.
// The split's normalised output and its log-sum-exp go either straight to the
// bf16 output (one split) or to fp32 partials that a merge kernel combines.
//
// Fused draft step (STEP = true): ring append + draft attention in one
// launch.  Every CTA reads p = n_seen[b] (the position being appended) and
// treats ring slot(p) as holding p: the CTA whose key range contains that slot
// copies the new K/V row over the stale one in its staged tile (its TMA read
// the ring before the append) and stores the row and its tag into the ring.
// The split partials always go to the merge kernel, which also commits
// n_seen[b] = p + 1 -- after this grid has finished, so no CTA can see the
// new count early.  Same splits and merge as the unfused draft, so the outputs
// are bit-identical to ring append + draft attention.
//
// Memory slots (memory-augmented draft): keys at or beyond mem_base are the
// materialized slots 0..count[b]-1 of a second store, read through the second
// pair of tensor maps, and every row sees all of them.
//
// Masks: verification is causal (query i sees positions <= seq_len - n_q + i);
// the draft sees a ring slot iff its tag t satisfies 0 <= t <= p and
// (t < sink or t > p - window); the split's tags are staged in shared memory
// with Q when they fit.  Keys masked for every row get their V row zeroed in
// shared memory so that stale or uninitialised cache bytes (even NaN
// patterns) cannot reach the output through 0 * NaN.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"
#include "wm_internal.h"
#include "../../include/wm_api.h"

namespace wm {

template <int D>
struct AttnCfg {
    static constexpr int TK = kKeyTile;                          // keys per stage
    static constexpr int NCH = D / 64;                           // 128-byte chunks per row
    static constexpr int TILE_BYTES = TK * D * 2;                // K (or V) tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int STAGES = staging_bytes(D) / STAGE_BYTES;  // 4 / 4 / 2
    static constexpr int NW = kConsumerWarps;
    static constexpr int KPW = TK / NW;                          // keys per warp in Q K^T
    static constexpr int DW = D / NW;                            // head-dim columns per warp in P V
    static constexpr int NTB = DW / 8;                           // n-tiles per warp in P V
    static_assert(KPW == 16, "Q K^T assumes 16 keys per warp");
    static_assert(NTB % 2 == 0, "P V loads V in pairs of n-tiles");
    static_assert(STAGES >= 2, "need at least double buffering");
};

// Ring tags a draft CTA stages in shared memory with Q (its whole split, when
// it has at most this many keys; longer splits read them from global memory a
// tile ahead).
constexpr int kTagCache = 1024;

template <int D, int MT>
struct AttnSmem {
    static constexpr int ROWS = MT * 16;
    static constexpr int Q_OFF = AttnCfg<D>::STAGES * AttnCfg<D>::STAGE_BYTES;
    static constexpr int P_OFF = Q_OFF + ROWS * D * 2;
    static constexpr int P_BYTES = ROWS * kKeyTile * 2;            // one P buffer (hi or lo part)
    static constexpr int RED_OFF = P_OFF + 4 * P_BYTES;            // red_max[2][NW][ROWS], red_l[NW][ROWS]
    static constexpr int RED_BYTES = 3 * kConsumerWarps * ROWS * 4;
    static constexpr int BAR_OFF = RED_OFF + RED_BYTES;            // full[STAGES], empty[STAGES]
    static constexpr int FLAG_OFF = BAR_OFF + 2 * AttnCfg<D>::STAGES * 8;
    static constexpr int NEW_OFF = FLAG_OFF + 16;                  // fused step: appended K and V rows
    static constexpr int TAG_OFF = NEW_OFF + 2 * D * 2;            // ring tags of the split (draft)
    static constexpr int TOTAL = TAG_OFF + kTagCache * 4 + 1024;   // + slack to 1024-align the base
    static_assert(Q_OFF % 1024 == 0 && P_OFF % 1024 == 0 && P_BYTES % 1024 == 0,
                  "swizzled regions need 1024-byte alignment");
    static_assert(NEW_OFF % 16 == 0, "16-byte vectors");
    static_assert(TOTAL <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void report_error(int32_t *err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

template <int D, int MT, bool STEP>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                const __grid_constant__ CUtensorMap tmk2, const __grid_constant__ CUtensorMap tmv2,
                const AttnParams p) {
    using C = AttnCfg<D>;
    using L = AttnSmem<D, MT>;
    constexpr int ROWS = L::ROWS;
    constexpr int TK = C::TK;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw);
    const uint32_t sQ = sbase + L::Q_OFF;
    const uint32_t sP = sbase + L::P_OFF;
    float *red_max = reinterpret_cast<float *>(gbase + L::RED_OFF);
    float *red_l = red_max + 2 * C::NW * ROWS;
    const uint32_t bar_full = sbase + L::BAR_OFF;
    const uint32_t bar_empty = bar_full + 8 * C::STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + L::FLAG_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int unit = blockIdx.y;
    const int b = unit / p.n_kv_heads;
    const int kvh = unit - b * p.n_kv_heads;
    const int split = blockIdx.x;

    pdl_wait();  // every global read below may depend on the previous kernel
    pdl_launch_dependents();

    // ---- keys of this split, and the position of query 0.  The ring's key
    // range does not depend on n_seen: only the compute warps read it (below),
    // so the producer's first copies are not held up by that load.
    int64_t n_keys, qpos0 = -1;
    if (p.source == KEYS_RING) {
        n_keys = p.n_slots;
        if (p.mem_count) {  // memory slots follow the ring's (tile-rounded) slots
            int64_t mc = p.mem_count[b];
            if (mc < 0 || mc > p.mem_cap) {
                if (threadIdx.x == 0) report_error(p.err, WM_DEVERR_BAD_LENGTH);
                mc = mc < 0 ? 0 : p.mem_cap;
            }
            n_keys = p.mem_base + mc;
        }
    } else {
        int64_t len = p.seq_lens[b];
        if (len < 0 || len > p.capacity) {
            if (threadIdx.x == 0) report_error(p.err, WM_DEVERR_BAD_LENGTH);
            len = len < 0 ? 0 : p.capacity;
        }
        n_keys = len;
        qpos0 = len - p.n_q;
    }
    const int64_t k_begin = (int64_t)split * p.keys_per_split;
    const int64_t k_end = min(k_begin + (int64_t)p.keys_per_split, n_keys);
    const int n_tiles = k_end > k_begin ? (int)((k_end - k_begin + TK - 1) / TK) : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, C::NW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // =========================================================== producer warp
    // Keys at or beyond mem_lo are memory slots (always visible to the query).
    const int64_t mem_lo = p.mem_count ? p.mem_base : INT64_MAX;
    if (warp == C::NW) {
        if (lane == 0 && n_tiles > 0) {
            const bool mem_tiles = k_end > mem_lo;
            if (k_begin < mem_lo) {
                prefetch_tensormap(&tmk);
                prefetch_tensormap(&tmv);
            }
            if (mem_tiles) {
                prefetch_tensormap(&tmk2);
                prefetch_tensormap(&tmv2);
            }
            // The cache is streamed once per call; the ring is read again by the
            // next draft step, so its lines keep normal priority.
            const uint64_t policy =
                p.source == KEYS_RING ? l2_policy_evict_normal() : l2_policy_evict_first();
            int issued = 0;
            // Paged: the tiles of a split step through its pages in order (a tile
            // never crosses a page), so the page and row advance without a
            // division, and each tile's block-table entry is loaded one tile ahead.
            const bool paged = p.source == KEYS_PAGED;
            int64_t pg = paged ? k_begin / p.page_size : 0;
            int pg_row = paged ? (int)(k_begin - pg * p.page_size) : 0;
            int32_t pg_entry = paged ? p.block_table[(int64_t)b * p.max_pages + pg] : 0;
            for (int t = 0; t < n_tiles; ++t) {
                if (t == p.stall_tile) break;  // tests of the timeout path only
                const int s = t % C::STAGES;
                if (t >= C::STAGES &&
                    !mbar_wait_bounded(bar_empty + 8 * s, ((t / C::STAGES) & 1) ^ 1, p.wait_limit)) {
                    report_error(p.err, WM_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const int64_t key0 = k_begin + (int64_t)t * TK;
                int c_row, c_outer;
                if (paged) {
                    int32_t page = pg_entry;
                    c_row = pg_row;
                    pg_row += TK;
                    if (pg_row >= p.page_size) {  // the next tile starts the next page
                        pg_row = 0;
                        ++pg;
                        if (t + 1 < n_tiles) pg_entry = p.block_table[(int64_t)b * p.max_pages + pg];
                    }
                    if (page < 0 || page >= p.n_pages) {
                        report_error(p.err, WM_DEVERR_BAD_PAGE);
                        page = 0;
                    }
                    c_outer = page;
                } else {
                    c_row = (int)(key0 >= mem_lo ? key0 - mem_lo : key0);  // a tile is all ring or all memory
                    c_outer = b;
                }
                const CUtensorMap *mk = key0 >= mem_lo ? &tmk2 : &tmk;
                const CUtensorMap *mv = key0 >= mem_lo ? &tmv2 : &tmv;
                const uint32_t sK = sbase + s * C::STAGE_BYTES;
                const uint32_t sV = sK + C::TILE_BYTES;
                mbar_arrive_expect_tx(bar_full + 8 * s, C::STAGE_BYTES);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_4d(sK + c * (TK * 128), mk, bar_full + 8 * s, c * 64, c_row, kvh, c_outer, policy);
                    tma_load_4d(sV + c * (TK * 128), mv, bar_full + 8 * s, c * 64, c_row, kvh, c_outer, policy);
                }
                issued = t + 1;
            }
            // Never leave the CTA with bulk copies still landing in its shared memory.
            for (int t = max(0, issued - C::STAGES); t < issued; ++t)
                mbar_wait_bounded(bar_full + 8 * (t % C::STAGES), (t / C::STAGES) & 1, p.wait_limit);
        }
        return;
    }

    // =========================================================== compute warps
    constexpr int NCT = C::NW * 32;  // compute threads
    // Prologue: issue every load first (n_seen, the split's ring tags, Q), then
    // store, so that their latencies overlap each other and the first tile's copy.
    const int32_t *tags = p.source == KEYS_RING ? p.pos_tag + (int64_t)b * p.n_slots : nullptr;
    int32_t *s_tags = reinterpret_cast<int32_t *>(gbase + L::TAG_OFF);
    const int64_t ring_end = min(k_end, (int64_t)p.n_slots);  // memory slots carry no tag
    const bool tags_cached = tags && ring_end - k_begin <= kTagCache;
    constexpr int TPT = kTagCache / NCT;  // staged tags per thread
    int64_t seen = p.source == KEYS_RING ? p.n_seen[b] : 0;
    int32_t tag_v[TPT];
#pragma unroll
    for (int j = 0; j < TPT; ++j) {
        const int64_t i = threadIdx.x + (int64_t)j * NCT;
        tag_v[j] = tags_cached && i < ring_end - k_begin ? __ldg(tags + k_begin + i) : -1;
    }
    constexpr int VPR = D / 8;              // 16-byte vectors per row
    constexpr int QPT = ROWS * VPR / NCT;   // Q vectors per thread
    static_assert(ROWS * VPR % NCT == 0, "Q staging: whole vectors per thread");
    const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
    uint4 q_v[QPT];
#pragma unroll
    for (int j = 0; j < QPT; ++j) {
        const int idx = threadIdx.x + j * NCT;
        const int r = idx / VPR, v = idx - (idx / VPR) * VPR;
        q_v[j] = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.rows) {
            const int i = r / p.group, hh = r - i * p.group;
            const int64_t row = ((int64_t)b * p.n_q + i) * p.n_q_heads + kvh * p.group + hh;
            q_v[j] = __ldg(reinterpret_cast<const uint4 *>(qg + row * D) + v);
        }
    }
    int64_t new_slot = -1;  // STEP: ring slot receiving position qpos0
    if (p.source == KEYS_RING) {
        if (seen < 0 || (STEP && seen >= INT32_MAX)) {  // STEP: p must fit an int32 tag
            if (threadIdx.x == 0) report_error(p.err, WM_DEVERR_BAD_LENGTH);
            seen = STEP ? -1 : 0;  // STEP: nothing is appended, every key is masked
        }
        qpos0 = STEP ? seen : seen - 1;
        if (STEP && seen >= 0) new_slot = seen < p.sink ? seen : p.sink + (seen - p.sink) % p.window;
    }
    // STEP: the CTA whose keys include slot(p) stages the appended K row
    // (threads 0..D/8-1) and V row (D/8..D/4-1) in shared memory with Q.
    constexpr int NVR = D / 8;
    const bool has_new = STEP && new_slot >= k_begin && new_slot < k_end;
    uint4 *s_new = reinterpret_cast<uint4 *>(gbase + L::NEW_OFF);
    if (has_new && threadIdx.x < 2 * NVR) {
        const uint4 *src = static_cast<const uint4 *>(threadIdx.x < NVR ? p.k_new : p.v_new);
        s_new[threadIdx.x] = __ldg(src + ((int64_t)b * p.n_kv_heads + kvh) * NVR + threadIdx.x % NVR);
    }
#pragma unroll
    for (int j = 0; j < QPT; ++j) {
        const int idx = threadIdx.x + j * NCT;
        const int r = idx / VPR, v = idx - (idx / VPR) * VPR;
        st_shared_v4(sQ + (v >> 3) * (ROWS * 128) + swz128(r, v & 7), q_v[j]);
    }
    if (tags_cached) {
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
            const int64_t i = threadIdx.x + (int64_t)j * NCT;
            if (i < ring_end - k_begin) s_tags[i] = tag_v[j];
        }
    }
    named_bar_sync(1, NCT);

    const int g = lane >> 2, t4 = lane & 3;
    const int lm_idx = lane >> 3;  // which 8x8 matrix this lane addresses in ldmatrix.x4
    float m_run[MT][2], l_run[MT][2];
    int64_t row_lim[MT][2];  // largest key position a row may see (-1: padding row)
    float oacc[MT][C::NTB][4];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            m_run[m][h] = -CUDART_INF_F;
            l_run[m][h] = 0.f;
            const int r = m * 16 + g + 8 * h;
            if (r >= p.rows)
                row_lim[m][h] = -1;
            else if (p.source == KEYS_RING)
                row_lim[m][h] = qpos0 < 0 ? -1 : INT64_MAX;  // ring masks per key (tags)
            else
                row_lim[m][h] = qpos0 + r / p.group;
        }
#pragma unroll
        for (int n = 0; n < C::NTB; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[m][n][e] = 0.f;
    }
    // Ring slot tags this thread needs for one tile: the four keys of its S
    // fragment and (lanes < 16) the key it checks for V-row zeroing.  Read from
    // the staged copy when the split fits it; otherwise fetched from global
    // memory one tile ahead so that their latency hides behind the tile.
    const bool tags_global = tags && !tags_cached;
    auto fetch_tags = [&](int64_t key0, int32_t(&tg)[2][2], int32_t &tg1) {
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int64_t kabs = key0 + warp * C::KPW + n * 8 + 2 * t4 + e;
                tg[n][e] = kabs < ring_end ? __ldg(tags + kabs) : -1;
            }
        const int64_t kl = key0 + warp * C::KPW + lane;
        tg1 = (lane < C::KPW && kl < ring_end) ? __ldg(tags + kl) : -1;
    };
    auto tag_of_key = [&](int64_t kabs, int32_t prefetched) -> int32_t {
        if (!tags_cached) return prefetched;
        return kabs < ring_end ? s_tags[kabs - k_begin] : -1;
    };
    auto tag_ok = [&](int64_t tg) {
        return tg >= 0 && tg <= qpos0 && (tg < p.sink || tg > qpos0 - p.window);
    };
    // The tag a key is judged by: STEP's appended slot holds qpos0 already.
    auto tag_of = [&](int64_t kabs, int32_t tg) -> int64_t {
        return STEP && kabs == new_slot ? qpos0 : (int64_t)tg;
    };
    int32_t tg_cur[2][2] = {{-1, -1}, {-1, -1}}, tg1_cur = -1, tg_nxt[2][2], tg1_nxt;
    if (tags_global && n_tiles > 0) fetch_tags(k_begin, tg_cur, tg1_cur);

    for (int t = 0; t < n_tiles; ++t) {
        if (tags_global && t + 1 < n_tiles) fetch_tags(k_begin + (int64_t)(t + 1) * TK, tg_nxt, tg1_nxt);
        const int s = t % C::STAGES;
        const int buf = t & 1;
        if (!*abort_flag && !mbar_wait_bounded(bar_full + 8 * s, (t / C::STAGES) & 1, p.wait_limit)) {
            report_error(p.err, WM_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
        const bool live = !*abort_flag;
        const int64_t key0 = k_begin + (int64_t)t * TK;
        const uint32_t sK = sbase + s * C::STAGE_BYTES;
        const uint32_t sV = sK + C::TILE_BYTES;

        // ---- STEP: the appended K/V row replaces the ring's stale row
        if (has_new && new_slot >= key0 && new_slot < key0 + TK) {
            if (live && threadIdx.x < 2 * NVR) {
                const int row = (int)(new_slot - key0), v = threadIdx.x % NVR;
                st_shared_v4((threadIdx.x < NVR ? sK : sV) + (v >> 3) * (TK * 128) + swz128(row, v & 7),
                             s_new[threadIdx.x]);
                fence_proxy_async_smem();  // the stage is refilled by TMA later
            }
            named_bar_sync(1, NCT);
        }

        // ---- S = Q K^T for this warp's 16 keys
        float sacc[MT][2][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[m][n][e] = 0.f;
        if (live) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t kb0, kb1, kb2, kb3;
                {
                    const int key = warp * C::KPW + (lm_idx >> 1) * 8 + (lane & 7);
                    const int d = kk * 16 + (lm_idx & 1) * 8;
                    ldsm_x4(sK + (d >> 6) * (TK * 128) + swz128(key, (d & 63) >> 3), kb0, kb1, kb2, kb3);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint32_t a[4];
                    const int row = m * 16 + (lm_idx & 1) * 8 + (lane & 7);
                    const int d = kk * 16 + (lm_idx >> 1) * 8;
                    ldsm_x4(sQ + (d >> 6) * (ROWS * 128) + swz128(row, (d & 63) >> 3), a[0], a[1], a[2],
                            a[3]);
                    mma_bf16(sacc[m][0], a, kb0, kb1);
                    mma_bf16(sacc[m][1], a, kb2, kb3);
                }
            }
        }

        // ---- masks, scaling to base 2, tile row maxima
        const bool tail = key0 + TK > k_end;
        const bool any_row_mask = p.source == KEYS_RING || tail || (key0 + TK - 1 > qpos0);
        bool key_ok[2][2];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int64_t kabs = key0 + warp * C::KPW + n * 8 + 2 * t4 + e;
                bool ok = kabs < k_end;
                if (ok && tags) ok = kabs >= mem_lo || tag_ok(tag_of(kabs, tag_of_key(kabs, tg_cur[n][e])));
                key_ok[n][e] = ok;
            }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float mx = -CUDART_INF_F;
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float v = sacc[m][n][2 * h + e] * p.scale_log2;
                        if (any_row_mask) {
                            const int64_t kabs = key0 + warp * C::KPW + n * 8 + 2 * t4 + e;
                            if (!key_ok[n][e] || kabs > row_lim[m][h]) v = -CUDART_INF_F;
                        }
                        sacc[m][n][2 * h + e] = v;
                        mx = fmaxf(mx, v);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                if (t4 == 0) red_max[(buf * C::NW + warp) * ROWS + m * 16 + g + 8 * h] = mx;
            }
        }

        // ---- keys masked for every row: zero their V rows in shared memory
        if (any_row_mask && live) {
            bool ok_all = false;
            if (lane < C::KPW) {
                const int64_t kabs = key0 + warp * C::KPW + lane;
                ok_all = kabs < k_end;
                if (ok_all && tags) ok_all = kabs >= mem_lo || tag_ok(tag_of(kabs, tag_of_key(kabs, tg1_cur)));
            }
            uint32_t bad = ~__ballot_sync(0xffffffffu, ok_all) & ((1u << C::KPW) - 1u);
            if (bad) {
                while (bad) {
                    const int kl = warp * C::KPW + __ffs(bad) - 1;
                    bad &= bad - 1;
                    if (lane < C::NCH * 8)
                        st_shared_v4(sV + (lane >> 3) * (TK * 128) + swz128(kl, lane & 7),
                                     make_uint4(0u, 0u, 0u, 0u));
                }
                fence_proxy_async_smem();
            }
        }
        named_bar_sync(1, NCT);

        // ---- online softmax: new row max, P = 2^(s - m) to shared memory, rescale
        float alpha[MT][2];
        const uint32_t sPb = sP + buf * 2 * L::P_BYTES;  // [hi | lo] of this tile
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float m_use[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = m * 16 + g + 8 * h;
                float tmax = red_max[(buf * C::NW + 0) * ROWS + row];
#pragma unroll
                for (int w = 1; w < C::NW; ++w) tmax = fmaxf(tmax, red_max[(buf * C::NW + w) * ROWS + row]);
                const float m_new = fmaxf(m_run[m][h], tmax);
                m_use[h] = m_new == -CUDART_INF_F ? 0.f : m_new;
                alpha[m][h] = ex2(m_run[m][h] - m_use[h]);
                m_run[m][h] = m_new;
            }
            float lsum[2] = {0.f, 0.f};
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const float p0 = ex2(sacc[m][n][0] - m_use[0]);
                const float p1 = ex2(sacc[m][n][1] - m_use[0]);
                const float p2 = ex2(sacc[m][n][2] - m_use[1]);
                const float p3 = ex2(sacc[m][n][3] - m_use[1]);
                lsum[0] += p0 + p1;
                lsum[1] += p2 + p3;
                const __nv_bfloat162 r0 = __floats2bfloat162_rn(p0, p1);  // row g, hi part
                const __nv_bfloat162 r1 = __floats2bfloat162_rn(p2, p3);  // row g + 8, hi part
                const __nv_bfloat162 e0 =
                    __floats2bfloat162_rn(p0 - __low2float(r0), p1 - __high2float(r0));
                const __nv_bfloat162 e1 =
                    __floats2bfloat162_rn(p2 - __low2float(r1), p3 - __high2float(r1));
                const int chunk = (warp * C::KPW + n * 8) >> 3;
                const uint32_t o0 = swz128(m * 16 + g, chunk) + 4 * t4;
                const uint32_t o1 = swz128(m * 16 + g + 8, chunk) + 4 * t4;
                st_shared_u32(sPb + o0, *reinterpret_cast<const uint32_t *>(&r0));
                st_shared_u32(sPb + o1, *reinterpret_cast<const uint32_t *>(&r1));
                st_shared_u32(sPb + L::P_BYTES + o0, *reinterpret_cast<const uint32_t *>(&e0));
                st_shared_u32(sPb + L::P_BYTES + o1, *reinterpret_cast<const uint32_t *>(&e1));
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) l_run[m][h] = l_run[m][h] * alpha[m][h] + lsum[h];
#pragma unroll
            for (int n = 0; n < C::NTB; ++n) {
                oacc[m][n][0] *= alpha[m][0];
                oacc[m][n][1] *= alpha[m][0];
                oacc[m][n][2] *= alpha[m][1];
                oacc[m][n][3] *= alpha[m][1];
            }
        }
        named_bar_sync(1, NCT);

        // ---- O += P V over this warp's head-dim columns
        if (live) {
#pragma unroll
            for (int kk = 0; kk < TK / 16; ++kk) {
                uint32_t a[MT][4], e[MT][4];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const int row = m * 16 + (lm_idx & 1) * 8 + (lane & 7);
                    const uint32_t off = swz128(row, kk * 2 + (lm_idx >> 1));
                    ldsm_x4(sPb + off, a[m][0], a[m][1], a[m][2], a[m][3]);
                    ldsm_x4(sPb + L::P_BYTES + off, e[m][0], e[m][1], e[m][2], e[m][3]);
                }
#pragma unroll
                for (int nb = 0; nb < C::NTB / 2; ++nb) {
                    uint32_t v0, v1, v2, v3;
                    const int key = kk * 16 + (lm_idx & 1) * 8 + (lane & 7);
                    const int d = warp * C::DW + nb * 16 + (lm_idx >> 1) * 8;
                    ldsm_x4_t(sV + (d >> 6) * (TK * 128) + swz128(key, (d & 63) >> 3), v0, v1, v2, v3);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        mma_bf16(oacc[m][2 * nb], a[m], v0, v1);
                        mma_bf16(oacc[m][2 * nb + 1], a[m], v2, v3);
                        mma_bf16(oacc[m][2 * nb], e[m], v0, v1);
                        mma_bf16(oacc[m][2 * nb + 1], e[m], v2, v3);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        if (tags_global) {
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) tg_cur[n][e] = tg_nxt[n][e];
            tg1_cur = tg1_nxt;
        }
    }

    // ---- STEP: store the appended entry into the ring (every tile that
    // staged its slot has been consumed)
    if (has_new) {
        if (threadIdx.x < 2 * NVR) {
            uint4 *dst = static_cast<uint4 *>(threadIdx.x < NVR ? p.ring_k : p.ring_v);
            dst[(((int64_t)b * p.n_kv_heads + kvh) * p.n_slots + new_slot) * NVR + threadIdx.x % NVR] =
                s_new[threadIdx.x];
        }
        if (kvh == 0 && threadIdx.x == 0) p.tag_w[(int64_t)b * p.n_slots + new_slot] = (int32_t)qpos0;
    }

    // ---- row sums across lanes and warps, normalise, write
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float l = l_run[m][h];
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (t4 == 0) red_l[warp * ROWS + m * 16 + g + 8 * h] = l;
        }
    named_bar_sync(1, NCT);

    const float kLn2 = 0.693147180559945309f;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = m * 16 + g + 8 * h;
            if (row >= p.rows) continue;
            float lt = 0.f;
#pragma unroll
            for (int w = 0; w < C::NW; ++w) lt += red_l[w * ROWS + row];
            const bool has = lt > 0.f;
            const float inv = has ? 1.f / lt : 0.f;
            const float lse = has ? (m_run[m][h] + lg2(lt)) * kLn2 : -CUDART_INF_F;
            const int i = row / p.group, hh = row - (row / p.group) * p.group;
            const int64_t orow = ((int64_t)b * p.n_q + i) * p.n_q_heads + kvh * p.group + hh;
            if (p.o_part) {
                float *dst = p.o_part + (orow * p.n_split + split) * D;
#pragma unroll
                for (int n = 0; n < C::NTB; ++n) {
                    const int col = warp * C::DW + n * 8 + 2 * t4;
                    *reinterpret_cast<float2 *>(dst + col) =
                        make_float2(oacc[m][n][2 * h] * inv, oacc[m][n][2 * h + 1] * inv);
                }
                if (warp == 0 && t4 == 0) p.lse_part[orow * p.n_split + split] = lse;
            } else {
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) + orow * D;
#pragma unroll
                for (int n = 0; n < C::NTB; ++n) {
                    const int col = warp * C::DW + n * 8 + 2 * t4;
                    *reinterpret_cast<__nv_bfloat162 *>(dst + col) =
                        __floats2bfloat162_rn(oacc[m][n][2 * h] * inv, oacc[m][n][2 * h + 1] * inv);
                }
                if (warp == 0 && t4 == 0 && p.lse) p.lse[orow] = lse;
            }
        }
}

template <int D, int MT>
cudaError_t launch_attn_mt(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk, const CUtensorMap &mv,
                           const AttnParams &p, cudaStream_t stream) {
    constexpr int smem = AttnSmem<D, MT>::TOTAL;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(attn_kernel<D, MT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const dim3 grid(p.n_split, p.batch * p.n_kv_heads);
    return launch_pdl(attn_kernel<D, MT, false>, grid, dim3(kThreads), smem, stream, k, v, mk, mv, p);
}

template <int D, int MT>
cudaError_t launch_step_mt(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk, const CUtensorMap &mv,
                           const AttnParams &p, cudaStream_t stream) {
    constexpr int smem = AttnSmem<D, MT>::TOTAL;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(attn_kernel<D, MT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const dim3 grid(p.n_split, p.batch * p.n_kv_heads);
    return launch_pdl(attn_kernel<D, MT, true>, grid, dim3(kThreads), smem, stream, k, v, mk, mv, p);
}

template <int D>
cudaError_t launch_attn(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk, const CUtensorMap &mv,
                        const AttnParams &p, int m_tiles, cudaStream_t stream) {
    switch (m_tiles) {
        case 1: return launch_attn_mt<D, 1>(k, v, mk, mv, p, stream);
        case 2: return launch_attn_mt<D, 2>(k, v, mk, mv, p, stream);
        case 3: return launch_attn_mt<D, 3>(k, v, mk, mv, p, stream);
        case 4: return launch_attn_mt<D, 4>(k, v, mk, mv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D, int MT, bool STEP>
int blocks_per_sm_mt() {
    constexpr int smem = AttnSmem<D, MT>::TOTAL;
    if (cudaFuncSetAttribute(attn_kernel<D, MT, STEP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel<D, MT, STEP>, kThreads, smem) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int D>
int blocks_per_sm(int m_tiles, bool step) {
    switch (m_tiles) {
        case 1: return step ? blocks_per_sm_mt<D, 1, true>() : blocks_per_sm_mt<D, 1, false>();
        case 2: return step ? blocks_per_sm_mt<D, 2, true>() : blocks_per_sm_mt<D, 2, false>();
        case 3: return step ? blocks_per_sm_mt<D, 3, true>() : blocks_per_sm_mt<D, 3, false>();
        case 4: return step ? blocks_per_sm_mt<D, 4, true>() : blocks_per_sm_mt<D, 4, false>();
        default: return 0;
    }
}

template <int D>
cudaError_t launch_step(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk, const CUtensorMap &mv,
                        const AttnParams &p, int m_tiles, cudaStream_t stream) {
    switch (m_tiles) {
        case 1: return launch_step_mt<D, 1>(k, v, mk, mv, p, stream);
        case 2: return launch_step_mt<D, 2>(k, v, mk, mv, p, stream);
        case 3: return launch_step_mt<D, 3>(k, v, mk, mv, p, stream);
        case 4: return launch_step_mt<D, 4>(k, v, mk, mv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace wm

// attn_tc.cuh -- split-KV decode attention on the 5th-generation tensor cores.
//
// One CTA handles one (sequence, KV head) pair and one key range (a split);
// its NR rows (padded to a multiple of 16) are every query that reads this KV
// head, so each KV byte is read from HBM once per GQA group.  Keys are the
// MMA's M dimension (128 per tile), which keeps small row counts cheap:
//
//   S^T[128 keys x NR]  = K_tile[128 x D] . Q^T            (tcgen05, K-major A and B)
//   O^T[D x NR]        += V_tile^T[D x 128] . P^T[128 x NR] (tcgen05, MN-major A and B)
//
// S (double-buffered) and O live in tensor memory; the softmax row sums are
// kept per key-thread in registers and reduced once at the end.  The shared
// memory split between K/V staging slots and P^T buffers is chosen per head
// dim and row count: as many staging slots as fit, then a second P^T buffer
// if it still fits -- except 16-row tiles at head_dim 128, which keep a short
// ring of three slots (see tc_short_ring).  Warp roles (2 + 4g warps, g = NR / 8
// up to 32 rows, else NR / 16):
//   warp 0    : TMA producer -- K and V tiles (128-byte swizzle) into a ring of
//               shared-memory slots, K_t then V_t;
//   warp 1    : allocates tensor memory; one lane issues whichever MMA is ready
//               (S for the next tile, or P.V for the oldest tile whose P is
//               written) and commits it to mbarriers;
//   warps 2.. : softmax -- one key per thread (a tensor-memory lane), g warps
//               per lane quadrant each owning NR / g rows: scale and mask
//               the logits, keep a running row maximum (from a finite floor)
//               that is raised (with a rescale of O and L) only when a logit
//               exceeds it by more than 2^8, write P^T to shared memory as two
//               bf16 parts
//               (hi = bf16(p), lo = bf16(p - hi)), and finally normalise and
//               store the output.  P^T is double-buffered when shared memory
//               allows, so the softmax of tile t+1 overlaps P_t.V_t.
// Masks: verification is causal (query i sees positions <= seq_len - n_q + i);
// the draft sees a ring slot iff its tag t satisfies 0 <= t <= p and
// (t < sink or t > p - window).  Keys masked for every row get their V row
// zeroed in shared memory before the P.V product, so stale cache bytes (even
// NaN patterns) cannot leak through 0 * NaN.  Padding rows (past the real
// rows) see all-zero queries and are never stored.  Every wait is bounded.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>

#include "launch.h"
#include "ptx.cuh"
#include "tc.cuh"
#include "wm_internal.h"
#include "../../include/wm_api.h"

namespace wm {

constexpr int kTcKeyTile = 128;
constexpr int kTcPageCache = 256;  // block-table entries of one split kept in shared memory
// Softmax warps for NR rows: groups of four (one per tensor-memory lane
// quadrant), each group owning 8 rows up to 32 rows and 16 rows beyond (more
// warps would leave too few registers per thread).  More, shorter softmax
// warps hide the latency of the tensor-memory loads, MUFU and barriers per tile.
__host__ __device__ constexpr int tc_softmax_warps(int nr) { return nr <= 32 ? 4 * (nr / 8) : 4 * (nr / 16); }
// V tiles in 64-key halves at head_dim 256 with 48 or 64 rows (see TcPlan), streamed
// by one more warp than the other configurations have.
__host__ __device__ constexpr bool tc_split_v(int d, int nr) { return d == 256 && nr >= 48; }
__host__ __device__ constexpr int tc_threads(int d, int nr) {
    return (2 + tc_softmax_warps(nr) + (tc_split_v(d, nr) ? 1 : 0)) * 32;
}
constexpr float kLazyRescale = 8.f;  // raise the running max only past 2^8
constexpr float kMaxFloor = -1e30f;  // running-max start, below any finite logit (log2 units)

// NVS_ > 0: K tiles use the NSLOT_ slots and V tiles are staged separately
// as 64-key halves in NVS_ half-tile slots; else K and V tiles share the ring.
template <int D, int NR, int NSLOT_, int NPB_, int NVS_ = 0>
struct TcLayout {
    static constexpr int TK = kTcKeyTile;
    static constexpr int NSLOT = NSLOT_, NPB = NPB_, NVS = NVS_;
    static constexpr int NCH = D / 64;                         // 128-byte column chunks of a row
    static constexpr int NOC = D / 128;                        // O accumulators (M = 128 each)
    static constexpr int REGION = TK * 128;                    // one 64-column chunk of a tile
    static constexpr int SLOT_BYTES = TK * D * 2;              // one K or V tile
    static constexpr int VREGION = (TK / 2) * 128;             // one 64-column chunk of a V half tile
    static constexpr int VSLOT_BYTES = (TK / 2) * D * 2;       // one V half tile (64 keys)
    static constexpr int V_OFF = NSLOT * SLOT_BYTES;
    static constexpr int PT_ROW = NR <= 16 ? 32 : NR <= 32 ? 64 : 128;  // bytes per key row of P^T
    static constexpr int PT_SWIZZLE = NR <= 16 ? 6 : NR <= 32 ? 4 : 2;  // 32B / 64B / 128B swizzle (descriptor code)
    static constexpr int PT_ATOM = PT_ROW * 8;                 // one 8-key swizzle atom
    static constexpr int Q_OFF = V_OFF + NVS * VSLOT_BYTES;
    static constexpr int Q_REGION = NR * 128;
    static constexpr int PT_OFF = Q_OFF + NCH * Q_REGION;      // NPB x (P^T hi, P^T lo)
    static constexpr int PT_BYTES = TK * PT_ROW;
    static constexpr int RED_OFF = PT_OFF + 2 * NPB * PT_BYTES;  // float red[4][NR]
    static constexpr int FLAG_OFF = RED_OFF + 4 * NR * 4;        // int flags[64]
    static constexpr int BT_OFF = FLAG_OFF + 256;                // int page_cache[kTcPageCache]
    static constexpr int BAR_OFF = BT_OFF + 4 * kTcPageCache;
    static constexpr int NBAR = 2 * NSLOT + 2 * NVS + 10;
    static constexpr int TPTR_OFF = BAR_OFF + NBAR * 8;
    static constexpr int TOTAL = TPTR_OFF + 16 + 1024;
    static constexpr bool FITS = TOTAL <= 227 * 1024;
};

// A short staging ring (three 32 KB slots, one P^T buffer) for 16-row tiles at
// head_dim 128 in the split-plan kernel.  It was sized for two CTAs per SM,
// but a kernel that allocates tensor memory is resident at one CTA per SM
// (the occupancy query answers 1 for it whatever its registers and shared
// memory, where the same kernel without the allocation gets several), so
// the second CTA never arrives.  At one CTA per SM the short ring still
// measured 0-9% faster than the full one over the ragged paged mixes with
// the split plan (many short CTAs, each filling its ring from cold), so it
// stays there; the persistent kernel, one long run per CTA, takes the full
// ring (SHORT = false).
__host__ __device__ constexpr bool tc_short_ring(int d, int nr) { return d == 128 && nr == 16; }

// V tiles in 64-key halves at head_dim 256 with 48 or 64 rows: the query and
// P^T buffers leave room for only two 64 KB tile slots, so with a shared ring the
// next V tile could be requested only after the current P.V completes.  With
// one K slot and V half slots, a V half waits only for the P.V half that used
// its slot, and each half is 32 KB of whole key rows.

// Shared-memory plan: the most K/V staging slots (up to 6) that fit with one
// P^T buffer -- keeping enough HBM requests in flight per SM (well over 100 KB
// at loaded HBM latency) matters most -- then a second P^T buffer if it fits.
template <int D, int NR, bool SHORT = tc_short_ring(D, NR)>
struct TcPlan {
    static constexpr int NVS = tc_split_v(D, NR) ? 2 : 0;
    static constexpr int NSLOT = tc_split_v(D, NR) ? 1
                                 : SHORT ? 3
                                 : TcLayout<D, NR, 6, 1>::FITS   ? 6
                                 : TcLayout<D, NR, 5, 1>::FITS ? 5
                                 : TcLayout<D, NR, 4, 1>::FITS ? 4
                                 : TcLayout<D, NR, 3, 1>::FITS ? 3 : 2;
    static constexpr int NPB = !SHORT && TcLayout<D, NR, NSLOT, 2, NVS>::FITS ? 2 : 1;
};

template <int D, int NR, bool SHORT = tc_short_ring(D, NR)>
struct TcCfg {
    using L = TcLayout<D, NR, TcPlan<D, NR, SHORT>::NSLOT, TcPlan<D, NR, SHORT>::NPB, TcPlan<D, NR, SHORT>::NVS>;
    static constexpr int NSLOT = L::NSLOT, NPB = L::NPB, NVS = L::NVS;
    static constexpr bool SV = NVS > 0;                        // V staged in half tiles
    static constexpr int V_OFF = L::V_OFF, VREGION = L::VREGION, VSLOT_BYTES = L::VSLOT_BYTES;
    static constexpr int TK = L::TK, NCH = L::NCH, NOC = L::NOC, REGION = L::REGION;
    static constexpr int SLOT_BYTES = L::SLOT_BYTES;
    static constexpr int PT_ROW = L::PT_ROW, PT_SWIZZLE = L::PT_SWIZZLE, PT_ATOM = L::PT_ATOM;
    static constexpr int Q_OFF = L::Q_OFF, Q_REGION = L::Q_REGION, PT_OFF = L::PT_OFF, PT_BYTES = L::PT_BYTES;
    static constexpr int RED_OFF = L::RED_OFF;
    static constexpr int FLAG_OFF = L::FLAG_OFF, BAR_OFF = L::BAR_OFF, TPTR_OFF = L::TPTR_OFF, TOTAL = L::TOTAL;
    static constexpr int BT_OFF = L::BT_OFF;
    static constexpr int NSW = tc_softmax_warps(NR);            // softmax warps
    static constexpr int THREADS = tc_threads(D, NR);
    static constexpr int HR = NR / (NSW / 4);                  // rows per softmax warp
    static constexpr int S_COL = 0;                            // 2 x NR
    static constexpr int O_COL = 2 * NR;                       // NOC x NR
    static constexpr int TMEM_USED = O_COL + NOC * NR;
    static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
    static_assert(D == 128 || D == 256, "tensor-core path covers head_dim 128 and 256");
    static_assert(NR % 16 == 0 && NR >= 16 && NR <= 64, "rows per KV head");
    static_assert(Q_OFF % 1024 == 0 && PT_OFF % 1024 == 0 && PT_BYTES % 1024 == 0, "1024-byte regions");
    static_assert(L::FITS, "shared memory budget");
    static_assert(!SV || (NVS >= 2 && NSLOT >= 1 && D == 256), "half-tile V staging");
};

__device__ __forceinline__ void tc_report(int32_t *err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// The abort flag as lane 0 of the calling warp sees it, so that every lane
// takes the same branch around warp-collective tcgen05 loads and stores.
__device__ __forceinline__ bool warp_aborted(volatile int *flags) {
    return __shfl_sync(0xffffffffu, flags[0], 0) != 0;
}

// Self-check of a shared-memory range [lo, lo + len) against [base, end).
__device__ __forceinline__ bool in_smem(uint32_t lo, uint32_t len, uint32_t base, uint32_t end) {
    return lo >= base && lo + len <= end;
}

// (The minimum of two blocks for the short-ring instance only caps its
// registers, at the 95 it was measured with.)
template <int D, int NR>
__global__ void __launch_bounds__(tc_threads(D, NR), tc_short_ring(D, NR) ? 2 : 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const AttnParams p) {
    using C = TcCfg<D, NR>;
    constexpr int TK = C::TK;
    constexpr int HR = C::HR;
    constexpr int NSW = C::NSW;
    constexpr int kTcThreads = C::THREADS;
    constexpr int NPB = C::NPB;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gb = smem_raw + (sbase - raw);
    const uint32_t sQ = sbase + C::Q_OFF;
    const uint32_t sPT = sbase + C::PT_OFF;
    float *red = reinterpret_cast<float *>(gb + C::RED_OFF);                   // [4][NR]
    volatile int *flags = reinterpret_cast<volatile int *>(gb + C::FLAG_OFF);  // [0] abort, [8 + 8*buf + w] votes
    const uint32_t bars = sbase + C::BAR_OFF;
    const uint32_t bar_full0 = bars;                          // [NSLOT]
    const uint32_t bar_empty0 = bars + 8 * C::NSLOT;          // [NSLOT]
    const uint32_t bar_vfull0 = bars + 16 * C::NSLOT;         // [NVS] (V half tiles)
    const uint32_t bar_vempty0 = bar_vfull0 + 8 * C::NVS;     // [NVS]
    const uint32_t bar_sfull = bars + 16 * C::NSLOT + 16 * C::NVS;  // [2]
    const uint32_t bar_sfree = bar_sfull + 16;                // [2]
    const uint32_t bar_pfull = bar_sfree + 16;                // [2]
    const uint32_t bar_odone = bar_pfull + 16;                // [2]
    const uint32_t bar_qfull = bar_odone + 16;
    const uint32_t bar_final = bar_qfull + 8;
    uint32_t *tptr = reinterpret_cast<uint32_t *>(gb + C::TPTR_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int unit = blockIdx.y;
    const int b = unit / p.n_kv_heads;
    const int kvh = unit - b * p.n_kv_heads;
    const int split = blockIdx.x;

    // Set-up that touches only shared and tensor memory runs before the wait
    // on the previous kernel, while it drains: the pipeline barriers and this
    // CTA's tensor-memory columns (an allocation that finds them still held by
    // a draining CTA of the previous kernel waits for them; that kernel never
    // waits on this one).
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(bar_full0 + 8 * s, 1);
            mbar_init(bar_empty0 + 8 * s, 1);
        }
        for (int s = 0; s < C::NVS; ++s) {
            mbar_init(bar_vfull0 + 8 * s, 1);
            mbar_init(bar_vempty0 + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_sfull + 8 * i, 1);
            mbar_init(bar_sfree + 8 * i, NSW);
            mbar_init(bar_pfull + 8 * i, NSW);
            mbar_init(bar_odone + 8 * i, 1);
        }
        mbar_init(bar_qfull, NSW);
        mbar_init(bar_final, 1);
        for (int i = 0; i < 64; ++i) flags[i] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(tptr), C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tptr;

    pdl_wait();  // every global access below may depend on the previous kernel
    pdl_launch_dependents();
    int64_t n_keys, qpos0;
    if (p.source == KEYS_RING) {
        int64_t seen = p.n_seen[b];
        if (seen < 0) {
            if (threadIdx.x == 0) tc_report(p.err, WM_DEVERR_BAD_LENGTH);
            seen = 0;
        }
        n_keys = p.n_slots;
        qpos0 = seen - 1;
    } else {
        int64_t len = p.seq_lens[b];
        if (len < 0 || len > p.capacity) {
            if (threadIdx.x == 0) tc_report(p.err, WM_DEVERR_BAD_LENGTH);
            len = len < 0 ? 0 : p.capacity;
        }
        n_keys = len;
        qpos0 = len - p.n_q;
    }
    const int64_t k_begin = (int64_t)split * p.keys_per_split;
    const int64_t k_end = min(k_begin + (int64_t)p.keys_per_split, n_keys);
    const int n_tiles = k_end > k_begin ? (int)((k_end - k_begin + TK - 1) / TK) : 0;

    if (n_tiles == 0) {
        // An empty split (past the end of a shorter sequence): record "no keys"
        // for its rows, hand the tensor memory back and leave.
        for (int r = threadIdx.x; r < p.rows; r += kTcThreads) {
            const int qi = r / p.group, hh = r - qi * p.group;
            const int64_t orow = ((int64_t)b * p.n_q + qi) * p.n_q_heads + kvh * p.group + hh;
            if (p.o_part) {
                p.lse_part[orow * p.n_split + split] = -CUDART_INF_F;
            } else {
                if (p.lse) p.lse[orow] = -CUDART_INF_F;
                for (int d = 0; d < D; ++d) static_cast<__nv_bfloat16 *>(p.out)[orow * D + d] = __float2bfloat16_rn(0.f);
            }
        }
        if (warp == 1) tc::tmem_dealloc(tmem, C::TMEM_COLS);
        return;
    }


    if (warp == 0 || (C::SV && warp == 2 + NSW)) {
        // ======================================================== TMA producer
        // (half-tile V: warp 0 streams K, the last warp V)
        // Paged caches: the whole warp first copies this split's block-table
        // entries into shared memory, so that the lane issuing the copies never
        // waits on a global load per box (entries past the cache are read from
        // global memory as they are needed).
        int32_t *page_cache = reinterpret_cast<int32_t *>(gb + C::BT_OFF);
        const int64_t first_page = p.source == KEYS_PAGED ? k_begin / p.page_size : 0;
        if (warp == 0 && p.source == KEYS_PAGED) {
            const int64_t n_pages_split = (k_end - 1) / p.page_size - first_page + 1;
            for (int i = lane; i < kTcPageCache && i < n_pages_split; i += 32) {
                int32_t page = p.block_table[(int64_t)b * p.max_pages + first_page + i];
                if (page < 0 || page >= p.n_pages) {
                    tc_report(p.err, WM_DEVERR_BAD_PAGE);
                    page = 0;
                }
                page_cache[i] = page;
            }
            __syncwarp();
        }
        if (C::SV) {  // the V warp reads the block-table cache that warp 0 fills
            if (warp == 0)
                named_bar_arrive(2, 64);
            else
                named_bar_sync(2, 64);
        }
        if (C::SV && lane == 0 && n_tiles > 0) {
            // Warp 0 streams the K tiles into the tile slots, the V warp the V
            // tiles as 64-key halves into the half-tile slots, each on its own
            // barriers, so that neither waits for the other's slots.  Paged
            // boxes step through the pages as below.
            const bool is_v = warp != 0;
            const CUtensorMap *map = is_v ? &tmv : &tmk;
            prefetch_tensormap(map);
            const uint64_t policy = l2_policy_evict_first();
            const int nslot = is_v ? C::NVS : C::NSLOT;
            const int n_units = is_v ? 2 * n_tiles : n_tiles;
            const int unit_keys = is_v ? TK / 2 : TK;
            const int box = is_v ? TK / 2 : p.box_rows;
            const uint32_t full0 = is_v ? bar_vfull0 : bar_full0;
            const uint32_t empty0 = is_v ? bar_vempty0 : bar_empty0;
            const uint32_t slot_bytes = is_v ? C::VSLOT_BYTES : C::SLOT_BYTES;
            const uint32_t region = is_v ? C::VREGION : C::REGION;
            const uint32_t area0 = sbase + (is_v ? C::V_OFF : 0);
            const uint32_t area1 = area0 + nslot * slot_bytes;
            int issued = 0;
            int32_t last_page = 0;
            int64_t next_local = 0;
            int next_row = (int)(k_begin - first_page * p.page_size);
            for (int u = 0; u < n_units; ++u) {
                if (u == p.stall_tile) break;  // tests of the timeout path only
                const int s = u % nslot;
                if (u >= nslot && !mbar_wait_bounded(empty0 + 8 * s, ((u / nslot) & 1) ^ 1, p.wait_limit)) {
                    tc_report(p.err, WM_DEVERR_TIMEOUT);
                    flags[0] = 1;
                    break;
                }
                if (flags[0]) break;
                const uint32_t dst = area0 + s * slot_bytes;
                const int64_t key0 = k_begin + (int64_t)u * unit_keys;
                mbar_arrive_expect_tx(full0 + 8 * s, slot_bytes);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h * box >= unit_keys) break;
                    const int64_t kh = key0 + (int64_t)h * box;
                    int c_row, c_outer;
                    if (p.source == KEYS_PAGED) {
                        if (kh < n_keys) {
                            int32_t page;
                            if (next_local < kTcPageCache) {
                                page = page_cache[next_local];
                            } else {
                                page = p.block_table[(int64_t)b * p.max_pages + first_page + next_local];
                                if (page < 0 || page >= p.n_pages) {
                                    tc_report(p.err, WM_DEVERR_BAD_PAGE);
                                    page = 0;
                                }
                            }
                            last_page = page;
                        }
                        c_row = next_row;  // past the end: any valid page, masked later
                        c_outer = last_page;
                        next_row += box;
                        if (next_row >= p.page_size) {
                            next_row = 0;
                            ++next_local;
                        }
                    } else {
                        c_row = (int)kh;
                        c_outer = b;
                    }
                    if (!in_smem(dst + (C::NCH - 1) * region + h * box * 128, box * 128, area0, area1) ||
                        c_row < 0 || c_outer < 0) {
                        tc_report(p.err, WM_DEVERR_INTERNAL);
                        flags[0] = 1;
                        break;
                    }
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_4d(dst + c * region + h * box * 128, map, full0 + 8 * s, c * 64, c_row, kvh,
                                    c_outer, policy);
                }
                issued = u + 1;
            }
            // Never leave the CTA with bulk copies still landing in its shared memory.
            for (int u = max(0, issued - nslot); u < issued; ++u)
                mbar_wait_bounded(full0 + 8 * (u % nslot), (u / nslot) & 1, p.wait_limit);
        } else if (!C::SV && lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
            const uint64_t policy = l2_policy_evict_first();
            int issued = 0;
            int32_t last_page = 0;
            // Paged: the boxes of a split step through its pages in order (a box
            // never crosses a page), so the page and row of each box advance
            // without a division per box.  Tile t's boxes serve K_t and V_t.
            int64_t next_local = 0;                                   // page of the next box, from first_page
            int next_row = (int)(k_begin - first_page * p.page_size);  // its first row in that page
            int box_page[2] = {0, 0}, box_row[2] = {0, 0};            // tile t's boxes (TK / box_rows <= 2)
            for (int u = 0; u < 2 * n_tiles; ++u) {
                if (u == p.stall_tile) break;  // tests of the timeout path only
                const int s = u % C::NSLOT;
                if (u >= C::NSLOT &&
                    !mbar_wait_bounded(bar_empty0 + 8 * s, ((u / C::NSLOT) & 1) ^ 1, p.wait_limit)) {
                    tc_report(p.err, WM_DEVERR_TIMEOUT);
                    flags[0] = 1;
                    break;
                }
                if (flags[0]) break;
                const int t = u >> 1;
                const CUtensorMap *map = (u & 1) ? &tmv : &tmk;
                const uint32_t dst = sbase + s * C::SLOT_BYTES;
                const int64_t key0 = k_begin + (int64_t)t * TK;
                if (p.source == KEYS_PAGED && (u & 1) == 0) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h * p.box_rows >= TK) break;
                        if (key0 + (int64_t)h * p.box_rows < n_keys) {
                            int32_t page;
                            if (next_local < kTcPageCache) {
                                page = page_cache[next_local];
                            } else {
                                page = p.block_table[(int64_t)b * p.max_pages + first_page + next_local];
                                if (page < 0 || page >= p.n_pages) {
                                    tc_report(p.err, WM_DEVERR_BAD_PAGE);
                                    page = 0;
                                }
                            }
                            last_page = page;
                        }
                        box_page[h] = last_page;  // past the end: any valid page, masked later
                        box_row[h] = next_row;
                        next_row += p.box_rows;
                        if (next_row >= p.page_size) {
                            next_row = 0;
                            ++next_local;
                        }
                    }
                }
                mbar_arrive_expect_tx(bar_full0 + 8 * s, C::SLOT_BYTES);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // TK / box_rows boxes: one (128 rows) or two (64)
                    if (h * p.box_rows >= TK) break;
                    const int64_t kh = key0 + (int64_t)h * p.box_rows;
                    int c_row, c_outer;
                    if (p.source == KEYS_PAGED) {
                        c_row = box_row[h];
                        c_outer = box_page[h];
                    } else {
                        c_row = (int)kh;
                        c_outer = b;
                    }
                    if (!in_smem(dst + (C::NCH - 1) * C::REGION + h * p.box_rows * 128, p.box_rows * 128,
                                 sbase, sbase + C::NSLOT * C::SLOT_BYTES) ||
                        c_row < 0 || c_outer < 0) {
                        tc_report(p.err, WM_DEVERR_INTERNAL);
                        flags[0] = 1;
                        break;
                    }
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_4d(dst + c * C::REGION + h * p.box_rows * 128, map, bar_full0 + 8 * s, c * 64,
                                    c_row, kvh, c_outer, policy);
                }
                issued = u + 1;
            }
            for (int u = max(0, issued - C::NSLOT); u < issued; ++u)
                mbar_wait_bounded(bar_full0 + 8 * (u % C::NSLOT), (u / C::NSLOT) & 1, p.wait_limit);
        }
    } else if (warp == 1) {
        // ======================================================== MMA issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t id_s = tc::idesc_bf16(128, NR, 0, 0);
            constexpr uint32_t id_pv = tc::idesc_bf16(128, NR, 1, 1);
            bool ok = mbar_wait_bounded(bar_qfull, 0, p.wait_limit);
            // Issue whichever product is ready -- S for the next tile (its K
            // landed and its tensor-memory buffer is free) or P.V for the
            // oldest tile whose P is written -- so that neither waits on the
            // other's inputs.
            int ts = 0, tp = 0;
            int th = 0;  // half-tile V: the half of tile tp whose P.V is next
            uint32_t idle = 0;
            while (ok && tp < n_tiles) {
                if (flags[0]) break;
                bool did = false;
                if (ts < n_tiles) {
                    // the K unit of tile ts: 2 ts in the shared ring, or ts in the K ring
                    const int uk = C::SV ? ts : 2 * ts, sk = uk % C::NSLOT;
                    // A parity test cannot tell "this fill landed" from "the fill
                    // before it has not landed yet" (the parities match), so only
                    // test once the slot's previous unit is known to have landed:
                    // its consumer (S for a K unit, P.V for a V unit) was issued.
                    // (A K ring holds K units only, consumed in order: always so.)
                    const int prev = uk - C::NSLOT;
                    const bool prev_in =
                        C::SV || prev < 0 || ((prev & 1) ? (prev >> 1) < tp : (prev >> 1) < ts);
                    if (prev_in && mbar_test(bar_full0 + 8 * sk, (uk / C::NSLOT) & 1) &&
                        (ts < 2 || mbar_test(bar_sfree + 8 * (ts & 1), ((ts - 2) >> 1) & 1))) {
                        tc::fence_after_sync();
                        const uint32_t d_s = tmem + C::S_COL + (ts & 1) * NR;
                        const uint32_t a_k = sbase + sk * C::SLOT_BYTES;
                        if (!in_smem(a_k, C::SLOT_BYTES, sbase, sbase + C::NSLOT * C::SLOT_BYTES) ||
                            !in_smem(sQ, C::NCH * C::Q_REGION, sbase + C::Q_OFF, sbase + C::PT_OFF)) {
                            tc_report(p.err, WM_DEVERR_INTERNAL);
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t a =
                                    tc::smem_desc(a_k + c * C::REGION + kk * 32, 16, 1024, tc::SWIZZLE_128B);
                                const uint64_t bq =
                                    tc::smem_desc(sQ + c * C::Q_REGION + kk * 32, 16, 1024, tc::SWIZZLE_128B);
                                tc::mma_f16_ss(d_s, a, bq, id_s, (c | kk) != 0);
                            }
                        tc::commit(bar_sfull + 8 * (ts & 1));
                        tc::commit(bar_empty0 + 8 * sk);
                        ++ts;
                        did = true;
                    }
                }
                if (C::SV && tp < ts) {
                    // P.V of one 64-key V half: the half's slot held an earlier
                    // half, whose P.V was issued before (halves go in order)
                    const int uv = 2 * tp + th, sv = uv % C::NVS;
                    if (mbar_test(bar_pfull + 8 * (tp & 1), (tp >> 1) & 1) &&
                        mbar_test(bar_vfull0 + 8 * sv, (uv / C::NVS) & 1)) {
                        tc::fence_after_sync();
                        const uint32_t a_v = sbase + C::V_OFF + sv * C::VSLOT_BYTES;
                        const uint32_t pt = sPT + (tp % NPB) * 2 * C::PT_BYTES;
                        if (!in_smem(a_v, C::VSLOT_BYTES, sbase + C::V_OFF, sbase + C::V_OFF + C::NVS * C::VSLOT_BYTES) ||
                            !in_smem(pt, 2 * C::PT_BYTES, sPT, sPT + 2 * NPB * C::PT_BYTES)) {
                            tc_report(p.err, WM_DEVERR_INTERNAL);
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int k4 = 0; k4 < TK / 32; ++k4) {  // 16-key steps within the half
                            const int kk = th * (TK / 32) + k4;
                            const uint32_t first = (tp == 0 && kk == 0) ? 0u : 1u;
                            const uint32_t koff = kk * 2 * C::PT_ATOM;
                            const uint64_t b_hi =
                                tc::smem_desc(pt + koff, C::PT_BYTES, C::PT_ATOM, C::PT_SWIZZLE);
                            const uint64_t b_lo =
                                tc::smem_desc(pt + C::PT_BYTES + koff, C::PT_BYTES, C::PT_ATOM, C::PT_SWIZZLE);
#pragma unroll
                            for (int m = 0; m < C::NOC; ++m) {
                                const uint64_t a = tc::smem_desc(a_v + 2 * m * C::VREGION + k4 * 2048, C::VREGION,
                                                                 1024, tc::SWIZZLE_128B);
                                const uint32_t d_o = tmem + C::O_COL + m * NR;
                                tc::mma_f16_ss(d_o, a, b_hi, id_pv, first);
                                tc::mma_f16_ss(d_o, a, b_lo, id_pv, 1u);
                            }
                        }
                        tc::commit(bar_vempty0 + 8 * sv);
                        if (th == 1) {
                            tc::commit(bar_odone + 8 * (tp & 1));
                            ++tp;
                            th = 0;
                        } else {
                            th = 1;
                        }
                        did = true;
                    }
                } else if (tp < ts) {
                    const int uv = 2 * tp + 1, sv = uv % C::NSLOT;
                    const int prev = uv - C::NSLOT;  // see the K test above
                    const bool prev_in = prev < 0 || ((prev & 1) ? (prev >> 1) < tp : (prev >> 1) < ts);
                    if (prev_in && mbar_test(bar_pfull + 8 * (tp & 1), (tp >> 1) & 1) &&
                        mbar_test(bar_full0 + 8 * sv, (uv / C::NSLOT) & 1)) {
                        tc::fence_after_sync();
                        const uint32_t a_v = sbase + sv * C::SLOT_BYTES;
                        const uint32_t pt = sPT + (tp % NPB) * 2 * C::PT_BYTES;
                        if (!in_smem(a_v, C::SLOT_BYTES, sbase, sbase + C::NSLOT * C::SLOT_BYTES) ||
                            !in_smem(pt, 2 * C::PT_BYTES, sPT, sPT + 2 * NPB * C::PT_BYTES)) {
                            tc_report(p.err, WM_DEVERR_INTERNAL);
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int kk = 0; kk < TK / 16; ++kk) {
                            const uint32_t first = (tp == 0 && kk == 0) ? 0u : 1u;
                            const uint32_t koff = kk * 2 * C::PT_ATOM;  // 16 keys = two 8-key atoms
                            const uint64_t b_hi =
                                tc::smem_desc(pt + koff, C::PT_BYTES, C::PT_ATOM, C::PT_SWIZZLE);
                            const uint64_t b_lo =
                                tc::smem_desc(pt + C::PT_BYTES + koff, C::PT_BYTES, C::PT_ATOM, C::PT_SWIZZLE);
#pragma unroll
                            for (int m = 0; m < C::NOC; ++m) {
                                const uint64_t a = tc::smem_desc(a_v + 2 * m * C::REGION + kk * 2048, C::REGION,
                                                                 1024, tc::SWIZZLE_128B);
                                const uint32_t d_o = tmem + C::O_COL + m * NR;
                                tc::mma_f16_ss(d_o, a, b_hi, id_pv, first);
                                tc::mma_f16_ss(d_o, a, b_lo, id_pv, 1u);
                            }
                        }
                        tc::commit(bar_odone + 8 * (tp & 1));
                        tc::commit(bar_empty0 + 8 * sv);
                        ++tp;
                        did = true;
                    }
                }
                if (did) {
                    idle = 0;
                } else if (++idle > p.wait_limit) {
                    ok = false;
                } else if (idle > 64) {
                    __nanosleep(32);
                }
            }
            if (!ok) {
                tc_report(p.err, WM_DEVERR_TIMEOUT);
                flags[0] = 1;
            }
            tc::commit(bar_final);  // every MMA issued above has completed once this fires
            mbar_wait_bounded(bar_final, 0, p.wait_limit);
        }
    } else {
        // ======================================================== softmax warps
        const int sw = warp - 2;                       // 0..NSW-1
        const int q4 = warp & 3;                       // tensor-memory lane quadrant
        const int r0 = (sw >> 2) * HR;                 // first row of this warp's group
        const int kt = 32 * q4 + lane;                 // key within the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const int ct = threadIdx.x - 64;               // 0..32*NSW-1
        {
            const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
            constexpr int VPR = D / 8;
            for (int idx = ct; idx < NR * VPR; idx += 32 * NSW) {
                const int r = idx / VPR, v = idx - (idx / VPR) * VPR;
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                if (r < p.rows) {
                    const int i = r / p.group, hh = r - i * p.group;
                    const int64_t row = ((int64_t)b * p.n_q + i) * p.n_q_heads + kvh * p.group + hh;
                    val = __ldg(reinterpret_cast<const uint4 *>(q + row * D) + v);
                }
                st_shared_v4(sQ + (v >> 3) * C::Q_REGION + swz128(r, v & 7), val);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_qfull);
        }
        const int32_t *tags = p.source == KEYS_RING ? p.pos_tag + (int64_t)b * p.n_slots : nullptr;
        // Running max (the same in every thread) and this key-thread's sum.  The
        // max starts at a finite floor rather than -inf: any visible logit exceeds
        // it by more than the lazy margin, so the first one raises it before a P
        // is formed, and 2^(s - m) needs no -inf guard (masked s = -inf gives 0).
        float m_run[HR], l_run[HR];
#pragma unroll
        for (int i = 0; i < HR; ++i) {
            m_run[i] = kMaxFloor;
            l_run[i] = 0.f;
        }
        // 8-row chunks of this warp's rows that hold real rows (warp-uniform);
        // padding rows (the MMA's N is a multiple of 16) get P = 0 without work
        const int live_chunks = min(HR / 8, max(0, (p.rows - r0 + 7) / 8));

        for (int t = 0; t < n_tiles; ++t) {
            const int64_t key0 = k_begin + (int64_t)t * TK;
            const int64_t kabs = key0 + kt;
            bool key_ok = kabs < k_end;
            if (key_ok && tags) {
                const int64_t tg = tags[kabs];
                key_ok = tg >= 0 && tg <= qpos0 && (tg < p.sink || tg > qpos0 - p.window);
            }
            float s[HR];
            bool live = !warp_aborted(flags);
            if (live && !mbar_wait_bounded(bar_sfull + 8 * (t & 1), (t >> 1) & 1, p.wait_limit)) {
                tc_report(p.err, WM_DEVERR_TIMEOUT);
                flags[0] = 1;
            }
            live = !warp_aborted(flags);
            tc::fence_after_sync();  // order the S loads after the MMA completion observed above
#pragma unroll
            for (int i = 0; i < HR; ++i) s[i] = -CUDART_INF_F;
            if (live) {
#pragma unroll
                for (int c = 0; c < HR / 8; ++c)
                    if (c < live_chunks)
                        tc::ld_32x32b_x8(tmem + lane_off + C::S_COL + (t & 1) * NR + r0 + 8 * c, s + 8 * c);
                tc::wait_ld();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_sfree + 8 * (t & 1));

            // scale to base 2; mask only tiles that reach a boundary
            const bool causal_tile = p.source != KEYS_RING && key0 + TK - 1 > qpos0;
            const bool key_tile = tags != nullptr || key0 + TK > k_end;
            const int64_t rel = qpos0 - kabs;  // key visible to row r iff rel + r / group >= 0
            // The logit in log2 units is s * f: boundary tiles store the scaled,
            // masked logit in s (f = 1); interior tiles keep the raw product and
            // fold the scale into the FFMA s * f - m of the vote and of P.
            bool need = false;
            float f = 1.f;
            if (key_tile || causal_tile) {
#pragma unroll
                for (int i = 0; i < HR; ++i) {
                    bool ok = i < 8 * live_chunks;
                    if (key_tile) ok = ok && key_ok;
                    if (causal_tile) ok = ok && rel + (r0 + i) / p.group >= 0;
                    const float v = ok ? s[i] * p.scale_log2 : -CUDART_INF_F;
                    s[i] = v;
                    need |= v - m_run[i] > kLazyRescale;
                }
            } else {  // interior tile: every key visible to every real row (padding rows stay -inf)
                f = p.scale_log2;
#pragma unroll
                for (int c = 0; c < HR / 8; ++c)
                    if (c < live_chunks) {
#pragma unroll
                        for (int i = 8 * c; i < 8 * c + 8; ++i) need |= fmaf(s[i], f, -m_run[i]) > kLazyRescale;
                    }
            }
            const unsigned any = __ballot_sync(0xffffffffu, need);
            if (lane == 0) flags[8 + 16 * (t & 1) + sw] = any != 0u;
            named_bar_sync(1, 32 * NSW);
            int votes = 0;
#pragma unroll
            for (int w = 0; w < NSW; ++w) votes |= flags[8 + 16 * (t & 1) + w];
            const bool rescale = votes != 0;  // the same in every softmax thread
            if (rescale) {
#pragma unroll
                for (int i = 0; i < HR; ++i) {
                    float mx = i < 8 * live_chunks ? s[i] * f : -CUDART_INF_F;
#pragma unroll
                    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    if (lane == 0) red[NR * q4 + r0 + i] = mx;
                }
                named_bar_sync(1, 32 * NSW);
            }
            bool o_stable = t == 0;  // P_{t-1}.V_{t-1} known complete
            if (rescale) {
                float alpha[HR];
#pragma unroll
                for (int i = 0; i < HR; ++i) {
                    const int r = r0 + i;
                    const float m_new =
                        fmaxf(m_run[i], fmaxf(fmaxf(red[r], red[NR + r]), fmaxf(red[2 * NR + r], red[3 * NR + r])));
                    alpha[i] = ex2(m_run[i] - m_new);
                    m_run[i] = m_new;
                    l_run[i] *= alpha[i];
                }
                if (t > 0) {
                    // O holds tiles 0..t-1 at the old maximum: wait for P_{t-1}.V_{t-1}, then rescale
                    if (!flags[0] && !mbar_wait_bounded(bar_odone + 8 * ((t - 1) & 1), ((t - 1) >> 1) & 1, p.wait_limit)) {
                        tc_report(p.err, WM_DEVERR_TIMEOUT);
                        flags[0] = 1;
                    }
                    o_stable = true;
                    tc::fence_after_sync();
                    if (!warp_aborted(flags)) {
#pragma unroll
                        for (int a = 0; a < C::NOC; ++a) {
                            const uint32_t col = C::O_COL + a * NR + r0;
#pragma unroll
                            for (int c = 0; c < HR / 8; ++c) {
                                float v8[8];
                                tc::ld_32x32b_x8(tmem + lane_off + col + 8 * c, v8);
                                tc::wait_ld();
#pragma unroll
                                for (int i = 0; i < 8; ++i) v8[i] *= alpha[8 * c + i];
                                tc::st_32x32b_x8(tmem + lane_off + col + 8 * c, v8);
                            }
                        }
                        tc::wait_st();
                    }
                }
            }

            // P = 2^(s - m) as bf16 hi + lo parts into P^T[key][row]
            uint32_t hi_w[HR / 2], lo_w[HR / 2];
#pragma unroll
            for (int i = 0; i < HR; i += 2) {
                if (i >= 8 * live_chunks) {  // padding rows
                    hi_w[i / 2] = 0u;
                    lo_w[i / 2] = 0u;
                    continue;
                }
                const float pa = ex2(fmaf(s[i], f, -m_run[i])), pb = ex2(fmaf(s[i + 1], f, -m_run[i + 1]));
                l_run[i] += pa;
                l_run[i + 1] += pb;
                const __nv_bfloat162 h = __floats2bfloat162_rn(pa, pb);
                const __nv_bfloat162 l = __floats2bfloat162_rn(pa - __low2float(h), pb - __high2float(h));
                hi_w[i / 2] = *reinterpret_cast<const uint32_t *>(&h);
                lo_w[i / 2] = *reinterpret_cast<const uint32_t *>(&l);
            }
            // the P^T buffer of this tile was last read by P_{t-NPB}.V_{t-NPB}
            if (t >= NPB && !(NPB == 1 && o_stable) && !flags[0] &&
                !mbar_wait_bounded(bar_odone + 8 * ((t - NPB) & 1), ((t - NPB) >> 1) & 1, p.wait_limit)) {
                tc_report(p.err, WM_DEVERR_TIMEOUT);
                flags[0] = 1;
            }
            const uint32_t pt = sPT + (t % NPB) * 2 * C::PT_BYTES;
#pragma unroll
            for (int j = 0; j < HR / 8; ++j) {
                // MN-major P^T: key kt's row of PT_ROW bytes, 16-byte chunks of
                // 8 rows permuted by the 128B (chunk ^ kt%8), 64B
                // (chunk ^ (kt/2)%4) or 32B (chunk ^ (kt/4)%2) swizzle
                const int chunk = r0 / 8 + j;
                const uint32_t phys = C::PT_ROW == 128 ? (uint32_t)(chunk ^ (kt & 7))
                                      : C::PT_ROW == 64 ? (uint32_t)(chunk ^ ((kt >> 1) & 3))
                                                        : (uint32_t)(chunk ^ ((kt >> 2) & 1));
                const uint32_t off = (uint32_t)kt * C::PT_ROW + (phys << 4);
                st_shared_v4(pt + off, make_uint4(hi_w[4 * j], hi_w[4 * j + 1], hi_w[4 * j + 2], hi_w[4 * j + 3]));
                st_shared_v4(pt + C::PT_BYTES + off,
                             make_uint4(lo_w[4 * j], lo_w[4 * j + 1], lo_w[4 * j + 2], lo_w[4 * j + 3]));
            }
            if (!key_ok && r0 == 0 && !flags[0]) {
                // A key no row may see: zero its V row once the V tile has landed.
                // The slot's previous unit is older than tile t-1's V, so once
                // P_{t-1}.V_{t-1} is complete that unit has landed too and the
                // parity wait below cannot mistake it for this tile's V.
                // (with half-tile V: the half holding key kt, whose slot's previous
                // half belongs to tile t-1 or earlier)
                const int uv = C::SV ? 2 * t + kt / (TK / 2) : 2 * t + 1;
                const int nsl = C::SV ? C::NVS : C::NSLOT, sv = uv % nsl;
                const uint32_t vfull = (C::SV ? bar_vfull0 : bar_full0) + 8 * sv;
                const bool prev_in =
                    t == 0 || mbar_wait_bounded(bar_odone + 8 * ((t - 1) & 1), ((t - 1) >> 1) & 1, p.wait_limit);
                if (prev_in && mbar_wait_bounded(vfull, (uv / nsl) & 1, p.wait_limit)) {
                    const uint32_t vrow = C::SV ? sbase + C::V_OFF + sv * C::VSLOT_BYTES : sbase + sv * C::SLOT_BYTES;
                    const uint32_t region = C::SV ? C::VREGION : C::REGION;
                    const int krow = C::SV ? kt % (TK / 2) : kt;
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_shared_v4(vrow + c * region + swz128(krow, j), make_uint4(0u, 0u, 0u, 0u));
                } else {
                    tc_report(p.err, WM_DEVERR_TIMEOUT);
                    flags[0] = 1;
                }
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pfull + 8 * (t & 1));
        }

        // ---- epilogue: this thread owns tensor-memory lane d = 32*q4 + lane of every O block
        if (n_tiles > 0 && !flags[0] &&
            !mbar_wait_bounded(bar_odone + 8 * ((n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1, p.wait_limit)) {
            tc_report(p.err, WM_DEVERR_TIMEOUT);
            flags[0] = 1;
        }
        tc::fence_after_sync();
        const bool have = n_tiles > 0 && !warp_aborted(flags);
        const float kLn2 = 0.693147180559945309f;
        // row sums: over the 32 keys of this warp, then over the 4 lane quadrants
        // (the barrier keeps slower warps' last reads of red[] ahead of these writes)
        named_bar_sync(1, 32 * NSW);
#pragma unroll
        for (int i = 0; i < HR; ++i) {
            float l = l_run[i];
#pragma unroll
            for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            if (lane == 0) red[NR * q4 + r0 + i] = l;
        }
        named_bar_sync(1, 32 * NSW);
#pragma unroll
        for (int c = 0; c < HR / 8; ++c) {
            float l8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = r0 + 8 * c + i;
                l8[i] = have ? red[r] + red[NR + r] + red[2 * NR + r] + red[3 * NR + r] : 0.f;
            }
#pragma unroll
            for (int m = 0; m < C::NOC; ++m) {
                float o8[8];
                if (have) {
                    tc::ld_32x32b_x8(tmem + lane_off + C::O_COL + m * NR + r0 + 8 * c, o8);
                    tc::wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) o8[i] = 0.f;
                }
                const int d = m * 128 + 32 * q4 + lane;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = r0 + 8 * c + i;
                    if (r >= p.rows) continue;
                    const float lt = l8[i];
                    const float o = lt > 0.f ? o8[i] / lt : 0.f;
                    const int qi = r / p.group, hh = r - qi * p.group;
                    const int64_t orow = ((int64_t)b * p.n_q + qi) * p.n_q_heads + kvh * p.group + hh;
                    if (p.o_part)
                        p.o_part[(orow * p.n_split + split) * D + d] = o;
                    else
                        static_cast<__nv_bfloat16 *>(p.out)[orow * D + d] = __float2bfloat16_rn(o);
                }
            }
            // lse of row r is written by the thread that owns tensor-memory lane r
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = r0 + 8 * c + i;
                if (r >= p.rows || kt != r) continue;
                const float lt = l8[i];
                const float lse = lt > 0.f ? (m_run[8 * c + i] + lg2(lt)) * kLn2 : -CUDART_INF_F;
                const int qi = r / p.group, hh = r - qi * p.group;
                const int64_t orow = ((int64_t)b * p.n_q + qi) * p.n_q_heads + kvh * p.group + hh;
                if (p.o_part)
                    p.lse_part[orow * p.n_split + split] = lse;
                else if (p.lse)
                    p.lse[orow] = lse;
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, int NR>
cudaError_t launch_attn_tc_nr(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p,
                              cudaStream_t stream) {
    constexpr int smem = TcCfg<D, NR>::TOTAL;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(attn_tc_kernel<D, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const dim3 grid(p.n_split, p.batch * p.n_kv_heads);
    return launch_pdl(attn_tc_kernel<D, NR>, grid, dim3(TcCfg<D, NR>::THREADS), smem, stream, k, v, p);
}

template <int D, int NR>
int tc_blocks_per_sm_nr() {
    constexpr int smem = TcCfg<D, NR>::TOTAL;
    if (cudaFuncSetAttribute(attn_tc_kernel<D, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_tc_kernel<D, NR>, TcCfg<D, NR>::THREADS, smem) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int D>
cudaError_t launch_attn_tc(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p, int n_rows16,
                           cudaStream_t stream) {
    switch (n_rows16) {
        case 16: return launch_attn_tc_nr<D, 16>(k, v, p, stream);
        case 32: return launch_attn_tc_nr<D, 32>(k, v, p, stream);
        case 48: return launch_attn_tc_nr<D, 48>(k, v, p, stream);
        case 64: return launch_attn_tc_nr<D, 64>(k, v, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
int tc_blocks_per_sm(int n_rows16) {
    switch (n_rows16) {
        case 16: return tc_blocks_per_sm_nr<D, 16>();
        case 32: return tc_blocks_per_sm_nr<D, 32>();
        case 48: return tc_blocks_per_sm_nr<D, 48>();
        case 64: return tc_blocks_per_sm_nr<D, 64>();
        default: return 0;
    }
}

}  // namespace wm

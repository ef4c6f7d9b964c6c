// attn_tcp.cuh -- persistent verify attention on the 5th-generation tensor
// cores for a batch of sequences of different lengths.
//
// The per-tile pipeline is the one of attn_tc_kernel (attn_tc.cuh): keys as
// the MMA's M dimension, S^T = K_tile . Q^T and O^T += V_tile^T . P^T in
// tensor memory, P as bf16 hi + lo parts, a TMA producer warp, one MMA-issuing
// lane and 4g softmax warps with a lazily raised running maximum.  What
// differs is the work of a CTA: instead of one (sequence, KV head, split),
// each of the grid's CTAs -- as many as are resident at once -- takes an
// equal run of the batch's key tiles laid end to end (verify_sched.cu), which
// may cross from one (sequence, KV head) unit into the next.  Each unit the
// run touches is a segment with its own queries, key range and causal
// boundary, and leaves one partial for the segment merge.
//
// Across segments every role keeps counting tiles, so the staging ring, the
// two S buffers and the P^T buffers roll on without a drain: the producer
// already streams the next segment's tiles while the softmax warps finish the
// current one.  Per segment boundary:
//   - the softmax warps write the next segment's queries into the (single)
//     query buffer as soon as they have read the last S of the current one
//     (every S product that read the old queries has completed by then) and
//     arrive on the query barrier, whose phase k belongs to segment k; the
//     MMA lane issues a segment's first S only after that phase completes;
//   - the first P.V of a segment overwrites the O accumulator (accumulate =
//     0).  It needs that segment's first P, which every softmax warp writes
//     only after it has read its part of the previous segment's O, so the O
//     buffer needs no barrier of its own;
//   - the running maxima and row sums restart.
// Configurations that stage V in half tiles (head_dim 256, > 32 rows) are not
// instantiated (tcp_supported).  Every wait is bounded.
#pragma once

#include "attn_tc.cuh"

namespace wm {

// Walks the segments of one CTA's run: tiles [t0, t0 + n) of unit (b, kvh).
// Every role keeps its own walker; all see the same sequence.
struct TcpWalk {
    int b, kvh;
    int t_off;  // next tile within unit (b, kvh)
    int left;   // tiles of the run not yet handed out
    __device__ __forceinline__ void init(int4 st) {
        b = st.x;
        kvh = st.y;
        t_off = st.z;
        left = st.w;
    }
    __device__ __forceinline__ bool next(const AttnParams &p, int &sb, int &skvh, int &t0, int &n) {
        while (left > 0 && b < p.batch) {
            const int nt = (int)(p.tile_prefix[b + 1] - p.tile_prefix[b]);
            if (nt <= 0) {  // a sequence without keys: no unit of it holds a tile
                ++b;
                kvh = 0;
                t_off = 0;
                continue;
            }
            if (t_off < nt) {
                const int take = min(nt - t_off, left);
                sb = b;
                skvh = kvh;
                t0 = t_off;
                n = take;
                left -= take;
                t_off += take;
                if (t_off >= nt) {
                    t_off = 0;
                    if (++kvh == p.n_kv_heads) {
                        kvh = 0;
                        ++b;
                    }
                }
                return true;
            }
            t_off = 0;
            if (++kvh == p.n_kv_heads) {
                kvh = 0;
                ++b;
            }
        }
        return false;
    }
};

// Length of sequence b, clamped as the schedule clamped it (the schedule
// kernel reports a bad length).
__device__ __forceinline__ int64_t tcp_len(const AttnParams &p, int b) {
    const int64_t len = p.seq_lens[b];
    return len < 0 ? 0 : len > p.capacity ? p.capacity : len;
}

// Every instance takes the full staging ring (TcCfg<D, NR, false>): one CTA
// per SM streams one long run.
template <int D, int NR>
using TcpCfg = TcCfg<D, NR, false>;

template <int D, int NR>
__global__ void __launch_bounds__(tc_threads(D, NR), 1)
    attn_tcp_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const AttnParams p) {
    using C = TcpCfg<D, NR>;
    static_assert(!C::SV, "half-tile V staging has no persistent form");
    constexpr int TK = C::TK;
    constexpr int HR = C::HR;
    constexpr int NSW = C::NSW;
    constexpr int NPB = C::NPB;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gb = smem_raw + (sbase - raw);
    const uint32_t sQ = sbase + C::Q_OFF;
    const uint32_t sPT = sbase + C::PT_OFF;
    float *red = reinterpret_cast<float *>(gb + C::RED_OFF);                   // [4][NR]
    volatile int *flags = reinterpret_cast<volatile int *>(gb + C::FLAG_OFF);  // [0] abort, [8 + 16*buf + w] votes
    const uint32_t bars = sbase + C::BAR_OFF;
    const uint32_t bar_full0 = bars;                          // [NSLOT]
    const uint32_t bar_empty0 = bars + 8 * C::NSLOT;          // [NSLOT]
    const uint32_t bar_sfull = bars + 16 * C::NSLOT;          // [2]
    const uint32_t bar_sfree = bar_sfull + 16;                // [2]
    const uint32_t bar_pfull = bar_sfree + 16;                // [2]
    const uint32_t bar_odone = bar_pfull + 16;                // [2]
    const uint32_t bar_qfull = bar_odone + 16;                // phase k: queries of segment k written
    const uint32_t bar_final = bar_qfull + 8;
    uint32_t *tptr = reinterpret_cast<uint32_t *>(gb + C::TPTR_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(bar_full0 + 8 * s, 1);
            mbar_init(bar_empty0 + 8 * s, 1);
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

    pdl_wait();  // the schedule and every input may come from earlier kernels
    pdl_launch_dependents();
    const int4 start = p.cta_start[blockIdx.x];
    const int n_all = start.w;  // tiles of this CTA's run
    if (n_all <= 0) {
        if (warp == 1) tc::tmem_dealloc(tmem, C::TMEM_COLS);
        return;
    }

    if (warp == 0) {
        // ============================================================ TMA producer
        // Per segment the whole warp copies the segment's first block-table
        // entries into shared memory (lane 0 has issued every copy of the
        // previous segment by then, and the copies hold no reference to the
        // cache); lane 0 then issues K_t and V_t of each tile, stepping the
        // page and row of each 64-row box without a division.
        int32_t *page_cache = reinterpret_cast<int32_t *>(gb + C::BT_OFF);
        if (lane == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        const uint64_t policy = l2_policy_evict_first();
        TcpWalk walk;
        walk.init(start);
        int sb = 0, skvh = 0, t0 = 0, n = 0;
        int g = 0;       // tiles of the run before this segment
        int issued = 0;  // units (K or V tiles) issued, lane 0
        bool stop = false;
        while (!stop && walk.next(p, sb, skvh, t0, n)) {
            const int64_t len = tcp_len(p, sb);
            const int64_t k_begin = (int64_t)t0 * TK;
            const int64_t k_end = min(k_begin + (int64_t)n * TK, len);
            const int64_t first_page = p.source == KEYS_PAGED ? k_begin / p.page_size : 0;
            if (p.source == KEYS_PAGED) {
                __syncwarp();
                const int64_t n_pages_seg = (k_end - 1) / p.page_size - first_page + 1;
                for (int i = lane; i < kTcPageCache && i < n_pages_seg; i += 32) {
                    int32_t page = p.block_table[(int64_t)sb * p.max_pages + first_page + i];
                    if (page < 0 || page >= p.n_pages) {
                        tc_report(p.err, WM_DEVERR_BAD_PAGE);
                        page = 0;
                    }
                    page_cache[i] = page;
                }
                __syncwarp();
            }
            if (lane == 0) {
                int32_t last_page = 0;
                int64_t next_local = 0;
                int next_row = (int)(k_begin - first_page * p.page_size);
                int box_page[2] = {0, 0}, box_row[2] = {0, 0};
                for (int ul = 0; ul < 2 * n; ++ul) {
                    const int u = 2 * g + ul;  // unit of the run: K of tile u/2, then its V
                    if (u == p.stall_tile) {   // tests of the timeout path only
                        stop = true;
                        break;
                    }
                    const int s = u % C::NSLOT;
                    if (u >= C::NSLOT &&
                        !mbar_wait_bounded(bar_empty0 + 8 * s, ((u / C::NSLOT) & 1) ^ 1, p.wait_limit)) {
                        tc_report(p.err, WM_DEVERR_TIMEOUT);
                        flags[0] = 1;
                        stop = true;
                        break;
                    }
                    if (flags[0]) {
                        stop = true;
                        break;
                    }
                    const int t = ul >> 1;
                    const CUtensorMap *map = (ul & 1) ? &tmv : &tmk;
                    const uint32_t dst = sbase + s * C::SLOT_BYTES;
                    const int64_t key0 = k_begin + (int64_t)t * TK;
                    if (p.source == KEYS_PAGED && (ul & 1) == 0) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (h * p.box_rows >= TK) break;
                            if (key0 + (int64_t)h * p.box_rows < k_end) {
                                int32_t page;
                                if (next_local < kTcPageCache) {
                                    page = page_cache[next_local];
                                } else {
                                    page = p.block_table[(int64_t)sb * p.max_pages + first_page + next_local];
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
                    bool bad = false;
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
                            c_outer = sb;
                        }
                        if (!in_smem(dst + (C::NCH - 1) * C::REGION + h * p.box_rows * 128, p.box_rows * 128,
                                     sbase, sbase + C::NSLOT * C::SLOT_BYTES) ||
                            c_row < 0 || c_outer < 0) {
                            tc_report(p.err, WM_DEVERR_INTERNAL);
                            flags[0] = 1;
                            bad = true;
                            break;
                        }
#pragma unroll
                        for (int c = 0; c < C::NCH; ++c)
                            tma_load_4d(dst + c * C::REGION + h * p.box_rows * 128, map, bar_full0 + 8 * s, c * 64,
                                        c_row, skvh, c_outer, policy);
                    }
                    issued = u + 1;
                    if (bad) {
                        stop = true;
                        break;
                    }
                }
            }
            stop = __shfl_sync(0xffffffffu, stop, 0);
            g += n;
        }
        // Never leave the CTA with bulk copies still landing in its shared memory.
        if (lane == 0)
            for (int u = max(0, issued - C::NSLOT); u < issued; ++u)
                mbar_wait_bounded(bar_full0 + 8 * (u % C::NSLOT), (u / C::NSLOT) & 1, p.wait_limit);
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_s = tc::idesc_bf16(128, NR, 0, 0);
            constexpr uint32_t id_pv = tc::idesc_bf16(128, NR, 1, 1);
            // Two walkers: one for the S products (tile ts), one for the P.V
            // products (tile tp <= ts), each knowing where its segment ends.
            TcpWalk walk_s, walk_p;
            walk_s.init(start);
            walk_p.init(start);
            int xb, xh, xt, xn;
            int ks = 0;                                  // segment of tile ts
            int ts_end = walk_s.next(p, xb, xh, xt, xn) ? xn : n_all;
            int tp_first = 0;                            // first tile of tp's segment
            int tp_end = walk_p.next(p, xb, xh, xt, xn) ? xn : n_all;
            bool q_ready = false;                        // queries of segment ks written
            bool ok = true;
            int ts = 0, tp = 0;
            uint32_t idle = 0;
            while (ok && tp < n_all) {
                if (flags[0]) break;
                bool did = false;
                if (ts < n_all) {
                    if (ts == ts_end) {  // the next segment: wait for its queries
                        ts_end = ts + (walk_s.next(p, xb, xh, xt, xn) ? xn : n_all);
                        ++ks;
                        q_ready = false;
                    }
                    if (!q_ready) q_ready = mbar_test(bar_qfull, ks & 1);
                    const int uk = 2 * ts, sk = uk % C::NSLOT;
                    // (see attn_tc_kernel: test a slot only once the consumer of its
                    // previous unit has been issued)
                    const int prev = uk - C::NSLOT;
                    const bool prev_in = prev < 0 || ((prev & 1) ? (prev >> 1) < tp : (prev >> 1) < ts);
                    if (q_ready && prev_in && mbar_test(bar_full0 + 8 * sk, (uk / C::NSLOT) & 1) &&
                        (ts < 2 || mbar_test(bar_sfree + 8 * (ts & 1), ((ts - 2) >> 1) & 1))) {
                        tc::fence_after_sync();
                        const uint32_t d_s = tmem + C::S_COL + (ts & 1) * NR;
                        const uint32_t a_k = sbase + sk * C::SLOT_BYTES;
                        if (!in_smem(a_k, C::SLOT_BYTES, sbase, sbase + C::NSLOT * C::SLOT_BYTES)) {
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
                if (tp < ts) {
                    if (tp == tp_end) {
                        tp_first = tp;
                        tp_end = tp + (walk_p.next(p, xb, xh, xt, xn) ? xn : n_all);
                    }
                    const int uv = 2 * tp + 1, sv = uv % C::NSLOT;
                    const int prev = uv - C::NSLOT;
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
                        const bool seg_first = tp == tp_first;
#pragma unroll
                        for (int kk = 0; kk < TK / 16; ++kk) {
                            const uint32_t first = (seg_first && kk == 0) ? 0u : 1u;
                            const uint32_t koff = kk * 2 * C::PT_ATOM;
                            const uint64_t b_hi = tc::smem_desc(pt + koff, C::PT_BYTES, C::PT_ATOM, C::PT_SWIZZLE);
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
        // ============================================================ softmax warps
        const int sw = warp - 2;                       // 0..NSW-1
        const int q4 = warp & 3;                       // tensor-memory lane quadrant
        const int r0 = (sw >> 2) * HR;                 // first row of this warp's group
        const int kt = 32 * q4 + lane;                 // key within the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const int ct = threadIdx.x - 64;               // 0..32*NSW-1
        const int live_chunks = min(HR / 8, max(0, (p.rows - r0 + 7) / 8));
        const float kLn2 = 0.693147180559945309f;

        // queries of unit (b, kvh) into the query buffer, then this warp's arrival
        auto stage_q = [&](int b, int kvh) {
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
        };

        TcpWalk walk;
        walk.init(start);
        int b = 0, kvh = 0, t0 = 0, n = 0;
        bool have_seg = walk.next(p, b, kvh, t0, n);
        if (have_seg) stage_q(b, kvh);
        int g = 0;  // tiles of the run before this segment
        while (have_seg) {
            const int64_t len = tcp_len(p, b);
            const int64_t k_begin = (int64_t)t0 * TK;
            const int64_t k_end = min(k_begin + (int64_t)n * TK, len);
            const int64_t qpos0 = len - p.n_q;
            int nb = 0, nkvh = 0, nt0 = 0, nn = 0;
            const bool have_next = walk.next(p, nb, nkvh, nt0, nn);

            float m_run[HR], l_run[HR];
#pragma unroll
            for (int i = 0; i < HR; ++i) {
                m_run[i] = kMaxFloor;
                l_run[i] = 0.f;
            }
            for (int t = 0; t < n; ++t) {
                const int gt = g + t;  // tile of the run: indexes every buffer and barrier phase
                const int64_t key0 = k_begin + (int64_t)t * TK;
                const int64_t kabs = key0 + kt;
                const bool key_ok = kabs < k_end;
                float s[HR];
                bool live = !warp_aborted(flags);
                if (live && !mbar_wait_bounded(bar_sfull + 8 * (gt & 1), (gt >> 1) & 1, p.wait_limit)) {
                    tc_report(p.err, WM_DEVERR_TIMEOUT);
                    flags[0] = 1;
                }
                live = !warp_aborted(flags);
                tc::fence_after_sync();
#pragma unroll
                for (int i = 0; i < HR; ++i) s[i] = -CUDART_INF_F;
                if (live) {
#pragma unroll
                    for (int c = 0; c < HR / 8; ++c)
                        if (c < live_chunks)
                            tc::ld_32x32b_x8(tmem + lane_off + C::S_COL + (gt & 1) * NR + r0 + 8 * c, s + 8 * c);
                    tc::wait_ld();
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sfree + 8 * (gt & 1));
                // The last S of the segment has been read: every S product that
                // reads the current queries has completed, so the next
                // segment's queries can take their place.
                if (t == n - 1 && have_next) stage_q(nb, nkvh);

                const bool causal_tile = key0 + TK - 1 > qpos0;
                const bool key_tile = key0 + TK > k_end;
                const int64_t rel = qpos0 - kabs;  // key visible to row r iff rel + r / group >= 0
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
                } else {
                    f = p.scale_log2;
#pragma unroll
                    for (int c = 0; c < HR / 8; ++c)
                        if (c < live_chunks) {
#pragma unroll
                            for (int i = 8 * c; i < 8 * c + 8; ++i) need |= fmaf(s[i], f, -m_run[i]) > kLazyRescale;
                        }
                }
                const unsigned any = __ballot_sync(0xffffffffu, need);
                if (lane == 0) flags[8 + 16 * (gt & 1) + sw] = any != 0u;
                named_bar_sync(1, 32 * NSW);
                int votes = 0;
#pragma unroll
                for (int w = 0; w < NSW; ++w) votes |= flags[8 + 16 * (gt & 1) + w];
                const bool rescale = votes != 0;
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
                // P_{gt-1}.V_{gt-1} known complete: at a segment's first tile the
                // previous segment's epilogue waited for it
                bool o_stable = t == 0;
                if (rescale) {
                    float alpha[HR];
#pragma unroll
                    for (int i = 0; i < HR; ++i) {
                        const int r = r0 + i;
                        const float m_new = fmaxf(
                            m_run[i], fmaxf(fmaxf(red[r], red[NR + r]), fmaxf(red[2 * NR + r], red[3 * NR + r])));
                        alpha[i] = ex2(m_run[i] - m_new);
                        m_run[i] = m_new;
                        l_run[i] *= alpha[i];
                    }
                    if (t > 0) {
                        // O holds this segment's tiles so far at the old maximum
                        if (!flags[0] &&
                            !mbar_wait_bounded(bar_odone + 8 * ((gt - 1) & 1), ((gt - 1) >> 1) & 1, p.wait_limit)) {
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

                uint32_t hi_w[HR / 2], lo_w[HR / 2];
#pragma unroll
                for (int i = 0; i < HR; i += 2) {
                    if (i >= 8 * live_chunks) {
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
                // the P^T buffer of this tile was last read by P_{gt-NPB}.V_{gt-NPB}
                if (gt >= NPB && !(NPB == 1 && o_stable) && !flags[0] &&
                    !mbar_wait_bounded(bar_odone + 8 * ((gt - NPB) & 1), ((gt - NPB) >> 1) & 1, p.wait_limit)) {
                    tc_report(p.err, WM_DEVERR_TIMEOUT);
                    flags[0] = 1;
                }
                const uint32_t pt = sPT + (gt % NPB) * 2 * C::PT_BYTES;
#pragma unroll
                for (int j = 0; j < HR / 8; ++j) {
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
                    // A key past the segment's end: zero its V row once the V tile
                    // has landed (see attn_tc_kernel for why P_{gt-1}.V_{gt-1} first)
                    const int uv = 2 * gt + 1, sv = uv % C::NSLOT;
                    const bool prev_in =
                        gt == 0 || mbar_wait_bounded(bar_odone + 8 * ((gt - 1) & 1), ((gt - 1) >> 1) & 1, p.wait_limit);
                    if (prev_in && mbar_wait_bounded(bar_full0 + 8 * sv, (uv / C::NSLOT) & 1, p.wait_limit)) {
                        const uint32_t vrow = sbase + sv * C::SLOT_BYTES;
#pragma unroll
                        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                st_shared_v4(vrow + c * C::REGION + swz128(kt, j), make_uint4(0u, 0u, 0u, 0u));
                    } else {
                        tc_report(p.err, WM_DEVERR_TIMEOUT);
                        flags[0] = 1;
                    }
                }
                fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_pfull + 8 * (gt & 1));
            }

            // ---- segment epilogue: this thread owns tensor-memory lane 32*q4 + lane of every O block
            const int g_last = g + n - 1;
            if (!flags[0] &&
                !mbar_wait_bounded(bar_odone + 8 * (g_last & 1), (g_last >> 1) & 1, p.wait_limit)) {
                tc_report(p.err, WM_DEVERR_TIMEOUT);
                flags[0] = 1;
            }
            tc::fence_after_sync();
            const bool have = !warp_aborted(flags);
            named_bar_sync(1, 32 * NSW);
#pragma unroll
            for (int i = 0; i < HR; ++i) {
                float l = l_run[i];
#pragma unroll
                for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                if (lane == 0) red[NR * q4 + r0 + i] = l;
            }
            named_bar_sync(1, 32 * NSW);
            const int64_t seg = (int64_t)blockIdx.x + (int64_t)b * p.n_kv_heads + kvh;  // partial slot c + u
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
                        p.o_part[(seg * p.rows + r) * D + d] = lt > 0.f ? o8[i] / lt : 0.f;
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = r0 + 8 * c + i;
                    if (r >= p.rows || kt != r) continue;
                    const float lt = l8[i];
                    p.lse_part[seg * p.rows + r] = lt > 0.f ? (m_run[8 * c + i] + lg2(lt)) * kLn2 : -CUDART_INF_F;
                }
            }
            // the O loads above are complete (wait_ld) before this warp's next
            // pfull arrival, which gates the next segment's first P.V
            tc::fence_before_sync();
            g += n;
            have_seg = have_next;
            b = nb;
            kvh = nkvh;
            t0 = nt0;
            n = nn;
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
cudaError_t tcp_configure() {
    constexpr int smem = TcpCfg<D, NR>::TOTAL;
    return cudaFuncSetAttribute(attn_tcp_kernel<D, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int D, int NR>
cudaError_t launch_attn_tcp_nr(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p, int n_cta,
                               cudaStream_t stream) {
    constexpr int smem = TcpCfg<D, NR>::TOTAL;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = tcp_configure<D, NR>();
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    return launch_pdl(attn_tcp_kernel<D, NR>, dim3(n_cta), dim3(TcpCfg<D, NR>::THREADS), smem, stream, k, v, p);
}

template <int D, int NR>
int tcp_blocks_per_sm_nr() {
    constexpr int smem = TcpCfg<D, NR>::TOTAL;
    if (tcp_configure<D, NR>() != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_tcp_kernel<D, NR>, TcpCfg<D, NR>::THREADS, smem) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace wm

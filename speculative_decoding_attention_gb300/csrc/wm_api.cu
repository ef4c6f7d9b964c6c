// wm_api.cu -- the C ABI: argument validation, split planning, TMA descriptor
// encoding and kernel launches.  Declarations and contracts: include/wm_api.h.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>

#include "wm_internal.h"
#include "../../include/wm_api.h"

namespace wm {
namespace {

__device__ int32_t g_device_error;  // first device-side data error (WM_DEVERR_*)

// Pipeline-wait settings of the attention launches made by this host thread
// (wm_set_test_stall): the default poll limit and no stall, except in tests of
// the timeout path.
thread_local uint32_t t_wait_limit = kWaitLimit;
thread_local int32_t t_stall_tile = -1;
// Arithmetic of the keys-as-M draft kernel for this host thread's calls
// (wm_set_draft_math): tensor cores (default) or CUDA cores.
thread_local int32_t t_draft_math = WM_DRAFT_MATH_MMA;

constexpr int kMaxDevices = 64;
constexpr int kMaxRows = 64;  // query rows per KV head (4 m-tiles of 16)
constexpr int64_t kMaxUnits = 65535;  // (sequence, KV head) pairs: the launch grid's y extent

int32_t *device_error_ptr() {
    static int32_t *ptrs[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int32_t *>(p);
    }
    return ptrs[dev];
}

int sm_count() {
    static int counts[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (!counts[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev] = n;
    }
    return counts[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Encoded tensor maps of recent calls.  A map is a pure function of the
// base address and the view's shape (it owns nothing), so a decode loop that
// calls with the same buffers every step reuses the encoding.
struct MapCacheEntry {
    bool used = false;
    const void *base = nullptr;
    int head_dim = 0, heads = 0, box_rows = 0;
    int64_t inner = 0, outer = 0;
    CUtensorMap map;
};
constexpr int kMapCacheSize = 64;

// A 4-d view [outer][heads][inner][D] of bf16 rows, read in boxes of
// 64 columns x box_rows rows with the 128-byte swizzle.
bool encode_kv_map(CUtensorMap *map, const void *base, int head_dim, int64_t inner, int heads, int64_t outer,
                   int box_rows) {
    static MapCacheEntry cache[kMapCacheSize];
    static std::mutex mu;
    uint64_t h = reinterpret_cast<uintptr_t>(base) >> 4;
    for (const uint64_t x : {(uint64_t)head_dim, (uint64_t)inner, (uint64_t)heads, (uint64_t)outer,
                             (uint64_t)box_rows})
        h = (h ^ x) * 0x100000001b3ull;
    MapCacheEntry &slot = cache[(h ^ (h >> 29)) % kMapCacheSize];
    {
        std::lock_guard<std::mutex> lock(mu);
        if (slot.used && slot.base == base && slot.head_dim == head_dim && slot.inner == inner &&
            slot.heads == heads && slot.outer == outer && slot.box_rows == box_rows) {
            *map = slot.map;
            return true;
        }
    }
    auto encode = tensor_map_encoder();
    if (!encode) return false;
    const cuuint64_t row = (cuuint64_t)head_dim * 2;
    cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)inner, (cuuint64_t)heads, (cuuint64_t)outer};
    cuuint64_t strides[3] = {row, row * (cuuint64_t)inner, row * (cuuint64_t)inner * (cuuint64_t)heads};
    cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
    cuuint32_t elem[4] = {1, 1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                              strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lock(mu);
    slot.used = true;
    slot.base = base;
    slot.head_dim = head_dim;
    slot.inner = inner;
    slot.heads = heads;
    slot.outer = outer;
    slot.box_rows = box_rows;
    slot.map = *map;
    return true;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

struct SplitPlan {
    int n_split = 0;
    int keys_per_split = 0;  // uniform splits: keys per split (the last one may be shorter)
    int plan_tiles = 0;      // balanced splits (keys-as-M draft kernel): tiles shared out as evenly as possible
};

// Which attention kernel serves a call.  Verification at head dim 128/256 runs
// on the tcgen05 kernel (128-key tiles, deep TMA staging, accumulators in
// tensor memory): it streams gigabytes and is HBM-bound.  The draft reads a
// few megabytes once per step; it is latency-bound, and the mma.sync kernel's
// 64-key tiles give twice as many CTAs with a shorter fixed cost per CTA.
bool use_tc_kernel(int op, int head_dim) { return op == WM_OP_VERIFY && head_dim != 64; }
// The draft with at most 8 query rows per KV head (every GQA group up to 8)
// runs on the keys-as-M kernel: the rows are the MMA's N, so no padding rows,
// and each compute warp owns its keys of a tile end to end.
bool use_draft_kernel(int op, int rows) { return op == WM_OP_DRAFT && rows <= kDraftRowsMax; }
int key_tile(int op, int head_dim) { return use_tc_kernel(op, head_dim) ? kTcTile : kKeyTile; }

// K+V bytes per split when a batch may be ragged (see plan_splits).
constexpr int64_t kRaggedSplitBytes = 8ll << 20;

// Resident CTAs per SM of the kernel that serves `op`.  For the draft the
// smaller of the plain and the fused-step instances, so that both split alike.
// At least 1 (also without a device).
int ctas_per_sm(int op, int head_dim, int rows) {
    static std::mutex mu;
    static int cache[kMaxDevices][3][4][2] = {};
    static int draft_cache[kMaxDevices][3][2] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    const int di = head_dim == 64 ? 0 : head_dim == 128 ? 1 : 2;
    const int mt = std::min(4, std::max(1, (rows + 15) / 16));
    const int oi = op == WM_OP_VERIFY ? 1 : 0;
    std::lock_guard<std::mutex> lock(mu);
    if (use_draft_kernel(op, rows)) {
        const bool fma = t_draft_math == WM_DRAFT_MATH_FMA;
        int &nd = draft_cache[dev][di][fma ? 1 : 0];
        if (!nd) {
            auto query = [&](bool step) {
                return di == 0 ? draft_blocks_per_sm_d64(step, fma)
                     : di == 1 ? draft_blocks_per_sm_d128(step, fma) : draft_blocks_per_sm_d256(step, fma);
            };
            nd = std::max(1, std::min(query(false), query(true)));
        }
        return nd;
    }
    int &n = cache[dev][di][mt - 1][oi];
    if (!n && use_tc_kernel(op, head_dim)) {
        n = std::max(1, head_dim == 128 ? attn_tc_blocks_per_sm_d128(16 * mt) : attn_tc_blocks_per_sm_d256(16 * mt));
    } else if (!n) {
        auto query = [&](bool step) {
            return di == 0 ? attn_blocks_per_sm_d64(mt, step)
                 : di == 1 ? attn_blocks_per_sm_d128(mt, step) : attn_blocks_per_sm_d256(mt, step);
        };
        const int plain = query(false);
        n = std::max(1, oi ? plain : std::min(plain, query(true)));
    }
    return n;
}

// Key splits for `units` (sequence, KV head) pairs over up to max_keys keys,
// never a split smaller than a tile.  By default: one wave of the kernel's
// resident CTAs (per_sm per SM).
// With several sequences the lengths may differ (only their maximum is known
// on the host), so splits are also capped at about kRaggedSplitBytes of K+V:
// short sequences then leave most of their splits empty (those CTAs exit at
// once) and the block scheduler balances the rest.  When the cap asks for
// more than one wave, the count is raised to fill the last wave (the most
// splits that still take that many waves): with equal lengths a partly empty
// last wave would leave SMs idle for a whole split's time.
// Balanced (the keys-as-M draft kernel): with tiles = q n + r, the first r
// splits take q + 1 tiles and the others q, so any split count up
// to the tile count is used as planned -- uniform splits
// of whole tiles can only realise the counts that divide the tiles evenly,
// which left a third of the SMs with one CTA less than the others.
SplitPlan plan_splits(int units, int batch, int64_t max_keys, int requested, int tile, int head_dim, int per_sm,
                      bool balanced = false) {
    SplitPlan pl;
    const int64_t tiles = std::max<int64_t>(1, (max_keys + tile - 1) / tile);
    int64_t ns = requested;
    if (ns <= 0) {
        const int sms = sm_count();
        const int64_t wave = (int64_t)per_sm * (sms > 0 ? sms : 1);
        const int64_t n_units = std::max(1, units);
        ns = std::max<int64_t>(1, wave / n_units);
        if (batch > 1) {
            const int64_t keys_cap = std::max<int64_t>(tile, kRaggedSplitBytes / (4 * head_dim) / tile * tile);
            const int64_t ns_cap = (max_keys + keys_cap - 1) / keys_cap;
            if (ns_cap > ns) {
                const int64_t waves = (n_units * ns_cap + wave - 1) / wave;
                ns = std::max(ns_cap, waves * wave / n_units);
            }
        }
    }
    ns = std::min<int64_t>(ns, tiles);
    const int64_t tps = (tiles + ns - 1) / ns;
    if (balanced) {
        pl.n_split = (int)ns;
        pl.plan_tiles = (int)std::min<int64_t>(tiles, INT32_MAX);
        pl.keys_per_split = (int)((tiles + ns - 1) / ns * tile);
        return pl;
    }
    pl.n_split = (int)((tiles + tps - 1) / tps);
    pl.keys_per_split = (int)(tps * tile);
    return pl;
}

size_t partial_bytes(int64_t rows_total, int n_split, int head_dim) {
    const size_t o = (size_t)rows_total * n_split * head_dim * sizeof(float);
    const size_t o_aligned = (o + 255) & ~(size_t)255;
    return o_aligned + (size_t)rows_total * n_split * sizeof(float);
}

// The persistent verify (attn_tcp.cuh) serves a batch of several sequences on
// the tcgen05 kernel when the caller leaves the split count to the library:
// it reads the actual lengths on the device and gives every resident CTA the
// same number of key tiles.  Returns its CTA count, or 0 when the call runs
// the split plan instead (one sequence, an explicit n_split, a configuration
// with half-tile V staging, or more than 2^30 key tiles per call, which keeps
// every tile count of the schedule within 32 bits).
int tcp_ctas(int op, int batch, int n_kv_heads, int rows, int head_dim, int64_t max_keys, int n_split) {
    const int nr = 16 * ((rows + 15) / 16);
    if (op != WM_OP_VERIFY || !use_tc_kernel(op, head_dim) || batch <= 1 || n_split != 0 ||
        !tcp_supported(head_dim, nr))
        return 0;
    const int64_t tiles = (max_keys + kTcTile - 1) / kTcTile;
    if ((int64_t)batch * n_kv_heads * tiles > (int64_t)1 << 30) return 0;
    static std::mutex mu;
    static int cache[kMaxDevices][2][4] = {};
    int dev = 0;
    int per_sm = 1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(mu);
        int &n = cache[dev][head_dim == 128 ? 0 : 1][nr / 16 - 1];
        if (!n) n = std::max(1, head_dim == 128 ? attn_tcp_blocks_per_sm_d128(nr) : attn_tcp_blocks_per_sm_d256(nr));
        per_sm = n;
    }
    const int sms = sm_count();
    return per_sm * (sms > 0 ? sms : 1);
}

// Workspace of the persistent verify: segment partials (n_cta + units - 1
// segments of `rows` rows), the schedule (chunk, total, tile prefix) and the
// CTAs' first tiles, each part 256-byte aligned.
struct TcpLayout {
    size_t o = 0, lse = 0, sched = 0, start = 0, total = 0;
};
TcpLayout tcp_layout(int n_cta, int64_t units, int rows, int head_dim, int batch) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t n_seg = (size_t)n_cta + (size_t)units - 1;
    TcpLayout l;
    l.o = 0;
    l.lse = up(n_seg * rows * head_dim * sizeof(float));
    l.sched = l.lse + up(n_seg * rows * sizeof(float));
    l.start = l.sched + up(((size_t)batch + 3) * sizeof(int64_t));
    l.total = l.start + (size_t)n_cta * sizeof(int4);
    return l;
}

// maps: K and V of the cache or ring, then K and V of the memory-slot store
// (the same two again when there is none).
cudaError_t launch_attn_any(int op, const CUtensorMap (&maps)[4], const AttnParams &p, bool step,
                            cudaStream_t st) {
    const int m_tiles = (p.rows + 15) / 16;
    if (use_draft_kernel(op, p.rows)) {
        const bool fma = t_draft_math == WM_DRAFT_MATH_FMA;
        switch (p.head_dim) {
            case 64: return launch_draft_d64(maps[0], maps[1], maps[2], maps[3], p, step, fma, st);
            case 128: return launch_draft_d128(maps[0], maps[1], maps[2], maps[3], p, step, fma, st);
            case 256: return launch_draft_d256(maps[0], maps[1], maps[2], maps[3], p, step, fma, st);
            default: return cudaErrorInvalidValue;
        }
    }
    if (!step && use_tc_kernel(op, p.head_dim)) {
        return p.head_dim == 128 ? launch_attn_tc_d128(maps[0], maps[1], p, 16 * m_tiles, st)
                                 : launch_attn_tc_d256(maps[0], maps[1], p, 16 * m_tiles, st);
    }
    switch (p.head_dim) {
        case 64:
            return step ? launch_step_d64(maps[0], maps[1], maps[2], maps[3], p, m_tiles, st)
                        : launch_attn_d64(maps[0], maps[1], maps[2], maps[3], p, m_tiles, st);
        case 128:
            return step ? launch_step_d128(maps[0], maps[1], maps[2], maps[3], p, m_tiles, st)
                        : launch_attn_d128(maps[0], maps[1], maps[2], maps[3], p, m_tiles, st);
        case 256:
            return step ? launch_step_d256(maps[0], maps[1], maps[2], maps[3], p, m_tiles, st)
                        : launch_attn_d256(maps[0], maps[1], maps[2], maps[3], p, m_tiles, st);
        default: return cudaErrorInvalidValue;
    }
}

bool ring_ok(const wm_ring *r) {
    return r && r->k && r->v && r->pos_tag && r->n_seen && r->batch > 0 && r->n_kv_heads > 0 &&
           head_dim_ok(r->head_dim) && r->sink >= 0 && r->window >= 1 &&
           (int64_t)r->sink + r->window <= INT32_MAX / 2 && aligned(r->k, 16) && aligned(r->v, 16) &&
           aligned(r->pos_tag, 4) && aligned(r->n_seen, 8);
}

// Shape checks of a contiguous or paged store; `need_tile_pages` enforces the
// attention kernel's page rule (whole key tiles per page).
wm_status kv_check(const wm_kv *kv, bool need_tile_pages) {
    if (!kv || !kv->k || !kv->v || !kv->seq_lens || kv->batch <= 0 || kv->n_kv_heads <= 0)
        return WM_ERR_INVALID_ARG;
    if (!head_dim_ok(kv->head_dim)) return WM_ERR_UNSUPPORTED;
    if (!aligned(kv->k, 16) || !aligned(kv->v, 16) || !aligned(kv->seq_lens, 8)) return WM_ERR_INVALID_ARG;
    if (kv->block_table) {
        if (kv->page_size <= 0 || kv->max_pages <= 0 || kv->n_pages <= 0 || !aligned(kv->block_table, 4))
            return WM_ERR_INVALID_ARG;
        if (need_tile_pages && kv->page_size % kKeyTile) return WM_ERR_UNSUPPORTED;  // whole 64-key boxes
        if (kv->n_pages > INT32_MAX) return WM_ERR_UNSUPPORTED;
        // split lengths are 32-bit: a sequence holds at most INT32_MAX positions
        if ((int64_t)kv->max_pages * kv->page_size > INT32_MAX) return WM_ERR_UNSUPPORTED;
    } else if (kv->n_cap <= 0 || kv->n_cap > INT32_MAX) {
        return kv->n_cap <= 0 ? WM_ERR_INVALID_ARG : WM_ERR_UNSUPPORTED;
    }
    return WM_OK;
}

wm_status launch_status(cudaError_t e) { return e == cudaSuccess ? WM_OK : WM_ERR_CUDA; }

bool mem_ok(const wm_mem *m) {
    return m && m->k && m->v && m->count && m->batch > 0 && m->n_kv_heads > 0 && head_dim_ok(m->head_dim) &&
           m->capacity > 0 && m->capacity <= INT32_MAX / 2 && aligned(m->k, 16) && aligned(m->v, 16) &&
           aligned(m->count, 8);
}

// First key index of the memory region: the ring's slots rounded up to whole
// 64-key tiles, so that every tile is all ring or all memory.
int64_t mem_base_of(const wm_ring *ring) {
    return ((int64_t)ring->sink + ring->window + kKeyTile - 1) / kKeyTile * kKeyTile;
}

}  // namespace
}  // namespace wm

using namespace wm;

extern "C" {

const char *wm_status_string(wm_status s) {
    switch (s) {
        case WM_OK: return "ok";
        case WM_ERR_INVALID_ARG: return "invalid argument";
        case WM_ERR_UNSUPPORTED: return "unsupported shape or layout";
        case WM_ERR_WORKSPACE: return "workspace missing or too small";
        case WM_ERR_CUDA: return "CUDA error";
        case WM_ERR_DEVICE_DATA: return "bad device-side data";
    }
    return "unknown status";
}

int32_t wm_version(void) { return 100; }

wm_status wm_set_draft_math(int32_t math) {
    if (math != WM_DRAFT_MATH_MMA && math != WM_DRAFT_MATH_FMA) return WM_ERR_INVALID_ARG;
    t_draft_math = math;
    return WM_OK;
}

wm_status wm_set_test_stall(int32_t stall_tile, uint32_t wait_polls) {
    if (stall_tile < -1 || (stall_tile >= 0 && wait_polls == 0)) return WM_ERR_INVALID_ARG;
    t_stall_tile = stall_tile;
    t_wait_limit = stall_tile < 0 ? kWaitLimit : wait_polls;
    return WM_OK;
}

int32_t wm_plan_splits(int32_t op, int32_t batch, int32_t n_kv_heads, int32_t n_q_heads, int32_t n_q,
                       int32_t head_dim, int64_t max_keys, int32_t n_split) {
    if ((op != WM_OP_DRAFT && op != WM_OP_VERIFY && op != WM_OP_DRAFT_STEP && op != WM_OP_DRAFT_MEM) || batch <= 0 ||
        n_kv_heads <= 0 ||
        n_q_heads <= 0 || n_q <= 0 || !head_dim_ok(head_dim) || max_keys < 0 || n_split < 0)
        return 0;
    if (op == WM_OP_DRAFT_STEP || op == WM_OP_DRAFT_MEM) {
        if (n_q != 1) return 0;
        op = WM_OP_DRAFT;  // all draft forms split alike
    }
    const int rows = n_q * (n_q_heads / n_kv_heads);
    const int n_cta = tcp_ctas(op, batch, n_kv_heads, rows, head_dim, max_keys, n_split);
    if (n_cta > 0) return n_cta;
    return plan_splits(batch * n_kv_heads, batch, max_keys, n_split, key_tile(op, head_dim), head_dim,
                       ctas_per_sm(op, head_dim, rows), use_draft_kernel(op, rows))
        .n_split;
}

int32_t wm_verify_persistent(int32_t batch, int32_t n_kv_heads, int32_t n_q_heads, int32_t n_q, int32_t head_dim,
                             int64_t max_keys, int32_t n_split) {
    if (batch <= 0 || n_kv_heads <= 0 || n_q_heads <= 0 || n_q <= 0 || n_q_heads % n_kv_heads ||
        !head_dim_ok(head_dim) || max_keys < 0 || n_split < 0)
        return 0;
    return tcp_ctas(WM_OP_VERIFY, batch, n_kv_heads, n_q * (n_q_heads / n_kv_heads), head_dim, max_keys, n_split);
}

size_t wm_workspace_size(int32_t op, int32_t batch, int32_t n_kv_heads, int32_t n_q_heads, int32_t n_q,
                         int32_t head_dim, int64_t max_keys, int32_t n_split) {
    const int32_t ns = wm_plan_splits(op, batch, n_kv_heads, n_q_heads, n_q, head_dim, max_keys, n_split);
    if (ns <= 0) return (size_t)-1;
    if (n_q_heads % n_kv_heads == 0) {
        const int rows = n_q * (n_q_heads / n_kv_heads);
        const int n_cta = tcp_ctas(op, batch, n_kv_heads, rows, head_dim, max_keys, n_split);
        if (n_cta > 0) return tcp_layout(n_cta, (int64_t)batch * n_kv_heads, rows, head_dim, batch).total;
    }
    if (op == WM_OP_DRAFT_STEP || op == WM_OP_DRAFT_MEM)  // partials even when unsplit (fused step)
        return partial_bytes((int64_t)batch * n_q_heads, ns, head_dim);
    if (ns == 1) return 0;
    return partial_bytes((int64_t)batch * n_q * n_q_heads, ns, head_dim);
}

wm_status wm_get_device_error(int32_t *code, void *stream) {
    if (!code) return WM_ERR_INVALID_ARG;
    int32_t *p = device_error_ptr();
    if (!p) return WM_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return WM_ERR_CUDA;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return WM_ERR_CUDA;
    const int32_t zero = 0;
    if (v != 0 && cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return WM_ERR_CUDA;
    *code = v;
    return v == WM_DEVERR_NONE ? WM_OK : WM_ERR_DEVICE_DATA;
}

wm_status wm_ring_append(const wm_ring *ring, const void *k_new, const void *v_new, void *stream) {
    if (!ring_ok(ring) || !k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16))
        return WM_ERR_INVALID_ARG;
    int32_t *err = device_error_ptr();
    if (!err) return WM_ERR_CUDA;
    return launch_status(launch_ring_append(ring->k, ring->v, ring->pos_tag, ring->n_seen, ring->batch,
                                            ring->n_kv_heads, ring->head_dim, ring->sink, ring->window,
                                            k_new, v_new, err, static_cast<cudaStream_t>(stream)));
}

wm_status wm_ring_fill(const wm_ring *ring, const wm_kv *hist, void *stream) {
    if (!ring_ok(ring)) return WM_ERR_INVALID_ARG;
    const wm_status ks = kv_check(hist, false);
    if (ks != WM_OK) return ks;
    if (hist->batch != ring->batch || hist->n_kv_heads != ring->n_kv_heads || hist->head_dim != ring->head_dim)
        return WM_ERR_INVALID_ARG;
    if ((int64_t)ring->batch * ring->n_kv_heads > kMaxUnits) return WM_ERR_UNSUPPORTED;
    int32_t *err = device_error_ptr();
    if (!err) return WM_ERR_CUDA;
    HistSource h;
    h.k = hist->k;
    h.v = hist->v;
    h.lens = hist->seq_lens;
    h.block_table = hist->block_table;
    h.n_cap = hist->n_cap;
    h.n_pages = hist->n_pages;
    h.page_size = hist->page_size;
    h.max_pages = hist->max_pages;
    return launch_status(launch_ring_fill(ring->k, ring->v, ring->pos_tag, ring->n_seen, ring->batch,
                                          ring->n_kv_heads, ring->head_dim, ring->sink, ring->window, h, err,
                                          static_cast<cudaStream_t>(stream)));
}

wm_status wm_ring_rollback(const wm_ring *ring, const int64_t *new_len, void *stream) {
    if (!ring_ok(ring) || !new_len || !aligned(new_len, 8)) return WM_ERR_INVALID_ARG;
    if (ring->batch > kMaxUnits) return WM_ERR_UNSUPPORTED;
    int32_t *err = device_error_ptr();
    if (!err) return WM_ERR_CUDA;
    return launch_status(launch_ring_rollback(ring->pos_tag, ring->n_seen, ring->batch,
                                              ring->sink + ring->window, new_len, err,
                                              static_cast<cudaStream_t>(stream)));
}

wm_status wm_lse_merge(const float *o_parts, const float *lse_parts, int32_t n_parts, int64_t rows,
                       int32_t head_dim, void *out, float *lse_out, void *stream) {
    if (!o_parts || !lse_parts || !out || n_parts <= 0 || rows < 0 || head_dim <= 0 || rows > INT32_MAX)
        return WM_ERR_INVALID_ARG;
    if (!aligned(o_parts, 16) || !aligned(lse_parts, 4) || !aligned(out, 8) || (lse_out && !aligned(lse_out, 4)))
        return WM_ERR_INVALID_ARG;
    if (head_dim % 4) return WM_ERR_UNSUPPORTED;
    return launch_status(launch_lse_merge(o_parts, lse_parts, n_parts, rows, head_dim, out, lse_out, nullptr, 0,
                                          static_cast<cudaStream_t>(stream)));
}

// Shared tail of the attention entry points: plan, check the workspace,
// launch the attention kernel and (if split, or always for the fused step)
// the merge -- which for the fused step also commits n_seen.
// encode_maps fills the four tensor maps; it runs after every host-side check
// (so that a bad argument is reported before any CUDA or driver call).
using MapEncoder = std::function<bool(CUtensorMap (&)[4])>;

static wm_status run_attention(int op, AttnParams &p, const MapEncoder &encode_maps, int64_t max_keys,
                               int32_t n_split, void *out, float *lse, void *ws, size_t ws_bytes, cudaStream_t st,
                               int64_t *commit_n_seen = nullptr) {
    const bool step = commit_n_seen != nullptr;
    if ((int64_t)p.batch * p.n_kv_heads > kMaxUnits) return WM_ERR_UNSUPPORTED;
    const int n_cta = step ? 0 : tcp_ctas(op, p.batch, p.n_kv_heads, p.rows, p.head_dim, max_keys, n_split);
    if (n_cta > 0) {
        // persistent verify: schedule (one CTA), the verify grid, the segment merge
        const TcpLayout l = tcp_layout(n_cta, (int64_t)p.batch * p.n_kv_heads, p.rows, p.head_dim, p.batch);
        if (!ws || ws_bytes < l.total || !aligned(ws, 256)) return WM_ERR_WORKSPACE;
        char *w = static_cast<char *>(ws);
        int64_t *sched = reinterpret_cast<int64_t *>(w + l.sched);
        int4 *cta_start = reinterpret_cast<int4 *>(w + l.start);
        p.n_split = n_cta;
        p.keys_per_split = 0;
        p.out = out;
        p.lse = lse;
        p.o_part = reinterpret_cast<float *>(w + l.o);
        p.lse_part = reinterpret_cast<float *>(w + l.lse);
        p.tile_prefix = sched + 2;
        p.cta_start = cta_start;
        p.err = device_error_ptr();
        if (!p.err) return WM_ERR_CUDA;
        p.wait_limit = t_wait_limit;
        p.stall_tile = t_stall_tile;
        CUtensorMap maps[4];
        if (!encode_maps(maps)) return WM_ERR_CUDA;
        const int nr = 16 * ((p.rows + 15) / 16);
        cudaError_t e = launch_verify_sched(p.seq_lens, p.batch, p.n_kv_heads, p.capacity, n_cta, sched, cta_start,
                                            p.err, st);
        if (e != cudaSuccess) return WM_ERR_CUDA;
        e = p.head_dim == 128 ? launch_attn_tcp_d128(maps[0], maps[1], p, nr, n_cta, st)
                              : launch_attn_tcp_d256(maps[0], maps[1], p, nr, n_cta, st);
        if (e != cudaSuccess) return WM_ERR_CUDA;
        e = launch_seg_merge(p.o_part, p.lse_part, sched, p.batch, p.n_kv_heads, p.n_q, p.n_q_heads, p.head_dim, out,
                             lse, st);
        return e == cudaSuccess ? WM_OK : WM_ERR_CUDA;
    }
    const bool keys_as_m = use_draft_kernel(op, p.rows);
    const SplitPlan pl = plan_splits(p.batch * p.n_kv_heads, p.batch, max_keys, n_split, key_tile(op, p.head_dim),
                                     p.head_dim, ctas_per_sm(op, p.head_dim, p.rows), keys_as_m);
    const int64_t rows_total = (int64_t)p.batch * p.n_q * p.n_q_heads;
    p.n_split = pl.n_split;
    p.keys_per_split = pl.keys_per_split;
    p.plan_tiles = pl.plan_tiles;
    p.out = out;
    p.lse = lse;
    p.o_part = nullptr;
    p.lse_part = nullptr;
    const bool partials = pl.n_split > 1 || step;
    if (partials) {
        const size_t need = partial_bytes(rows_total, pl.n_split, p.head_dim);
        if (!ws || ws_bytes < need || !aligned(ws, 256)) return WM_ERR_WORKSPACE;
        const size_t o = (size_t)rows_total * pl.n_split * p.head_dim * sizeof(float);
        p.o_part = static_cast<float *>(ws);
        p.lse_part = reinterpret_cast<float *>(static_cast<char *>(ws) + ((o + 255) & ~(size_t)255));
    }
    p.err = device_error_ptr();
    if (!p.err) return WM_ERR_CUDA;
    p.wait_limit = t_wait_limit;
    p.stall_tile = t_stall_tile;
    CUtensorMap maps[4];
    if (!encode_maps(maps)) return WM_ERR_CUDA;
    cudaError_t e = launch_attn_any(op, maps, p, step, st);
    if (e != cudaSuccess) return WM_ERR_CUDA;
    if (partials) {
        e = launch_lse_merge(p.o_part, p.lse_part, pl.n_split, rows_total, p.head_dim, out, lse, commit_n_seen,
                             p.n_q * p.n_q_heads, st);
        if (e != cudaSuccess) return WM_ERR_CUDA;
    }
    return WM_OK;
}

// Validation and parameters shared by the draft calls (plain, with memory
// slots, fused with the append).  On success fills p (ring and, if mem, the
// memory region), the tensor-map encoder and the key count to plan over.
static wm_status draft_setup(const wm_ring *ring, const wm_mem *mem, const void *q, int32_t n_q_heads,
                             float scale, int32_t n_split, void *out, float *lse, AttnParams &p,
                             MapEncoder &maps, int64_t &plan_keys) {
    if (!ring_ok(ring) || !q || !out || n_q_heads <= 0 || n_split < 0 || !std::isfinite(scale))
        return WM_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4))) return WM_ERR_INVALID_ARG;
    if (n_q_heads % ring->n_kv_heads) return WM_ERR_INVALID_ARG;
    if (mem && (!mem_ok(mem) || mem->batch != ring->batch || mem->n_kv_heads != ring->n_kv_heads ||
                mem->head_dim != ring->head_dim))
        return WM_ERR_INVALID_ARG;
    const int group = n_q_heads / ring->n_kv_heads;
    if (group > kMaxRows) return WM_ERR_UNSUPPORTED;
    const int n_slots = ring->sink + ring->window;
    maps = [ring, mem, n_slots](CUtensorMap (&m)[4]) {
        if (!encode_kv_map(&m[0], ring->k, ring->head_dim, n_slots, ring->n_kv_heads, ring->batch, kKeyTile) ||
            !encode_kv_map(&m[1], ring->v, ring->head_dim, n_slots, ring->n_kv_heads, ring->batch, kKeyTile))
            return false;
        if (!mem) {
            m[2] = m[0];
            m[3] = m[1];
            return true;
        }
        return encode_kv_map(&m[2], mem->k, mem->head_dim, mem->capacity, mem->n_kv_heads, mem->batch, kKeyTile) &&
               encode_kv_map(&m[3], mem->v, mem->head_dim, mem->capacity, mem->n_kv_heads, mem->batch, kKeyTile);
    };
    std::memset(&p, 0, sizeof p);
    p.source = KEYS_RING;
    p.batch = ring->batch;
    p.n_kv_heads = ring->n_kv_heads;
    p.head_dim = ring->head_dim;
    p.pos_tag = ring->pos_tag;
    p.n_seen = ring->n_seen;
    p.n_slots = n_slots;
    p.sink = ring->sink;
    p.window = ring->window;
    p.capacity = n_slots;
    p.box_rows = kKeyTile;
    p.q = q;
    p.n_q = 1;
    p.n_q_heads = n_q_heads;
    p.group = group;
    p.rows = group;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    plan_keys = n_slots;
    if (mem) {
        p.mem_count = mem->count;
        p.mem_cap = mem->capacity;
        p.mem_base = mem_base_of(ring);
        plan_keys = p.mem_base + mem->capacity;
    }
    return WM_OK;
}

}  // extern "C"

namespace wm {

int32_t draft_args_status(const wm_ring *ring, const void *q, int32_t n_q_heads, float scale, int32_t n_split,
                          const void *out, const float *lse) {
    AttnParams p;
    MapEncoder maps;
    int64_t keys = 0;
    return draft_setup(ring, nullptr, q, n_q_heads, scale, n_split, const_cast<void *>(out),
                       const_cast<float *>(lse), p, maps, keys);
}

}  // namespace wm

extern "C" {

wm_status wm_draft_attn(const wm_ring *ring, const void *q, int32_t n_q_heads, float scale, int32_t n_split,
                        void *out, float *lse, void *workspace, size_t workspace_bytes, void *stream) {
    AttnParams p;
    MapEncoder maps;
    int64_t keys = 0;
    const wm_status s = draft_setup(ring, nullptr, q, n_q_heads, scale, n_split, out, lse, p, maps, keys);
    if (s != WM_OK) return s;
    return run_attention(WM_OP_DRAFT, p, maps, keys, n_split, out, lse, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream));
}

wm_status wm_draft_attn_mem(const wm_ring *ring, const wm_mem *mem, const void *q, int32_t n_q_heads, float scale,
                            int32_t n_split, void *out, float *lse, void *workspace, size_t workspace_bytes,
                            void *stream) {
    if (!mem) return WM_ERR_INVALID_ARG;
    AttnParams p;
    MapEncoder maps;
    int64_t keys = 0;
    const wm_status s = draft_setup(ring, mem, q, n_q_heads, scale, n_split, out, lse, p, maps, keys);
    if (s != WM_OK) return s;
    return run_attention(WM_OP_DRAFT, p, maps, keys, n_split, out, lse, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream));
}

wm_status wm_draft_step(const wm_ring *ring, const wm_mem *mem, const void *k_new, const void *v_new,
                        const void *q, int32_t n_q_heads, float scale, int32_t n_split, void *out, float *lse,
                        void *workspace, size_t workspace_bytes, void *stream) {
    if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return WM_ERR_INVALID_ARG;
    AttnParams p;
    MapEncoder maps;
    int64_t keys = 0;
    const wm_status s = draft_setup(ring, mem, q, n_q_heads, scale, n_split, out, lse, p, maps, keys);
    if (s != WM_OK) return s;
    p.k_new = k_new;
    p.v_new = v_new;
    p.ring_k = ring->k;
    p.ring_v = ring->v;
    p.tag_w = ring->pos_tag;
    return run_attention(WM_OP_DRAFT, p, maps, keys, n_split, out, lse, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream), ring->n_seen);
}

wm_status wm_mem_append(const wm_mem *mem, const void *k_new, const void *v_new, void *stream) {
    if (!mem_ok(mem) || !k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)) return WM_ERR_INVALID_ARG;
    int32_t *err = device_error_ptr();
    if (!err) return WM_ERR_CUDA;
    return launch_status(launch_mem_append(mem->k, mem->v, mem->count, mem->capacity, mem->batch, mem->n_kv_heads,
                                           mem->head_dim, k_new, v_new, err, static_cast<cudaStream_t>(stream)));
}

wm_status wm_mem_rollback(const wm_mem *mem, const int64_t *new_count, void *stream) {
    if (!mem_ok(mem) || !new_count || !aligned(new_count, 8)) return WM_ERR_INVALID_ARG;
    int32_t *err = device_error_ptr();
    if (!err) return WM_ERR_CUDA;
    return launch_status(
        launch_mem_rollback(mem->count, mem->batch, new_count, err, static_cast<cudaStream_t>(stream)));
}

wm_status wm_verify_attn(const wm_kv *kv, const void *q, int32_t n_q, int32_t n_q_heads, float scale,
                         int32_t n_split, void *out, float *lse, void *workspace, size_t workspace_bytes,
                         void *stream) {
    const wm_status ks = kv_check(kv, true);
    if (ks != WM_OK) return ks;
    if (!q || !out || n_q <= 0 || n_q_heads <= 0 || n_split < 0 || !std::isfinite(scale))
        return WM_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4))) return WM_ERR_INVALID_ARG;
    if (n_q_heads % kv->n_kv_heads) return WM_ERR_INVALID_ARG;
    const int group = n_q_heads / kv->n_kv_heads;
    if ((int64_t)group * n_q > kMaxRows) return WM_ERR_UNSUPPORTED;
    const bool paged = kv->block_table != nullptr;
    const int64_t capacity = paged ? (int64_t)kv->max_pages * kv->page_size : kv->n_cap;
    const int64_t inner = paged ? kv->page_size : kv->n_cap;
    const int64_t outer = paged ? kv->n_pages : kv->batch;
    const int tile = key_tile(WM_OP_VERIFY, kv->head_dim);
    const int box = paged && kv->page_size % tile ? kKeyTile : tile;  // a box never crosses a page
    // 33-64 rows at head dim 256: the tensor-core kernel stages V in 64-key halves
    const int rows = group * n_q;
    const int vbox = kv->head_dim == 256 && rows > 32 ? kKeyTile : box;
    const MapEncoder maps = [kv, inner, outer, box, vbox](CUtensorMap (&m)[4]) {
        if (!encode_kv_map(&m[0], kv->k, kv->head_dim, inner, kv->n_kv_heads, outer, box) ||
            !encode_kv_map(&m[1], kv->v, kv->head_dim, inner, kv->n_kv_heads, outer, vbox))
            return false;
        m[2] = m[0];
        m[3] = m[1];
        return true;
    };
    AttnParams p;
    std::memset(&p, 0, sizeof p);
    p.source = paged ? KEYS_PAGED : KEYS_CONTIG;
    p.batch = kv->batch;
    p.n_kv_heads = kv->n_kv_heads;
    p.head_dim = kv->head_dim;
    p.seq_lens = kv->seq_lens;
    p.block_table = kv->block_table;
    p.capacity = capacity;
    p.n_pages = kv->n_pages;
    p.page_size = kv->page_size;
    p.max_pages = kv->max_pages;
    p.box_rows = box;
    p.q = q;
    p.n_q = n_q;
    p.n_q_heads = n_q_heads;
    p.group = group;
    p.rows = group * n_q;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    return run_attention(WM_OP_VERIFY, p, maps, capacity, n_split, out, lse, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream));
}

}  // extern "C"

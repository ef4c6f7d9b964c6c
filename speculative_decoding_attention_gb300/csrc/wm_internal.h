// wm_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

struct wm_ring;  // include/wm_api.h

namespace wm {

// Key source of an attention launch.
enum KeySource : int32_t {
    KEYS_CONTIG = 0,  // verify over a contiguous cache [B][Hkv][n_cap][D]
    KEYS_PAGED = 1,   // verify over a paged cache [pages][Hkv][page][D]
    KEYS_RING = 2,    // draft over the ring [B][Hkv][S+W][D] with slot tags
};

// Keys handled per pipeline stage by the attention kernel (all head dims).
constexpr int kKeyTile = 64;
// Shared-memory bytes the mma.sync attention kernel gives to K/V staging
// (stages = this / stage bytes): 4 stages of 64 keys at head_dim 64 and 128 --
// small enough for two CTAs per SM, whose independent tile loops overlap --
// and the two stages head_dim 256 needs at one CTA per SM.
constexpr int staging_bytes(int head_dim) { return head_dim == 256 ? 128 * 1024 : 64 * 1024; }
// Consumer warps + one producer warp.
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
// Polls of an mbarrier before a wait is declared lost.
constexpr uint32_t kWaitLimit = 1u << 22;

struct AttnParams {
    int32_t source;       // KeySource
    int32_t batch;
    int32_t n_kv_heads;
    int32_t head_dim;
    // verify (contiguous / paged)
    const int64_t *seq_lens;
    const int32_t *block_table;
    int64_t capacity;     // positions a sequence can hold (n_cap or max_pages * page_size)
    int64_t n_pages;
    int32_t page_size;
    int32_t max_pages;
    int32_t box_rows;     // key rows per TMA box (64, or 128 for the tensor-core kernel)
    // draft (ring)
    const int32_t *pos_tag;
    const int64_t *n_seen;
    int32_t n_slots;
    int32_t sink;
    int32_t window;
    // queries: rows of one KV head = n_q positions x group heads, row r = i * group + hh
    const void *q;        // verify [B][n_q][Hq][D]; draft [B][Hq][D]
    int32_t n_q;
    int32_t n_q_heads;
    int32_t group;
    int32_t rows;
    float scale_log2;     // scale * log2(e)
    // split
    int32_t n_split;
    int32_t keys_per_split;  // multiple of the kernel's key tile
    // outputs
    void *out;            // bf16, same layout as q
    float *lse;           // [B][n_q][Hq] or NULL
    float *o_part;        // [B*n_q*Hq][n_split][D] fp32, NULL when unsplit
    float *lse_part;      // [B*n_q*Hq][n_split]
    int32_t *err;         // device error word
    // fused draft step (ring append + draft attention in one launch)
    const void *k_new;    // [B][Hkv][D] bf16: the entries appended at p = n_seen[b]
    const void *v_new;
    void *ring_k;         // the ring's K and V, written at slot(p)
    void *ring_v;
    int32_t *tag_w;       // writable pos_tag of the ring
    // memory slots (memory-augmented draft): keys mem_base .. mem_base + count[b] - 1
    // are slots 0 .. count[b] - 1, read through the second pair of tensor maps
    const int64_t *mem_count;  // [B]; NULL: no memory slots
    int64_t mem_cap;           // slots the memory store holds per (sequence, KV head)
    int64_t mem_base;          // first key index of the memory region (ring tiles x 64)
    // pipeline waits: polls before a wait is declared lost, and (tests of the
    // timeout path only) the key tile at which the producer stops issuing
    // copies, -1 for none
    uint32_t wait_limit;
    int32_t stall_tile;
    // keys-as-M draft kernel only: balanced splits of the plan's key tiles
    // (plan_tiles = q * n_split + r: the first r splits take q + 1 tiles, the rest q)
    int32_t plan_tiles;
    // persistent tcgen05 verify over a batch (device-side schedule, verify_sched.cu):
    // tiles of one KV head before each sequence ([batch + 1]) and each CTA's run;
    // its partials are o_part [segments][rows][D] and lse_part [segments][rows]
    const int64_t *tile_prefix;
    const int4 *cta_start;  // [grid]: (sequence, KV head, first tile in that unit, tiles)
};

// Launch the attention kernel for head dim D (defined in attn_d<D>.cu).  mk/mv
// map the memory-slot store when p.mem_count is set (else any valid maps).
cudaError_t launch_attn_d64(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                            const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream);
cudaError_t launch_attn_d128(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                             const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream);
cudaError_t launch_attn_d256(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                             const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream);

// Keys-as-M draft kernel (draft_d<D>.cu) for up to kDraftRowsMax query rows per
// KV head: the plain draft attention, or (step) the fused draft step, which
// always writes split partials; fma selects the CUDA-core variant of its
// products (measurement only) instead of mma.sync.
constexpr int kDraftRowsMax = 8;
cudaError_t launch_draft_d64(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                             const CUtensorMap &mv, const AttnParams &p, bool step, bool fma, cudaStream_t stream);
cudaError_t launch_draft_d128(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                              const CUtensorMap &mv, const AttnParams &p, bool step, bool fma, cudaStream_t stream);
cudaError_t launch_draft_d256(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                              const CUtensorMap &mv, const AttnParams &p, bool step, bool fma, cudaStream_t stream);
// Resident CTAs per SM of that kernel (0 if unknown).
int draft_blocks_per_sm_d64(bool step, bool fma);
int draft_blocks_per_sm_d128(bool step, bool fma);
int draft_blocks_per_sm_d256(bool step, bool fma);

// Resident CTAs per SM of the mma.sync attention kernel for head dim D with
// m_tiles row tiles (step: the fused draft-step instance); 0 if unknown.
int attn_blocks_per_sm_d64(int m_tiles, bool step);
int attn_blocks_per_sm_d128(int m_tiles, bool step);
int attn_blocks_per_sm_d256(int m_tiles, bool step);

// Fused draft step (ring append + draft attention) for head dim D; always
// writes split partials (o_part / lse_part) for the merge kernel.
cudaError_t launch_step_d64(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                            const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream);
cudaError_t launch_step_d128(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                             const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream);
cudaError_t launch_step_d256(const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &mk,
                             const CUtensorMap &mv, const AttnParams &p, int m_tiles, cudaStream_t stream);

// Tensor-core (tcgen05) attention kernel for head dims 128 and 256 (attn_tc_d<D>.cu);
// n_rows16 is the row count per KV head rounded up to 16, 128-key tiles.
cudaError_t launch_attn_tc_d128(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p,
                                int n_rows16, cudaStream_t stream);
cudaError_t launch_attn_tc_d256(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p,
                                int n_rows16, cudaStream_t stream);
constexpr int kTcTile = 128;
// Resident CTAs per SM of the tcgen05 kernel for n_rows16 rows (0 if unknown).
int attn_tc_blocks_per_sm_d128(int n_rows16);
int attn_tc_blocks_per_sm_d256(int n_rows16);

// Persistent tcgen05 verify for a batch of sequences (attn_tcp_d<D>.cu): n_cta
// CTAs, each streaming the run of key tiles the schedule gives it.  Not
// instantiated for the configurations that stage V in half tiles (head_dim
// 256 with more than 32 rows): tcp_supported says which are.
__host__ __device__ constexpr bool tcp_supported(int head_dim, int n_rows16) {
    return (head_dim == 128 || head_dim == 256) && n_rows16 >= 16 && n_rows16 <= 64 && n_rows16 % 16 == 0 &&
           !(head_dim == 256 && n_rows16 >= 48);
}
cudaError_t launch_attn_tcp_d128(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p, int n_rows16,
                                 int n_cta, cudaStream_t stream);
cudaError_t launch_attn_tcp_d256(const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p, int n_rows16,
                                 int n_cta, cudaStream_t stream);
int attn_tcp_blocks_per_sm_d128(int n_rows16);
int attn_tcp_blocks_per_sm_d256(int n_rows16);

// The schedule of the persistent verify (verify_sched.cu): sched [batch + 3]
// int64 (chunk, total tiles, tile prefix [batch + 1]) and cta_start [n_cta];
// and the merge of its segment partials into out / lse_out.
cudaError_t launch_verify_sched(const int64_t *seq_lens, int batch, int n_kv_heads, int64_t capacity, int n_cta,
                                int64_t *sched, int4 *cta_start, int32_t *err, cudaStream_t stream);
cudaError_t launch_seg_merge(const float *o_seg, const float *lse_seg, const int64_t *sched, int batch,
                             int n_kv_heads, int n_q, int n_q_heads, int head_dim, void *out, float *lse_out,
                             cudaStream_t stream);

// Ring and merge kernels (ring.cu, merge.cu).
cudaError_t launch_ring_append(void *rk, void *rv, int32_t *tag, int64_t *n_seen, int batch,
                               int n_kv_heads, int head_dim, int sink, int window,
                               const void *k_new, const void *v_new, int32_t *err,
                               cudaStream_t stream);

struct HistSource {
    const void *k;
    const void *v;
    const int64_t *lens;
    const int32_t *block_table;
    int64_t n_cap;
    int64_t n_pages;
    int32_t page_size;
    int32_t max_pages;
};

cudaError_t launch_ring_fill(void *rk, void *rv, int32_t *tag, int64_t *n_seen, int batch,
                             int n_kv_heads, int head_dim, int sink, int window,
                             const HistSource &hist, int32_t *err, cudaStream_t stream);

// Memory-slot store of the memory-augmented draft (mem.cu): append one slot per
// sequence at count[b], and truncate the counts.
cudaError_t launch_mem_append(void *mk, void *mv, int64_t *count, int64_t capacity, int batch, int n_kv_heads,
                              int head_dim, const void *k_new, const void *v_new, int32_t *err,
                              cudaStream_t stream);
cudaError_t launch_mem_rollback(int64_t *count, int batch, const int64_t *new_count, int32_t *err,
                                cudaStream_t stream);

cudaError_t launch_ring_rollback(int32_t *tag, int64_t *n_seen, int batch, int n_slots,
                                 const int64_t *new_len, int32_t *err, cudaStream_t stream);

// Merge of split partials.  With commit_n_seen != NULL (the fused draft step)
// it also advances n_seen[b] by one for every sequence b whose value is >= 0;
// rows_per_seq rows of the output belong to each sequence.
cudaError_t launch_lse_merge(const float *o_parts, const float *lse_parts, int n_parts,
                             int64_t rows, int head_dim, void *out, float *lse_out,
                             int64_t *commit_n_seen, int rows_per_seq, cudaStream_t stream);

// The host-side argument checks of wm_draft_attn alone (ring, query, heads,
// scale, split count, output alignment): a wm_status code, WM_OK when they pass.
// Nothing is planned, encoded or launched.
int32_t draft_args_status(const ::wm_ring *ring, const void *q, int32_t n_q_heads, float scale, int32_t n_split,
                          const void *out, const float *lse);

}  // namespace wm

/*
 * wm_api.h -- C ABI of the Windowed-MTP decode-attention library (libwm.so).
 *
 * The operations are the decode-time attention of one speculative-decoding
 * step as described in "Windowed-MTP: Removing the Full-Context Draft-KV Tax
 * at Million-Token Context" (Abstract):
 *
 *   - the MTP draft head attends only to a StreamingLLM-style key set, the
 *     first S positions (attention sinks) plus the W most recent positions,
 *     held in a compact ring buffer of S + W slots   -> wm_ring_append,
 *     wm_ring_fill, wm_draft_attn;
 *   - the target's full-attention verification of the k+1 proposed positions
 *     over the entire bf16 KV cache stays intact      -> wm_verify_attn;
 *   - the split-KV partial results of either are combined by a log-sum-exp
 *     merge                                            -> wm_lse_merge.
 *
 * Conventions shared by every entry point
 *   - Element types: K, V, q and out are bf16 (IEEE binary16-brain, 2 bytes);
 *     lse and split partials are fp32; positions/lengths int64; tags and page
 *     indices int32.  Every tensor is dense row-major in the documented shape.
 *   - Ownership: every pointer is caller-owned DEVICE memory unless stated;
 *     the library allocates no device memory.  Its only state across calls
 *     is host-side: the TMA descriptors of recent calls.  A descriptor depends
 *     only on an address and a shape and owns nothing, so freeing or reusing
 *     a buffer needs no notice.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *     default stream).  Every call only enqueues work on that stream and
 *     returns without synchronising; positions and lengths are read on the
 *     device, so sequences of calls can be captured in a CUDA graph.
 *   - Validation: arguments are checked on the host before anything is
 *     enqueued; a failing check returns WM_ERR_INVALID_ARG / WM_ERR_UNSUPPORTED
 *     / WM_ERR_WORKSPACE and enqueues nothing.  A failed launch returns
 *     WM_ERR_CUDA.
 *   - Device-side data errors (a negative length, a length beyond the
 *     capacity, a block-table entry outside the page pool) cannot be seen on
 *     the host without a synchronisation.  The kernels clamp or skip the bad
 *     access, record the first such error in a device word and never trap;
 *     wm_get_device_error() reads and clears that word.
 *   - GQA: query head h reads KV head floor(h / G), G = n_q_heads / n_kv_heads.
 *   - Outputs: out is bf16 rounded to nearest-even once; lse is the natural
 *     log-sum-exp of the scaled logits in fp32.  A row with no key to attend
 *     to gets out = 0 and lse = -inf.
 *   - head_dim must be 64, 128 or 256; n_q_heads a multiple of n_kv_heads;
 *     G * (query positions) at most 64 rows per KV head; batch * n_kv_heads
 *     at most 65535 for the attention calls and wm_ring_fill, batch at most
 *     65535 for wm_ring_rollback; a wm_kv holds at most INT32_MAX positions
 *     per sequence (n_cap, or max_pages * page_size) and at most INT32_MAX
 *     pages (WM_ERR_UNSUPPORTED otherwise).
 */
#ifndef WM_API_H
#define WM_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum wm_status {
    WM_OK = 0,
    WM_ERR_INVALID_ARG = 1, /* null pointer, bad size or misaligned pointer */
    WM_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement */
    WM_ERR_WORKSPACE = 3,   /* workspace missing or smaller than wm_workspace_size() */
    WM_ERR_CUDA = 4,        /* a CUDA runtime call or a launch failed */
    WM_ERR_DEVICE_DATA = 5  /* reported by wm_get_device_error(): bad device-side data */
} wm_status;

/* Device error codes recorded by the kernels (read with wm_get_device_error). */
#define WM_DEVERR_NONE 0
#define WM_DEVERR_BAD_LENGTH 1   /* negative length/position or one beyond capacity */
#define WM_DEVERR_BAD_PAGE 2     /* block-table entry outside [0, n_pages) */
#define WM_DEVERR_TIMEOUT 3      /* a pipeline wait exceeded its iteration limit */
#define WM_DEVERR_INTERNAL 4     /* a kernel's own address-range self-check failed (the access was skipped) */

/*
 * The draft's compact ring buffer (one per draft attention layer).
 *   k, v     [batch][n_kv_heads][sink + window][head_dim] bf16
 *   pos_tag  [batch][sink + window] int32: absolute position held by the
 *            slot, -1 = empty.  Initialise to -1 (all bytes 0xFF).
 *   n_seen   [batch] int64: number of positions appended so far.
 *            Initialise to 0.
 * Slot of position p:  p                      if p < sink,
 *                      sink + (p - sink) % window   otherwise.
 * So the ring holds the sinks 0..S-1 and the W most recent positions; every
 * older non-sink position has been overwritten ("reclaimed").
 */
typedef struct wm_ring {
    void *k;
    void *v;
    int32_t *pos_tag;
    int64_t *n_seen;
    int32_t batch;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t sink;   /* S >= 0 */
    int32_t window; /* W >= 1 */
} wm_ring;

/*
 * Compressed memory slots of a memory-augmented sliding-window draft
 * ("Strong Drafts Need Compact Memories: Long-Context Speculative Decoding
 * with Compressed KV Cache", 4.1-4.3): at every r-token
 * boundary the draft's adaptor materializes one memory slot (its K/V come
 * from the caller; the adaptor is not part of this library) that stays after
 * the raw tokens leave the window.  A draft query attends to the sinks, the
 * window AND every slot materialized so far (wm_draft_attn_mem, wm_draft_step).
 *   k, v     [batch][n_kv_heads][capacity][head_dim] bf16
 *   count    [batch] int64: slots materialized so far, slot i at index i.
 *            Initialise to 0.
 */
typedef struct wm_mem {
    void *k;
    void *v;
    int64_t *count;
    int64_t capacity; /* slots per (sequence, KV head), >= 1 */
    int32_t batch;
    int32_t n_kv_heads;
    int32_t head_dim;
} wm_mem;

/*
 * A full-context KV cache (the target's), contiguous or paged.
 *   contiguous (block_table == NULL):
 *       k, v  [batch][n_kv_heads][n_cap][head_dim] bf16
 *   paged (block_table != NULL):
 *       k, v  [n_pages][n_kv_heads][page_size][head_dim] bf16
 *       block_table [batch][max_pages] int32: position j of sequence b lives
 *       in page block_table[b][j / page_size], row j % page_size.
 *       page_size must be a multiple of 64 (whole 64-key boxes per page).
 *   seq_lens [batch] int64: number of valid positions of each sequence.
 * k and v must be 16-byte aligned.
 */
typedef struct wm_kv {
    const void *k;
    const void *v;
    const int64_t *seq_lens;
    const int32_t *block_table;
    int64_t n_cap;   /* contiguous: positions per (sequence, head) row */
    int64_t n_pages; /* paged: pages in the pool */
    int32_t page_size;
    int32_t max_pages;
    int32_t batch;
    int32_t n_kv_heads;
    int32_t head_dim;
} wm_kv;

/*
 * Append one draft KV entry per sequence (Abstract: the draft's KV is kept in
 * a compact ring buffer).  For each sequence b, with p = n_seen[b]:
 * writes k_new[b], v_new[b] into slot(p), sets pos_tag[b][slot(p)] = p and
 * n_seen[b] = p + 1.
 *   k_new, v_new  [batch][n_kv_heads][head_dim] bf16.
 * Tags are int32, so p must lie in [0, INT32_MAX): any other n_seen[b]
 * records WM_DEVERR_BAD_LENGTH and appends nothing for b.
 */
wm_status wm_ring_append(const wm_ring *ring, const void *k_new, const void *v_new, void *stream);

/*
 * Bulk-initialise the ring from a history store: the result is bit-identical
 * to appending positions 0 .. hist->seq_lens[b]-1 one at a time to a ring in
 * its current state whose n_seen is 0.  Slots that would stay unwritten keep
 * their K/V bytes and get pos_tag = -1.  hist describes the draft's KV by
 * absolute position (contiguous or paged, same shape rules as wm_kv; its
 * n_kv_heads and head_dim must equal the ring's).
 */
wm_status wm_ring_fill(const wm_ring *ring, const wm_kv *hist, void *stream);

/*
 * Speculative rollback: forget draft entries at positions >= new_len[b]
 * (device int64 [batch]).  Sets n_seen[b] = min(n_seen[b], new_len[b]) and
 * pos_tag = -1 for every slot holding a position >= the new length.  Window
 * entries that the rejected positions overwrote are not restored; the window
 * is short until new appends refill it.
 */
wm_status wm_ring_rollback(const wm_ring *ring, const int64_t *new_len, void *stream);

/*
 * Windowed draft attention (Abstract: the draft attends to a sliding window
 * plus attention sinks only).  For sequence b the query sits at position
 * p = n_seen[b] - 1 (the entry appended last) and attends to every ring slot
 * whose tag t satisfies  0 <= t <= p  and  (t < sink  or  t > p - window).
 *   q    [batch][n_q_heads][head_dim] bf16
 *   out  [batch][n_q_heads][head_dim] bf16
 *   lse  [batch][n_q_heads] fp32, may be NULL
 *   scale  multiplies q.k before the softmax.
 *   n_split  0 = chosen by the library; else the number of key splits.
 *   workspace  device scratch of at least wm_workspace_size(WM_OP_DRAFT, ...)
 *              bytes (may be NULL when that size is 0); 256-byte aligned.
 */
wm_status wm_draft_attn(const wm_ring *ring, const void *q, int32_t n_q_heads, float scale,
                        int32_t n_split, void *out, float *lse, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Memory-augmented draft attention ("Strong Drafts Need Compact Memories:
 * Long-Context Speculative Decoding with Compressed KV Cache", 4.1 and
 * Appendix C: a raw-token query sees the sink tokens, the available memory
 * slots and a bounded local window).  As wm_draft_attn, and
 * in the same softmax the query also attends to memory slots
 * 0 .. mem->count[b]-1.  mem must match the ring's batch, n_kv_heads and
 * head_dim.  A count outside 0..capacity records WM_DEVERR_BAD_LENGTH and is
 * clamped.  Workspace: wm_workspace_size(WM_OP_DRAFT_MEM, ...) with
 * max_keys = 64 * ceil((sink + window) / 64) + capacity.
 */
wm_status wm_draft_attn_mem(const wm_ring *ring, const wm_mem *mem, const void *q, int32_t n_q_heads,
                            float scale, int32_t n_split, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * Materialize one memory slot per sequence: slot count[b] <- k_new[b], v_new[b]
 * (all KV heads), then count[b] += 1.  k_new, v_new [batch][n_kv_heads][head_dim].
 * A full store (count[b] == capacity) or a negative count records
 * WM_DEVERR_BAD_LENGTH and leaves that sequence unchanged.
 */
wm_status wm_mem_append(const wm_mem *mem, const void *k_new, const void *v_new, void *stream);

/*
 * Rollback of memory slots materialized after the accepted prefix (same
 * page, 4.3):
 * count[b] = min(count[b], new_count[b]), new_count a device int64 [batch].
 */
wm_status wm_mem_rollback(const wm_mem *mem, const int64_t *new_count, void *stream);

/*
 * Full-context verification attention (Abstract: full-attention verification
 * left intact).  Query i (0 <= i < n_q) of sequence b sits at position
 * seq_lens[b] - n_q + i -- the n_q proposed tokens' own K/V are the last n_q
 * cache entries -- and attends causally to keys 0 .. seq_lens[b] - n_q + i.
 *   q    [batch][n_q][n_q_heads][head_dim] bf16
 *   out  [batch][n_q][n_q_heads][head_dim] bf16
 *   lse  [batch][n_q][n_q_heads] fp32, may be NULL
 *   n_split, workspace: as for wm_draft_attn with WM_OP_VERIFY.
 * With n_q = 1 this is the native full-context decode attention.
 */
wm_status wm_verify_attn(const wm_kv *kv, const void *q, int32_t n_q, int32_t n_q_heads,
                         float scale, int32_t n_split, void *out, float *lse, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * Log-sum-exp merge of split partials, per row r:
 *   M = max_s lse_s,  lse = M + ln sum_s exp(lse_s - M),
 *   out = sum_s exp(lse_s - lse) * o_s.
 *   o_parts   [rows][n_parts][head_dim] fp32, each part normalised by its own sum
 *   lse_parts [rows][n_parts] fp32 natural log; -inf marks an empty part
 *   out       [rows][head_dim] bf16;  lse_out [rows] fp32, may be NULL.
 * A row whose parts are all empty gets out = 0, lse = -inf.
 * head_dim must be a multiple of 4 (WM_ERR_UNSUPPORTED otherwise); o_parts must
 * be 16-byte and out 8-byte aligned (WM_ERR_INVALID_ARG otherwise).
 */
wm_status wm_lse_merge(const float *o_parts, const float *lse_parts, int32_t n_parts, int64_t rows,
                       int32_t head_dim, void *out, float *lse_out, void *stream);

/*
 * Draft attention for callers that cannot allocate device memory.
 *
 * Windowed-MTP describes no such call: this is a deployment convenience.  Some
 * callers have no way to obtain the workspace that wm_draft_attn needs --
 * runtimes that reserve all device memory at start-up and refuse any later
 * allocation, plugins hosted by a framework that owns the GPU allocator and
 * hands them no scratch, and tight decode loops where a cudaMalloc would
 * synchronise the device.  This entry point computes exactly what
 * wm_draft_attn computes (same arguments minus the workspace), keeping the
 * split partials in a scratch array built into the library instead.
 *
 *   - The scratch is WM_STATIC_SCRATCH_BYTES per device and stays allocated on
 *     every GPU that loads the library until the process exits.
 *   - If the split partials of a call would need more than that (see
 *     wm_workspace_size with WM_OP_DRAFT), the call returns WM_ERR_WORKSPACE and
 *     enqueues nothing; pass a smaller n_split or use wm_draft_attn.
 *   - The first call on a device looks up the scratch array's device address
 *     (with that device current) and caches it; make that first call before
 *     any stream capture.
 *   - Every call on a device shares the one array and leaves its partials in
 *     it.  Nothing in it needs to start at zero.  Calls whose kernels can
 *     overlap on the GPU (different streams without ordering between them)
 *     race on the array: order them on one stream.
 *   - Allocates nothing: no cudaMalloc, no cudaFree.
 */
#define WM_STATIC_SCRATCH_BYTES (8u << 20)
wm_status wm_draft_attn_static(const wm_ring *ring, const void *q, int32_t n_q_heads, float scale,
                               int32_t n_split, void *out, float *lse, void *stream);

/*
 * Fused draft step: wm_ring_append followed by wm_draft_attn, with the append
 * folded into the attention launch (one attention launch + one merge launch
 * instead of append + attention (+ merge)).  The windowed draft reads only
 * the sinks and the window (Abstract: the draft attends to a sliding window
 * plus attention sinks held in a compact ring buffer), a few megabytes per
 * step, so its cost is launch and latency bound and the separate append
 * launch is a large part of it.  For each sequence b, with p = n_seen[b] on
 * entry:
 *   - the query q[b] sits at position p and attends to every ring slot whose
 *     tag t satisfies 0 <= t <= p and (t < sink or t > p - window), where
 *     slot(p) counts as holding p with K/V = k_new[b], v_new[b];
 *   - on completion slot(p) holds k_new[b], v_new[b], pos_tag[b][slot(p)] = p
 *     and n_seen[b] = p + 1 -- the state wm_ring_append leaves.
 *   k_new, v_new  [batch][n_kv_heads][head_dim] bf16
 *   q, out        [batch][n_q_heads][head_dim] bf16;  lse [batch][n_q_heads] fp32 or NULL
 *   mem           NULL, or memory slots the query also attends to (as
 *                 wm_draft_attn_mem).
 *   n_split       as for wm_draft_attn (same plan).
 *   workspace     at least wm_workspace_size(WM_OP_DRAFT_STEP, batch, n_kv_heads,
 *                 n_q_heads, 1, head_dim, sink + window, n_split) bytes (with mem:
 *                 WM_OP_DRAFT_MEM and its max_keys) -- never 0: the split
 *                 partials always pass through the merge, which commits
 *                 n_seen -- 256-byte aligned; no initial contents needed.
 * out, lse and the ring are bit-identical to wm_ring_append followed by
 * wm_draft_attn (wm_draft_attn_mem) with the same n_split.  An n_seen[b]
 * outside [0, INT32_MAX) (tags are int32) records WM_DEVERR_BAD_LENGTH,
 * appends nothing for b and gives its rows out = 0, lse = -inf.
 */
wm_status wm_draft_step(const wm_ring *ring, const wm_mem *mem, const void *k_new, const void *v_new,
                        const void *q, int32_t n_q_heads, float scale, int32_t n_split, void *out,
                        float *lse, void *workspace, size_t workspace_bytes, void *stream);

/* Operations for wm_workspace_size / wm_plan_splits. */
#define WM_OP_DRAFT 0
#define WM_OP_VERIFY 1
#define WM_OP_DRAFT_STEP 2
#define WM_OP_DRAFT_MEM 3 /* draft with memory slots, fused or not */

/*
 * Number of key splits an attention call will use, for a cache holding up to
 * max_keys positions per sequence (draft: sink + window).  n_split > 0 is
 * taken as given (at most one split per key tile).  n_split = 0 plans one
 * wave of the kernel's resident CTAs over the batch x n_kv_heads (sequence,
 * KV head) pairs.  With batch > 1 (lengths may differ, only their maximum is
 * known here) splits are also capped at about 8 MB of K+V each, and a cap
 * that needs more than one wave is rounded up to fill its last one.  Depends
 * on the current device's SM count and the kernels' measured residency.
 * Exception: a verify call that wm_verify_persistent accepts makes its
 * schedule on the device; for it this returns the persistent grid's CTA count.
 * Returns 0 on invalid arguments.
 */
int32_t wm_plan_splits(int32_t op, int32_t batch, int32_t n_kv_heads, int32_t n_q_heads,
                       int32_t n_q, int32_t head_dim, int64_t max_keys, int32_t n_split);

/*
 * Whether wm_verify_attn with these arguments runs the persistent verify,
 * and its CTA count (0: it runs the split plan).  The persistent verify
 * serves batch > 1 at head_dim 128 (up to 64 rows per KV head, rows = n_q x
 * n_q_heads / n_kv_heads) and 256 (up to 32 rows) when n_split = 0 and the
 * call holds at most 2^30 key tiles of 128 (batch x n_kv_heads x
 * ceil(max_keys / 128)).  The host sees only the largest length, so it cannot
 * split a ragged batch evenly; the call reads the actual lengths on the
 * device instead.  A one-CTA kernel lays the batch's key tiles end to end (the
 * (sequence, KV head) pairs in order), and each of the grid's CTAs (as many
 * as are resident at once) streams an equal run of them, with one partial
 * per pair its run touches.  A merge kernel combines the partials.  Three
 * launches per call; workspace as wm_workspace_size(WM_OP_VERIFY, ...) says.
 * Returns 0 on invalid arguments.
 */
int32_t wm_verify_persistent(int32_t batch, int32_t n_kv_heads, int32_t n_q_heads, int32_t n_q,
                             int32_t head_dim, int64_t max_keys, int32_t n_split);

/*
 * Workspace bytes an attention call needs for the same arguments (0 when it
 * runs unsplit; never 0 for WM_OP_DRAFT_STEP and WM_OP_DRAFT_MEM, which cover
 * the fused step).  For WM_OP_DRAFT and WM_OP_DRAFT_STEP pass n_q = 1 and
 * max_keys = sink + window; for WM_OP_DRAFT_MEM n_q = 1 and max_keys =
 * 64 * ceil((sink + window) / 64) + memory capacity;
 * for WM_OP_VERIFY, max_keys = n_cap (contiguous) or max_pages * page_size.
 * Returns (size_t)-1 on invalid arguments.
 */
size_t wm_workspace_size(int32_t op, int32_t batch, int32_t n_kv_heads, int32_t n_q_heads,
                         int32_t n_q, int32_t head_dim, int64_t max_keys, int32_t n_split);

/*
 * Synchronise `stream`, then read and clear the device error word of the
 * current device.  *code receives a WM_DEVERR_* value; returns WM_OK if it is
 * WM_DEVERR_NONE, WM_ERR_DEVICE_DATA otherwise, WM_ERR_CUDA if the read failed.
 */
wm_status wm_get_device_error(int32_t *code, void *stream);

/* Static description of a status code. */
const char *wm_status_string(wm_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t wm_version(void);

/*
 * Arithmetic of the draft attention kernel for the draft calls made by the
 * calling host thread (wm_draft_attn, wm_draft_attn_mem, wm_draft_step and
 * wm_draft_attn_static with at most 8 query heads per KV head; no counterpart
 * on the pages).  WM_DRAFT_MATH_MMA (the default): the Q.K^T and P.V products
 * on the tensor cores with mma.sync, keys as the M dimension.
 * WM_DRAFT_MATH_FMA: the same kernel with both products as fp32 FMA on the
 * CUDA cores and the softmax maxima reduced with warp shuffles; the same
 * results within the parity tolerance, kept to measure the choice between
 * the two.  The split plan is queried per setting (wm_plan_splits and
 * wm_workspace_size answer for the calling thread's setting).  Returns
 * WM_ERR_INVALID_ARG for any other value.
 */
#define WM_DRAFT_MATH_MMA 0
#define WM_DRAFT_MATH_FMA 1
wm_status wm_set_draft_math(int32_t math);

/*
 * Test support for the pipeline-wait timeout path (no counterpart on the
 * pages).  Every wait inside the attention kernels is bounded: after a limit
 * of polls the kernel records WM_DEVERR_TIMEOUT in the device error word,
 * stops its remaining work, waits (again bounded) for its own copies in
 * flight and returns, so a lost arrival can never hang the GPU.  This call
 * makes that path reachable on purpose: after it, every attention launch made
 * by the calling host thread has its producer stop issuing copies at copy
 * unit `stall_tile` of each split (a key tile in the mma.sync kernels; in the
 * tcgen05 verify kernel a K or V tile, or a 64-key V half where V is staged
 * in halves), so that unit never arrives, and gives up a wait after
 * `wait_polls` polls (about 0.1 us each, or more: a poll may suspend the
 * thread briefly).  stall_tile = -1 restores the defaults
 * (no stall, the production limit of 2^22 polls).  Outputs of a stalled call
 * are undefined; the context stays usable and the next call is normal.
 * Returns WM_ERR_INVALID_ARG for stall_tile < -1 or wait_polls = 0 with a stall.
 * Not for production use.
 */
wm_status wm_set_test_stall(int32_t stall_tile, uint32_t wait_polls);

#ifdef __cplusplus
}
#endif

#endif /* WM_API_H */

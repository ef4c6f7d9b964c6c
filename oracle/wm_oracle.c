/*
 * wm_oracle.c -- fp64 CPU oracle for Windowed-MTP decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * bench's CPU-baseline leg load the library built from this file.  It shares
 * no code, header, table or helper with the CUDA library; neither includes,
 * links or imports the other.
 *
 * What it computes, from "Windowed-MTP: Removing the Full-Context Draft-KV Tax
 * at Million-Token Context" (Abstract):
 *
 *   - Draft attention.  The MTP draft head attends only to a StreamingLLM-style
 *     key set: the attention sinks (the first S positions) plus a sliding
 *     window of the W most recent positions, the query's own position
 *     included.  For a query at position p the key set is
 *         M(p) = { j : 0 <= j <= p  and  (j < S  or  j > p - W) }.
 *   - Verification attention.  The full-attention target is left intact: query
 *     i of the T = k+1 proposed positions of sequence b sits at position
 *     P_i = N_b - T + i and attends causally to every key 0..P_i of the cache.
 *
 * Both are plain softmax attention,
 *     l_j = s * sum_d q_d K_{j,d},   m = max_j l_j,   Z = sum_j exp(l_j - m),
 *     o_d = (1/Z) sum_j exp(l_j - m) V_{j,d},   lse = m + ln Z,
 * evaluated in fp64 from the bf16 inputs (widened exactly), one row at a time,
 * in two passes over the key set: no ring buffer, no splitting of the keys,
 * no running rescale.  Rows are independent; OpenMP only spreads whole rows
 * over the host cores and changes no arithmetic.
 *
 *   - Memory-augmented draft ("Strong Drafts Need Compact Memories:
 *     Long-Context Speculative Decoding with Compressed KV Cache", 4.1 and
 *     Appendix C).  The draft's working memory is the sinks, the exact
 *     local window and the compressed memory slots materialized so far; a
 *     raw-token query attends to all three, M(p) plus slots 0..count-1.
 *
 * The log-sum-exp merge of partial results is the textbook identity
 *     lse = M + ln sum_s exp(lse_s - M),  o = sum_s exp(lse_s - lse) o_s.
 *
 * Conventions (readings of the pages, which give no formulas):
 *   - query head h reads KV head floor(h / G), G = Hq / Hkv (contiguous groups);
 *   - the window includes the query's own position; sink and window overlap is
 *     a set union (no key counted twice);
 *   - a row with an empty key set returns o = 0 and lse = -inf.
 *
 * Compile-time switch WMO_PLANT selects a deliberately wrong variant; it exists
 * only so that the tests can show that their pins catch plausible mistakes.
 * The product oracle is built with WMO_PLANT undefined.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef WMO_PLANT
#define WMO_PLANT 0
#endif

/* Key/value storage of one attention layer, seen through its logical index
 * (sequence b, kv head h, position j).
 *   contiguous (block_table == NULL): k, v are [batch][n_kv_heads][n_cap][head_dim]
 *   paged      (block_table != NULL): k, v are [n_pages][n_kv_heads][page_size][head_dim]
 *              and position j of sequence b lives in page
 *              block_table[b * max_pages + j / page_size], row j % page_size. */
typedef struct {
    const uint16_t *k;
    const uint16_t *v;
    const int32_t *block_table;
    int64_t n_cap;
    int64_t n_pages;
    int32_t page_size;
    int32_t max_pages;
    int32_t batch;
    int32_t n_kv_heads;
    int32_t head_dim;
} wmo_kv;

/* bf16 is the upper half of an IEEE binary32; widening it is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Address of the bf16 row holding position j of (b, h); NULL if out of range. */
static const uint16_t *kv_row(const wmo_kv *kv, const uint16_t *base, int b, int h, int64_t j)
{
    if (j < 0) return NULL;
    if (kv->block_table == NULL) {
        if (j >= kv->n_cap) return NULL;
        return base + (((int64_t)b * kv->n_kv_heads + h) * kv->n_cap + j) * kv->head_dim;
    }
    int64_t slot = j / kv->page_size;
    if (slot >= kv->max_pages) return NULL;
#if WMO_PLANT == 8
    int64_t page = kv->block_table[slot]; /* planted: block table row of sequence 0 for all */
#else
    int64_t page = kv->block_table[(int64_t)b * kv->max_pages + slot];
#endif
    if (page < 0 || page >= kv->n_pages) return NULL;
    return base + ((page * kv->n_kv_heads + h) * kv->page_size + j % kv->page_size) * kv->head_dim;
}

/* Which positions 0..n_pos-1 a row attends to. */
enum { KEYS_CAUSAL = 0, KEYS_SINK_WINDOW = 1 };
typedef struct {
    int kind;
    int64_t pos;  /* query position */
    int64_t sink; /* S */
    int64_t window; /* W */
} keyset;

static int in_keyset(const keyset *ks, int64_t j)
{
    if (j > ks->pos) return 0;
    if (ks->kind == KEYS_CAUSAL) return 1;
#if WMO_PLANT == 1
    /* planted: window that excludes the query's own position */
    return j < ks->sink || (j > ks->pos - ks->window - 1 && j < ks->pos);
#elif WMO_PLANT == 2
    /* planted: window one position too wide */
    return j < ks->sink || j >= ks->pos - ks->window;
#elif WMO_PLANT == 3
    /* planted: sink dropped */
    return j > ks->pos - ks->window;
#else
    return j < ks->sink || j > ks->pos - ks->window;
#endif
}

/* One row of softmax attention: query q (bf16, D) against every member of the
 * key set among positions 0..ks->pos of (b, h).  Returns 0, or -1 if a member
 * position has no storage. */
static int attend_row(const wmo_kv *kv, int b, int h, const uint16_t *q, double scale,
                      const keyset *ks, double *out, double *lse)
{
    const int D = kv->head_dim;
    const int64_t n_pos = ks->pos + 1;
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *logit = (double *)malloc(sizeof(double) * (size_t)(n_pos > 0 ? n_pos : 1));
    int rc = 0;
    for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(q[d]);
    for (int d = 0; d < D; ++d) out[d] = 0.0;

    /* pass 1: logits of the members and their maximum */
    double m = -INFINITY;
    int64_t n_members = 0;
    for (int64_t j = 0; j < n_pos; ++j) {
        if (!in_keyset(ks, j)) continue;
        const uint16_t *kr = kv_row(kv, kv->k, b, h, j);
        if (!kr) { rc = -1; goto done; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * bf16_to_double(kr[d]);
#if WMO_PLANT == 4
        logit[j] = dot; /* planted: scale ignored */
#else
        logit[j] = scale * dot;
#endif
        if (logit[j] > m) m = logit[j];
        ++n_members;
    }
    if (n_members == 0) { *lse = -INFINITY; goto done; }

    /* pass 2: normaliser and weighted sum of the values */
    double z = 0.0;
    for (int64_t j = 0; j < n_pos; ++j) {
        if (!in_keyset(ks, j)) continue;
        const uint16_t *vr = kv_row(kv, kv->v, b, h, j);
        if (!vr) { rc = -1; goto done; }
        double w = exp(logit[j] - m);
        z += w;
        for (int d = 0; d < D; ++d) out[d] += w * bf16_to_double(vr[d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= z;
#if WMO_PLANT == 7
    *lse = log(z); /* planted: max term dropped from the log-sum-exp */
#else
    *lse = m + log(z);
#endif
done:
    free(qd);
    free(logit);
    return rc;
}

static int check_kv(const wmo_kv *kv)
{
    if (!kv || !kv->k || !kv->v) return -1;
    if (kv->head_dim <= 0 || kv->n_kv_heads <= 0 || kv->batch <= 0) return -1;
    if (kv->block_table && (kv->page_size <= 0 || kv->max_pages <= 0 || kv->n_pages <= 0)) return -1;
    if (!kv->block_table && kv->n_cap < 0) return -1;
    return 0;
}

/* GQA: query head h of Hq reads KV head floor(h / (Hq / Hkv)). */
static int kv_head_of(int h, int n_q_heads, int n_kv_heads)
{
#if WMO_PLANT == 5
    (void)n_q_heads;
    return h % n_kv_heads; /* planted: interleaved instead of contiguous groups */
#else
    return h / (n_q_heads / n_kv_heads);
#endif
}

int wmo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the OpenMP loops from now on (n > 0; ignored without OpenMP). */
void wmo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Verification attention.
 * q: [batch][T][Hq][D] bf16; seq_lens: [batch] (N_b, the verify tokens' own
 * K/V being the last T cache entries).  rows: indices into the flattened
 * [batch][T][Hq] row space to evaluate (NULL = all, in order); out: [n][D],
 * lse: [n] for the n evaluated rows.  Returns 0, -1 on bad arguments, -2 if a
 * key position has no storage. */
int wmo_verify(const wmo_kv *kv, int T, int n_q_heads, const uint16_t *q,
               const int64_t *seq_lens, double scale, const int64_t *rows, int64_t n_rows,
               double *out, double *lse)
{
    if (check_kv(kv) || !q || !seq_lens || !out || !lse || T <= 0 || n_q_heads <= 0) return -1;
    if (n_q_heads % kv->n_kv_heads) return -1;
    const int64_t total = (int64_t)kv->batch * T * n_q_heads;
    const int64_t n = rows ? n_rows : total;
    const int D = kv->head_dim;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t s = 0; s < n; ++s) {
        int64_t r = rows ? rows[s] : s;
        if (r < 0 || r >= total) { err = -1; continue; }
        int b = (int)(r / ((int64_t)T * n_q_heads));
        int i = (int)((r / n_q_heads) % T);
        int h = (int)(r % n_q_heads);
#if WMO_PLANT == 6
        keyset ks = { KEYS_CAUSAL, seq_lens[b] - T + i - 1, 0, 0 }; /* planted: own key dropped */
#else
        keyset ks = { KEYS_CAUSAL, seq_lens[b] - T + i, 0, 0 };
#endif
        if (attend_row(kv, b, kv_head_of(h, n_q_heads, kv->n_kv_heads), q + r * D, scale, &ks,
                       out + s * D, lse + s))
            err = -2;
    }
    return err;
}

/* Draft attention over the sink + window key set.
 * hist: the draft's KV history indexed by absolute position; q: [batch][Hq][D]
 * bf16; pos: [batch] query position p_b (the position just appended).
 * rows index the flattened [batch][Hq] space (NULL = all). */
int wmo_draft(const wmo_kv *hist, int n_q_heads, const uint16_t *q, const int64_t *pos,
              int64_t sink, int64_t window, double scale, const int64_t *rows, int64_t n_rows,
              double *out, double *lse)
{
    if (check_kv(hist) || !q || !pos || !out || !lse || n_q_heads <= 0) return -1;
    if (n_q_heads % hist->n_kv_heads || sink < 0 || window < 1) return -1;
    const int64_t total = (int64_t)hist->batch * n_q_heads;
    const int64_t n = rows ? n_rows : total;
    const int D = hist->head_dim;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t s = 0; s < n; ++s) {
        int64_t r = rows ? rows[s] : s;
        if (r < 0 || r >= total) { err = -1; continue; }
        int b = (int)(r / n_q_heads);
        int h = (int)(r % n_q_heads);
        keyset ks = { KEYS_SINK_WINDOW, pos[b], sink, window };
        if (attend_row(hist, b, kv_head_of(h, n_q_heads, hist->n_kv_heads), q + r * D, scale, &ks,
                       out + s * D, lse + s))
            err = -2;
    }
    return err;
}

/* Memory-augmented sliding-window draft ("Strong Drafts Need Compact
 * Memories: Long-Context Speculative Decoding with Compressed KV Cache", 4.1
 * and Appendix C): the working memory of the draft is the
 * union of the attention sinks, the exact local window and the compressed
 * memory slots materialized so far, and an ordinary raw-token query sees
 * exactly those.  So for a query at position p of sequence b the key set is
 * M(p) over the draft history (as in wmo_draft) plus memory slots
 * 0..mem_count[b]-1 of `mem`, under one softmax.  The slots' K/V come from
 * the draft's adaptor; here they are inputs.  mem is a contiguous store
 * [batch][n_kv_heads][capacity][head_dim] (its n_cap is the capacity). */
static int attend_row_mem(const wmo_kv *hist, const wmo_kv *mem, int64_t n_mem, int b, int h,
                          const uint16_t *q, double scale, const keyset *ks, double *out, double *lse)
{
    const int D = hist->head_dim;
    const int64_t n_pos = ks->pos + 1 > 0 ? ks->pos + 1 : 0;
#if WMO_PLANT == 9
    n_mem = n_mem > 0 ? n_mem - 1 : 0; /* planted: the newest memory slot dropped */
#endif
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *logit = (double *)malloc(sizeof(double) * (size_t)(n_pos + n_mem > 0 ? n_pos + n_mem : 1));
    int rc = 0;
    for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(q[d]);
    for (int d = 0; d < D; ++d) out[d] = 0.0;

    /* pass 1: logits of the window members (index j) and the slots (n_pos + s) */
    double m = -INFINITY;
    int64_t n_members = 0;
    for (int64_t i = 0; i < n_pos + n_mem; ++i) {
        const uint16_t *kr;
        if (i < n_pos) {
            if (!in_keyset(ks, i)) continue;
            kr = kv_row(hist, hist->k, b, h, i);
        } else {
            kr = kv_row(mem, mem->k, b, h, i - n_pos);
        }
        if (!kr) { rc = -1; goto done; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * bf16_to_double(kr[d]);
        logit[i] = scale * dot;
        if (logit[i] > m) m = logit[i];
        ++n_members;
    }
    if (n_members == 0) { *lse = -INFINITY; goto done; }

    /* pass 2: normaliser and weighted sum of the values */
    double z = 0.0;
    for (int64_t i = 0; i < n_pos + n_mem; ++i) {
        const uint16_t *vr;
        if (i < n_pos) {
            if (!in_keyset(ks, i)) continue;
            vr = kv_row(hist, hist->v, b, h, i);
        } else {
            vr = kv_row(mem, mem->v, b, h, i - n_pos);
        }
        if (!vr) { rc = -1; goto done; }
        double w = exp(logit[i] - m);
        z += w;
        for (int d = 0; d < D; ++d) out[d] += w * bf16_to_double(vr[d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= z;
    *lse = m + log(z);
done:
    free(qd);
    free(logit);
    return rc;
}

/* Draft attention over sinks + window + memory slots.  As wmo_draft, plus
 * mem (contiguous, same batch / heads / head_dim as hist) and mem_count
 * [batch]: slots materialized so far (0..capacity).  Returns -1 on bad
 * arguments, -2 if a key has no storage. */
int wmo_draft_mem(const wmo_kv *hist, const wmo_kv *mem, const int64_t *mem_count, int n_q_heads,
                  const uint16_t *q, const int64_t *pos, int64_t sink, int64_t window, double scale,
                  const int64_t *rows, int64_t n_rows, double *out, double *lse)
{
    if (check_kv(hist) || check_kv(mem) || mem->block_table || !mem_count || !q || !pos || !out || !lse ||
        n_q_heads <= 0)
        return -1;
    if (n_q_heads % hist->n_kv_heads || sink < 0 || window < 1) return -1;
    if (mem->batch != hist->batch || mem->n_kv_heads != hist->n_kv_heads || mem->head_dim != hist->head_dim)
        return -1;
    const int64_t total = (int64_t)hist->batch * n_q_heads;
    const int64_t n = rows ? n_rows : total;
    const int D = hist->head_dim;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t s = 0; s < n; ++s) {
        int64_t r = rows ? rows[s] : s;
        if (r < 0 || r >= total) { err = -1; continue; }
        int b = (int)(r / n_q_heads);
        int h = (int)(r % n_q_heads);
        if (mem_count[b] < 0 || mem_count[b] > mem->n_cap) { err = -1; continue; }
        keyset ks = { KEYS_SINK_WINDOW, pos[b], sink, window };
        if (attend_row_mem(hist, mem, mem_count[b], b, kv_head_of(h, n_q_heads, hist->n_kv_heads), q + r * D,
                           scale, &ks, out + s * D, lse + s))
            err = -2;
    }
    return err;
}

/* Softmax attention of one query over an explicit subset of n keys:
 * k, v: [n][D] bf16, member: [n] (nonzero = in the set). */
int wmo_attend_subset(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint8_t *member,
                      int64_t n, int D, double scale, double *out, double *lse)
{
    if (!q || !k || !v || !member || !out || !lse || n < 0 || D <= 0) return -1;
    double m = -INFINITY;
    double *logit = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    int64_t n_members = 0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        if (!member[j]) continue;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(k[j * D + d]);
        logit[j] = scale * dot;
        if (logit[j] > m) m = logit[j];
        ++n_members;
    }
    if (n_members == 0) { *lse = -INFINITY; free(logit); return 0; }
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        if (!member[j]) continue;
        double w = exp(logit[j] - m);
        z += w;
        for (int d = 0; d < D; ++d) out[d] += w * bf16_to_double(v[j * D + d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= z;
    *lse = m + log(z);
    free(logit);
    return 0;
}

/* Log-sum-exp merge of n_parts partial results per row.
 * o_parts: [rows][n_parts][D], lse_parts: [rows][n_parts] (natural log;
 * -inf marks an empty part).  out: [rows][D], lse: [rows]. */
int wmo_lse_merge(const double *o_parts, const double *lse_parts, int n_parts, int64_t rows, int D,
                  double *out, double *lse)
{
    if (!o_parts || !lse_parts || !out || !lse || n_parts <= 0 || rows < 0 || D <= 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const double *ls = lse_parts + r * n_parts;
        double M = -INFINITY;
        for (int s = 0; s < n_parts; ++s)
            if (ls[s] > M) M = ls[s];
        for (int d = 0; d < D; ++d) out[r * D + d] = 0.0;
        if (M == -INFINITY) { lse[r] = -INFINITY; continue; }
        double z = 0.0;
        for (int s = 0; s < n_parts; ++s) z += exp(ls[s] - M);
        double total = M + log(z);
        lse[r] = total;
        for (int s = 0; s < n_parts; ++s) {
            double w = exp(ls[s] - total);
            const double *o = o_parts + (r * n_parts + s) * D;
            for (int d = 0; d < D; ++d) out[r * D + d] += w * o[d];
        }
    }
    return 0;
}

/*
 * pa_oracle.c -- plain, slow fp64 CPU oracle for paged GQA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file:
 * only tests/, the smoke check and the CPU-baseline leg of the benchmark use it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (cited by page and section):
 *   [page832 §1]  luanjiahao.me feed, post "784 -> 832 KV page for the DCU vendor
 *                 paged attention", section 1: logical_page = t // BLOCK_SIZE,
 *                 page_offset = t % BLOCK_SIZE, physical_page = block_table[logical_page],
 *                 then the K/V stride, KV head and head dim give the address.
 *   [page832 §4]  same post, section 4: cache tensor [num_pages, 2, BLOCK_SIZE, 4, 256]
 *                 BF16; after unbind(1) K and V are each [num_pages, BLOCK_SIZE, 4, 256].
 *                 24 query heads over 4 KV heads (GQA ratio 6), head size 256.
 *   [page832 §5]  same post, section 5: per key tile, score = dot(Q, K) * scale, then a
 *                 softmax over the scores weights V.  The oracle does the softmax exactly
 *                 (max-shifted, fp64), not online.
 *   [page832 §6]  same post, section 6: chunked prefill is full causal attention of the
 *                 chunk's queries over all earlier tokens plus the chunk itself.
 *   [input-prep §3.2] jsqmd.com "single-token decode input preparation on DCU",
 *                 section 3.2: slot = block_table[pos // block_size] * block_size
 *                 + pos % block_size.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - query head h reads KV head h / (Hq / Hkv)  (consecutive grouping);
 *   - a prefill query at absolute position p sees keys 0..p inclusive;
 *   - a negative position is a padding token with slot -1, and a slot < 0 is not
 *     written;
 *   - the caches are two separate arrays with a common page stride in elements,
 *     which covers both a plain [pages, BS, Hkv, D] tensor and the unbind(1) views.
 *
 * All floating point is fp64 over the exact values of the BF16 inputs.
 * Every parallel loop below only splits independent (row, head) problems across
 * threads; the arithmetic of each problem is the sequential loop written here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact value of a BF16 bit pattern: BF16 is the high half of an IEEE binary32. */
static double bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Address of token t of KV head g in one cache, through one sequence's block table
 * row [page832 §1].  Returns NULL if the block table maps the token outside the pool. */
static const uint16_t *paged_row(const uint16_t *cache, int64_t page_stride, int64_t num_pages,
                                 const int32_t *block_table_row, int block_size,
                                 int num_kv_heads, int head_dim, int64_t t, int g) {
    int64_t logical_page = t / block_size;
    int64_t page_offset = t % block_size;
    int64_t physical_page = block_table_row[logical_page];
    if (physical_page < 0 || physical_page >= num_pages) return NULL;
    return cache + physical_page * page_stride + (page_offset * num_kv_heads + g) * head_dim;
}

int pa_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Slot mapping [input-prep §3.2].  seq_idx may be NULL (every token in sequence 0).
 * A negative position marks a padding token: its slot is -1 (a reading; the pages do
 * not say).  Returns 0. */
int pa_oracle_slot_mapping(const int32_t *positions, const int32_t *seq_idx,
                           const int32_t *block_table, int64_t bt_stride, int num_tokens,
                           int block_size, int64_t *slot_mapping) {
    for (int i = 0; i < num_tokens; ++i) {
        int64_t pos = positions[i];
        int64_t s = seq_idx ? seq_idx[i] : 0;
        if (pos < 0) { slot_mapping[i] = -1; continue; }
        int64_t logical_block = pos / block_size;
        int64_t block_number = block_table[s * bt_stride + logical_block];
        int64_t block_offset = pos % block_size;
        slot_mapping[i] = block_number * block_size + block_offset;
    }
    return 0;
}

/* Decode-step inputs [input-prep §2, §4, §5]: num_seqs entries, each either a sequence
 * that decodes one token at positions[s] (tokens already cached) or a padding entry
 * (positions[s] < 0).  The step's metadata is written once:
 *   seq_lens[s] = position + 1, and 0 for a padding entry;
 *   input_ids[s] = the token sampled by the previous step;
 *   query_start_loc[0] = 0 and query_start_loc[s + 1] = query_start_loc[s] + (query rows
 *   of entry s): one row for a sequence, none for a padding entry.  With one sequence
 *   followed by padding this gives the pages' [0, 1, 1, ...] beside [position + 1, 0, 0,
 *   ...] (§2): a padded entry has no keys and owns no query row.
 * Then every KV-cache group g, with its own block table and block size, gets its slot
 * mapping by the slot formula above (row s of the group's table for sequence s). */
int pa_oracle_decode_input_prep(const int32_t *positions, const int32_t *sampled_ids,
                                int32_t *input_ids, int32_t *seq_lens,
                                int32_t *query_start_loc, int num_seqs, int num_groups,
                                const int32_t *const *block_tables, const int64_t *bt_strides,
                                const int *block_sizes, int64_t *const *slot_mappings) {
    query_start_loc[0] = 0;
    for (int s = 0; s < num_seqs; ++s) {
        int32_t pos = positions[s];
        int query_rows = pos >= 0 ? 1 : 0;
        seq_lens[s] = pos >= 0 ? pos + 1 : 0;
        if (sampled_ids) input_ids[s] = sampled_ids[s];
        query_start_loc[s + 1] = query_start_loc[s] + query_rows;
    }
    for (int g = 0; g < num_groups; ++g) {
        for (int s = 0; s < num_seqs; ++s) {
            int32_t seq = s;
            pa_oracle_slot_mapping(&positions[s], &seq, block_tables[g], bt_strides[g], 1,
                                   block_sizes[g], &slot_mappings[g][s]);
        }
    }
    return 0;
}

/* KV write: token i's rows (all KV heads, [Hkv, D] contiguous) go to page slot/BS,
 * offset slot%BS of each cache [page832 §4 layout].  Negative slots are skipped. */
void pa_oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                                 uint16_t *k_cache, uint16_t *v_cache, int64_t page_stride,
                                 const int64_t *slot_mapping, int num_tokens,
                                 int num_kv_heads, int head_dim, int block_size) {
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        int64_t page = slot / block_size, offset = slot % block_size;
        for (int64_t e = 0; e < row; ++e) {
            k_cache[page * page_stride + offset * row + e] = key[(int64_t)i * row + e];
            v_cache[page * page_stride + offset * row + e] = value[(int64_t)i * row + e];
        }
    }
}

/*
 * The definition of attention for one query row q (head_dim BF16 values) of one
 * query head, over keys 0..num_keys-1 of KV head g of one sequence:
 *     s_t = scale * sum_d q[d] k_t[d]
 *     w_t = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u)
 *     out[d] = sum_t w_t v_t[d]
 * k_t, v_t are fetched through the block table [page832 §1, §5].
 * If weights != NULL the softmax weights w_t are stored there.
 * Returns 0, -1 on bad arguments, -2 if a key maps outside the page pool.
 */
int pa_oracle_attend_row(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         int64_t page_stride, int64_t num_pages, const int32_t *block_table_row,
                         int block_size, int num_kv_heads, int head_dim, int g, int64_t num_keys,
                         double scale, double *out, double *weights) {
    if (num_keys <= 0 || head_dim <= 0 || block_size <= 0) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)num_keys);
    if (!s) return -1;
    int rc = 0;
    /* scores */
    for (int64_t t = 0; t < num_keys; ++t) {
        const uint16_t *k = paged_row(k_cache, page_stride, num_pages, block_table_row,
                                      block_size, num_kv_heads, head_dim, t, g);
        if (!k) { rc = -2; goto done; }
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += bf16_value(q[d]) * bf16_value(k[d]);
        s[t] = scale * dot;
    }
    /* softmax, shifted by the maximum score */
    double m = s[0];
    for (int64_t t = 1; t < num_keys; ++t) if (s[t] > m) m = s[t];
    double z = 0.0;
    for (int64_t t = 0; t < num_keys; ++t) { s[t] = exp(s[t] - m); z += s[t]; }
    for (int64_t t = 0; t < num_keys; ++t) s[t] /= z;
    if (weights) memcpy(weights, s, sizeof(double) * (size_t)num_keys);
    /* weighted sum of values */
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    for (int64_t t = 0; t < num_keys; ++t) {
        const uint16_t *v = paged_row(v_cache, page_stride, num_pages, block_table_row,
                                      block_size, num_kv_heads, head_dim, t, g);
        if (!v) { rc = -2; goto done; }
        for (int d = 0; d < head_dim; ++d) out[d] += s[t] * bf16_value(v[d]);
    }
done:
    free(s);
    return rc;
}

/*
 * q=1 decode for a batch: sequence i has seq_lens[i] keys (the new token included)
 * and block table row block_table + i*bt_stride.  q and out are [num_seqs, Hq, D].
 * Query head h reads KV head h / (Hq / Hkv).
 */
int pa_oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                     int64_t page_stride, int64_t num_pages, const int32_t *block_table,
                     int64_t bt_stride, const int32_t *seq_lens, int num_seqs,
                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                     double scale, double *out, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads) return -1;
    int group = num_q_heads / num_kv_heads;
    int rc = 0;
    int64_t n = (int64_t)num_seqs * num_q_heads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads > 0 ? num_threads : 1) reduction(min : rc)
#endif
    for (int64_t i = 0; i < n; ++i) {
        int s = (int)(i / num_q_heads), h = (int)(i % num_q_heads);
        int r = pa_oracle_attend_row(q + i * head_dim, k_cache, v_cache, page_stride, num_pages,
                                     block_table + (int64_t)s * bt_stride, block_size,
                                     num_kv_heads, head_dim, h / group, seq_lens[s], scale,
                                     out + i * head_dim, NULL);
        if (r < rc) rc = r;
    }
    (void)num_threads;
    return rc;
}

/*
 * Chunked prefill of one sequence [page832 §6]: query row i (0 <= i < q_len) sits at
 * absolute position q_start + i.  With causal != 0 it sees keys 0..q_start+i; otherwise
 * all q_start + q_len keys.  Only the (row, head) pairs listed are computed:
 * rows[j], heads[j] -> out[j*D .. j*D+D).  q is [q_len, Hq, D].
 */
int pa_oracle_prefill_rows(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                           int64_t page_stride, int64_t num_pages, const int32_t *block_table_row,
                           int q_len, int q_start, int causal, int num_q_heads, int num_kv_heads,
                           int head_dim, int block_size, double scale, const int32_t *rows,
                           const int32_t *heads, int64_t count, double *out, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads) return -1;
    int group = num_q_heads / num_kv_heads;
    int rc = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads > 0 ? num_threads : 1) reduction(min : rc)
#endif
    for (int64_t j = 0; j < count; ++j) {
        int i = rows[j], h = heads[j];
        if (i < 0 || i >= q_len || h < 0 || h >= num_q_heads) { if (-1 < rc) rc = -1; continue; }
        int64_t num_keys = causal ? (int64_t)q_start + i + 1 : (int64_t)q_start + q_len;
        int r = pa_oracle_attend_row(q + ((int64_t)i * num_q_heads + h) * head_dim, k_cache,
                                     v_cache, page_stride, num_pages, block_table_row, block_size,
                                     num_kv_heads, head_dim, h / group, num_keys, scale,
                                     out + j * head_dim, NULL);
        if (r < rc) rc = r;
    }
    (void)num_threads;
    return rc;
}

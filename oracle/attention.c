/*
 * oracle/attention.c -- plain, slow fp64 CPU oracle for chunked-prefill attention
 * over a paged KV cache and for the slot_mapping KV write.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this file's library. It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it follows (page titles and sections):
 *  - "Chunked-Prefills" article, section 3.2.1 (chunked attention): a chunk's
 *    queries score against the concatenation of the cached history keys and the
 *    chunk's own keys, softmax, then the weighted sum of the matching values.
 *    Readings taken where the page is silent or garbled:
 *      * the score scale is 1/sqrt(head_dim) (the page divides by sqrt of its
 *        hidden size H; with per-head attention that is the head dimension);
 *      * the mask is causal: query i of request r sits at absolute position
 *        h_r + i and sees keys 0 .. h_r + i (h_r = seq_len - query_len);
 *      * grouped-query heads: q head h reads kv head h / (Hq / Hkv).
 *  - Ascend dual-stream article, section 3.1 (attn_metadata): slot_mapping maps
 *    every new token to its cache slot, block_table lists each request's pages,
 *    seq_lens count history plus the current tokens, query_lens the current ones.
 *    Reading: slot s lives in page s / P at offset s % P, and the cache layout is
 *    [num_pages][Hkv][P][d]; a negative slot is a padding token and is skipped.
 *
 * Arithmetic is fp64 throughout; bf16 inputs are widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * KV write: for every token t with slot = slot_mapping[t] >= 0, copy
 * k[t][h][:] into k_cache[slot / P][h][slot % P][:] (and the same for v).
 * Returns the number of tokens whose slot was out of range (those are skipped).
 */
long oracle_kv_cache_write(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                           long num_tokens, int num_kv_heads, int head_dim, int page_size,
                           long num_pages, uint16_t *k_cache, uint16_t *v_cache)
{
    long bad = 0;
    for (long t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_pages * page_size) {
            ++bad;
            continue;
        }
        int64_t page = slot / page_size;
        int64_t off = slot % page_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = (((size_t)page * num_kv_heads + h) * page_size + off) * head_dim;
            size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
            for (int x = 0; x < head_dim; ++x) {
                k_cache[dst + x] = k[src + x];
                v_cache[dst + x] = v[src + x];
            }
        }
    }
    return bad;
}

/*
 * Attention for selected query tokens.
 *
 * rows[n] are global token indices into q (0 .. num_tokens-1); when rows is NULL
 * every token is computed and n_rows must equal num_tokens. out is
 * [n_rows][num_q_heads][head_dim] fp64. Returns 0, or a negative code for a
 * malformed batch (-1: sum of query_lens != num_tokens, -2: seq_len < query_len,
 * -3: a row index out of range, -4: a needed block_table entry out of range).
 */
int oracle_paged_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *query_lens, const int32_t *seq_lens,
                           const int32_t *block_table, int num_reqs, int max_blocks,
                           long num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                           int page_size, long num_pages, double scale,
                           const int64_t *rows, long n_rows, double *out)
{
    long *start = (long *)malloc(sizeof(long) * (size_t)(num_reqs + 1));
    if (!start)
        return -5;
    start[0] = 0;
    for (int r = 0; r < num_reqs; ++r) {
        if (seq_lens[r] < query_lens[r] || query_lens[r] < 0) {
            free(start);
            return -2;
        }
        start[r + 1] = start[r] + query_lens[r];
    }
    if (start[num_reqs] != num_tokens) {
        free(start);
        return -1;
    }
    if (scale <= 0.0)
        scale = 1.0 / sqrt((double)head_dim);
    int group = num_q_heads / num_kv_heads;
    int status = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (long n = 0; n < n_rows * num_q_heads; ++n) {
        long row = n / num_q_heads;
        int h = (int)(n % num_q_heads);
        long t = rows ? (long)rows[row] : row;
        double *o = out + ((size_t)row * num_q_heads + h) * head_dim;
        if (t < 0 || t >= num_tokens) {
#pragma omp atomic write
            status = -3;
            continue;
        }
        /* find the request that owns token t */
        int r = 0;
        while (r < num_reqs && start[r + 1] <= t)
            ++r;
        long i = t - start[r];                 /* index inside this request's new tokens */
        long hist = seq_lens[r] - query_lens[r];
        long last_key = hist + i;              /* causal: keys 0 .. hist + i */
        int kvh = h / group;
        const uint16_t *qrow = q + ((size_t)t * num_q_heads + h) * head_dim;
        long nkeys = last_key + 1;
        double *score = (double *)malloc(sizeof(double) * (size_t)nkeys);
        if (!score) {
#pragma omp atomic write
            status = -5;
            continue;
        }
        int bad = 0;
        double mx = -INFINITY;
        for (long j = 0; j < nkeys; ++j) {
            int32_t page = block_table[(size_t)r * max_blocks + j / page_size];
            if (page < 0 || page >= num_pages) {
                bad = 1;
                break;
            }
            const uint16_t *krow = k_cache + (((size_t)page * num_kv_heads + kvh) * page_size +
                                              j % page_size) * head_dim;
            double dot = 0.0;
            for (int x = 0; x < head_dim; ++x)
                dot += widen_bf16(qrow[x]) * widen_bf16(krow[x]);
            score[j] = dot * scale;
            if (score[j] > mx)
                mx = score[j];
        }
        if (bad) {
            free(score);
#pragma omp atomic write
            status = -4;
            continue;
        }
        double denom = 0.0;
        for (long j = 0; j < nkeys; ++j) {
            score[j] = exp(score[j] - mx);
            denom += score[j];
        }
        for (int x = 0; x < head_dim; ++x)
            o[x] = 0.0;
        for (long j = 0; j < nkeys; ++j) {
            int32_t page = block_table[(size_t)r * max_blocks + j / page_size];
            const uint16_t *vrow = v_cache + (((size_t)page * num_kv_heads + kvh) * page_size +
                                              j % page_size) * head_dim;
            double p = score[j] / denom;
            for (int x = 0; x < head_dim; ++x)
                o[x] += p * widen_bf16(vrow[x]);
        }
        free(score);
    }
    free(start);
    return status;
}

/* Number of OpenMP threads the oracle uses (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

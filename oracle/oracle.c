/*
 * Reference oracle for paged decode attention: plain, slow, fp64, on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. The library never calls this code; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg load it. It
 * shares no code, header or table with the CUDA path.
 *
 * What it computes, and where the pages fix it:
 *   - A sequence's tokens live in fixed-size blocks of one pool
 *     ("Building a minimal vLLM implementation", config.py:
 *     kvcache_block_size), found through the sequence's block_table, the map
 *     from logical to physical blocks (same page, sequence.py: block_table).
 *     Logical token t of a sequence therefore sits in physical block
 *     block_table[t / block_size], at row t % block_size of that block.
 *   - The pool is [num_blocks, block_size, num_kv_heads, head_dim] bf16, so a
 *     cache "slot" block * block_size + offset names one contiguous row of
 *     num_kv_heads * head_dim values (the reading this build takes of the
 *     slot_mapping that the store writes through; the pages print no layout).
 *   - Decode sends one new token per sequence ("Building a minimal vLLM
 *     implementation", sequence.py __getstate__: only the last token leaves
 *     for the workers in decode), so each query head has one query row and
 *     attends to all context_lens[s] tokens of its sequence.
 *   - Attention is plain scaled dot-product attention, softmax(q K^T * scale) V,
 *     per query head. Query head h reads KV head h / (Hq / Hkv) (grouped-query
 *     attention with consecutive groups). The pages state no formula; this is
 *     the standard definition.
 *   - A sequence of length 0 has nothing to attend to; its output is zero.
 *
 * Everything is computed in double: bf16 inputs widen exactly, scores, the
 * softmax and the weighted sum are double, and the output is double.
 *
 * Each (sequence, query head) output is independent of every other; the
 * optional OpenMP loop hands whole outputs to threads and changes no
 * arithmetic inside any of them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#include "oracle.h"

/* bf16 is the upper half of an IEEE binary32: widening is a 16-bit shift. */
static double bf16_to_double(uint16_t x)
{
    uint32_t bits = ((uint32_t)x) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int oracle_store_kvcache_layout(const uint16_t *k, const uint16_t *v,
                                uint16_t *k_cache, uint16_t *v_cache,
                                const int64_t *slot_mapping, int64_t num_tokens,
                                int num_kv_heads, int head_dim, int block_size,
                                int64_t num_blocks, int layout)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return ORACLE_ERR_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    const int64_t num_slots = num_blocks * block_size;
    /* check every slot before writing anything */
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < -1 || slot >= num_slots)
            return ORACLE_ERR_RANGE;
    }
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot == -1)
            continue; /* padding entry: nothing is written */
        if (layout == ORACLE_LAYOUT_HEAD_MAJOR) {
            /* [block][kv head][offset]: the row's heads land block_size rows apart */
            const int64_t block = slot / block_size, off = slot % block_size;
            for (int h = 0; h < num_kv_heads; ++h) {
                const int64_t dst = ((block * num_kv_heads + h) * block_size + off) * head_dim;
                memcpy(k_cache + dst, k + i * row + (int64_t)h * head_dim,
                       (size_t)head_dim * sizeof(uint16_t));
                memcpy(v_cache + dst, v + i * row + (int64_t)h * head_dim,
                       (size_t)head_dim * sizeof(uint16_t));
            }
            continue;
        }
        memcpy(k_cache + slot * row, k + i * row, (size_t)row * sizeof(uint16_t));
        memcpy(v_cache + slot * row, v + i * row, (size_t)row * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

int oracle_store_kvcache(const uint16_t *k, const uint16_t *v,
                         uint16_t *k_cache, uint16_t *v_cache,
                         const int64_t *slot_mapping, int64_t num_tokens,
                         int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks)
{
    return oracle_store_kvcache_layout(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                       num_kv_heads, head_dim, block_size, num_blocks,
                                       ORACLE_LAYOUT_TOKEN_MAJOR);
}

/* One output row: query head h of query row q_index, attending to the first
 * min(context_lens[s], cap) tokens of sequence s, written to out[0..head_dim).
 * Single-token decode has q_index = s and cap = context_lens[s]. */
static int decode_one(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, double scale,
                      int s, int h, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int64_t num_blocks, int q_index, int cap, int layout,
                      double *out)
{
    const int group = num_q_heads / num_kv_heads;
    const int kvh = h / group;
    const int L = context_lens[s] < 0 || context_lens[s] <= cap ? context_lens[s]
                                                                 : (cap > 0 ? cap : 0);
    const uint16_t *qrow = q + ((int64_t)q_index * num_q_heads + h) * head_dim;

    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (L == 0)
        return ORACLE_OK;
    if (L < 0 || (int64_t)(L + block_size - 1) / block_size > max_blocks_per_seq)
        return ORACLE_ERR_RANGE;

    double *score = (double *)malloc((size_t)L * sizeof(double));
    if (!score)
        return ORACLE_ERR_ARG;

    /* scores: s_t = scale * sum_d q_d * K_t,d, K_t gathered through the table */
    for (int t = 0; t < L; ++t) {
        int64_t block = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
        if (block < 0 || block >= num_blocks) {
            free(score);
            return ORACLE_ERR_RANGE;
        }
        const uint16_t *krow = layout == ORACLE_LAYOUT_HEAD_MAJOR
            ? k_cache + ((block * num_kv_heads + kvh) * block_size + t % block_size) * (int64_t)head_dim
            : k_cache + ((block * block_size + t % block_size) * num_kv_heads + kvh) * (int64_t)head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += bf16_to_double(qrow[d]) * bf16_to_double(krow[d]);
        score[t] = scale * dot;
    }

    /* softmax over the L scores, shifted by their maximum */
    double mx = score[0];
    for (int t = 1; t < L; ++t)
        if (score[t] > mx)
            mx = score[t];
    double denom = 0.0;
    for (int t = 0; t < L; ++t) {
        score[t] = exp(score[t] - mx);
        denom += score[t];
    }

    /* out = sum_t p_t V_t, V_t gathered the same way as K_t */
    for (int t = 0; t < L; ++t) {
        int64_t block = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
        const uint16_t *vrow = layout == ORACLE_LAYOUT_HEAD_MAJOR
            ? v_cache + ((block * num_kv_heads + kvh) * block_size + t % block_size) * (int64_t)head_dim
            : v_cache + ((block * block_size + t % block_size) * num_kv_heads + kvh) * (int64_t)head_dim;
        double p = score[t] / denom;
        for (int d = 0; d < head_dim; ++d)
            out[d] += p * bf16_to_double(vrow[d]);
    }
    free(score);
    return ORACLE_OK;
}

static int check_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int max_blocks_per_seq)
{
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq < 0 || num_q_heads % num_kv_heads != 0)
        return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

int oracle_decode_layout(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, double scale, double *out,
                         int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, int layout, int num_threads)
{
    int rc = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq);
    if (rc != ORACLE_OK)
        return rc;
    const int64_t total = (int64_t)num_seqs * num_q_heads;
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int64_t i = 0; i < total; ++i) {
        const int s = (int)(i / num_q_heads);
        int r = decode_one(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           scale, s, (int)(i % num_q_heads), num_q_heads, num_kv_heads,
                           head_dim, block_size, num_blocks, s, context_lens[s], layout,
                           out + i * head_dim);
        if (r != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            err = r;
        }
    }
    (void)num_threads;
    return err;
}

int oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *context_lens, double scale, double *out,
                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                  int block_size, int64_t num_blocks, int num_threads)
{
    return oracle_decode_layout(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, scale, out, num_seqs, num_q_heads, num_kv_heads,
                                head_dim, block_size, num_blocks, ORACLE_LAYOUT_TOKEN_MAJOR,
                                num_threads);
}

int oracle_decode_pairs(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, double scale,
                        const int32_t *pairs, int64_t num_pairs, double *out,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int64_t num_blocks, int num_threads)
{
    int rc = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq);
    if (rc != ORACLE_OK)
        return rc;
    for (int64_t i = 0; i < num_pairs; ++i)
        if (pairs[2 * i] < 0 || pairs[2 * i] >= num_seqs || pairs[2 * i + 1] < 0 ||
            pairs[2 * i + 1] >= num_q_heads)
            return ORACLE_ERR_RANGE;
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int64_t i = 0; i < num_pairs; ++i) {
        int r = decode_one(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           scale, pairs[2 * i], pairs[2 * i + 1], num_q_heads, num_kv_heads,
                           head_dim, block_size, num_blocks, pairs[2 * i],
                           context_lens[pairs[2 * i]], ORACLE_LAYOUT_TOKEN_MAJOR,
                           out + i * head_dim);
        if (r != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            err = r;
        }
    }
    (void)num_threads;
    return err;
}

/*
 * Several new tokens per sequence (the verification step of speculative
 * decoding, "Implementation Details", Speculative Decoding -- EAGLE Proposer:
 * draft tokens are checked by the target model in one pass). Query token i of
 * the q_len new tokens of sequence s sits at position L - q_len + i, where L =
 * context_lens[s] counts them all, and attends causally to tokens
 * t <= L - q_len + i; a query with no such token outputs zero.
 * q and out are [num_seqs, q_len, num_q_heads, head_dim].
 */
int oracle_decode_multi(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, int q_len, double scale, double *out,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int64_t num_blocks, int num_threads)
{
    int rc = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq);
    if (rc != ORACLE_OK)
        return rc;
    if (q_len < 1)
        return ORACLE_ERR_ARG;
    const int64_t total = (int64_t)num_seqs * q_len * num_q_heads;
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int64_t r_i = 0; r_i < total; ++r_i) {
        const int64_t row = r_i / num_q_heads;          /* s * q_len + i */
        const int s = (int)(row / q_len), i = (int)(row % q_len);
        const int cap = context_lens[s] - q_len + i + 1;
        int r = decode_one(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           scale, s, (int)(r_i % num_q_heads), num_q_heads, num_kv_heads,
                           head_dim, block_size, num_blocks, (int)row, cap,
                           ORACLE_LAYOUT_TOKEN_MAJOR, out + r_i * head_dim);
        if (r != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            err = r;
        }
    }
    (void)num_threads;
    return err;
}

/*
 * Prefill of a chunk of new tokens per sequence over the paged cache (the
 * prompt phase, "A vLLM engine small enough to read in one sitting": prefill
 * and decode both run over the paged KV cache). The rows of q are packed
 * sequence after sequence: sequence s owns rows [query_start_loc[s],
 * query_start_loc[s + 1]); with n_s of them, row i of the sequence is the
 * token at position context_lens[s] - n_s + i and attends causally to tokens
 * t <= context_lens[s] - n_s + i (all of them stored in the cache). q and out
 * are [total_q, num_q_heads, head_dim].
 */
int oracle_prefill(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                   const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *context_lens, const int32_t *query_start_loc, double scale,
                   double *out, int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                   int head_dim, int block_size, int64_t num_blocks, int num_threads)
{
    int rc = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq);
    if (rc != ORACLE_OK)
        return rc;
    if (total_q < 0 || query_start_loc[0] != 0 || query_start_loc[num_seqs] != total_q)
        return ORACLE_ERR_ARG;
    for (int s = 0; s < num_seqs; ++s)
        if (query_start_loc[s + 1] < query_start_loc[s])
            return ORACLE_ERR_ARG;
    const int64_t total = (int64_t)total_q * num_q_heads;
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 16) num_threads(num_threads)
#endif
    for (int64_t r_i = 0; r_i < total; ++r_i) {
        const int row = (int)(r_i / num_q_heads);
        int s = 0;
        while (query_start_loc[s + 1] <= row)
            ++s;
        const int n = query_start_loc[s + 1] - query_start_loc[s];
        const int i = row - query_start_loc[s];
        const int cap = context_lens[s] - n + i + 1;
        int r = decode_one(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           scale, s, (int)(r_i % num_q_heads), num_q_heads, num_kv_heads,
                           head_dim, block_size, num_blocks, row, cap,
                           ORACLE_LAYOUT_TOKEN_MAJOR, out + r_i * head_dim);
        if (r != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            err = r;
        }
    }
    (void)num_threads;
    return err;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Reference oracle for paged decode attention (fp64, CPU).
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the library.
 *
 * All arrays are host memory, row-major and contiguous:
 *   q            bf16 bits [num_seqs, num_q_heads, head_dim]
 *   k, v         bf16 bits [num_tokens, num_kv_heads, head_dim]
 *   k_cache,
 *   v_cache      bf16 bits [num_blocks, block_size, num_kv_heads, head_dim]
 *   slot_mapping int64 [num_tokens]; -1 = skip, else block * block_size + offset
 *   block_tables int32 [num_seqs, max_blocks_per_seq]
 *   context_lens int32 [num_seqs]
 *   out          double [num_seqs, num_q_heads, head_dim]
 */
#ifndef PAGED_DECODE_ORACLE_H
#define PAGED_DECODE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_OK = 0, ORACLE_ERR_ARG = 1, ORACLE_ERR_RANGE = 2 };

/* Pool layouts: token-major [num_blocks][block_size][num_kv_heads][head_dim]
 * (the default), head-major [num_blocks][num_kv_heads][block_size][head_dim]. */
enum { ORACLE_LAYOUT_TOKEN_MAJOR = 0, ORACLE_LAYOUT_HEAD_MAJOR = 1 };

/* Copy row i of k and v to cache slot slot_mapping[i]; -1 rows are skipped.
 * Nothing is written if any slot is out of range. */
int oracle_store_kvcache(const uint16_t *k, const uint16_t *v,
                         uint16_t *k_cache, uint16_t *v_cache,
                         const int64_t *slot_mapping, int64_t num_tokens,
                         int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks);

/* softmax(q K^T * scale) V per (sequence, query head) over the sequence's
 * context_lens[s] tokens, gathered through its block table.
 * num_threads <= 0 uses every OpenMP thread. */
int oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *context_lens, double scale, double *out,
                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                  int block_size, int64_t num_blocks, int num_threads);

/* The same, for the listed (sequence, query head) pairs only:
 * pairs int32 [num_pairs, 2], out double [num_pairs, head_dim]. */
int oracle_decode_pairs(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, double scale,
                        const int32_t *pairs, int64_t num_pairs, double *out,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int64_t num_blocks, int num_threads);

/* Several new tokens per sequence: query token i of the q_len new tokens of
 * sequence s attends causally to tokens t <= context_lens[s] - q_len + i.
 * q and out are [num_seqs, q_len, num_q_heads, head_dim]. */
int oracle_decode_multi(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, int q_len, double scale, double *out,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int64_t num_blocks, int num_threads);

/* The store and decode above for a pool in either layout. */
int oracle_store_kvcache_layout(const uint16_t *k, const uint16_t *v,
                                uint16_t *k_cache, uint16_t *v_cache,
                                const int64_t *slot_mapping, int64_t num_tokens,
                                int num_kv_heads, int head_dim, int block_size,
                                int64_t num_blocks, int layout);
int oracle_decode_layout(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, double scale, double *out,
                         int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, int layout, int num_threads);

/* Prefill: rows [query_start_loc[s], query_start_loc[s + 1]) of q belong to
 * sequence s; with n_s of them, row i is the token at position
 * context_lens[s] - n_s + i and attends to tokens t <= that position.
 * q and out are [total_q, num_q_heads, head_dim]. */
int oracle_prefill(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                   const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *context_lens, const int32_t *query_start_loc, double scale,
                   double *out, int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                   int head_dim, int block_size, int64_t num_blocks, int num_threads);

/* Threads the OpenMP loops use by default. */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif

#endif

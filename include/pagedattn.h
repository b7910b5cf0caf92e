/*
 * libpagedattn -- paged KV-cache store, decode attention (one or several new
 * tokens per sequence) and paged prefill attention, for NVIDIA GB300 (sm_103a).
 *
 * The operations follow the pages that describe a minimal vLLM engine:
 *   - KV is kept in fixed-size token blocks of one pool
 *     ("Building a minimal vLLM implementation", config.py, kvcache_block_size);
 *   - each sequence's block_table maps its logical blocks to physical blocks
 *     (same page, sequence.py, block_table);
 *   - block 0 of the pool is a reserved null block that no sequence owns
 *     ("Implementation Details", PagedAttention -- BlockPool);
 *   - decode runs one new token per sequence (sequence.py __getstate__:
 *     in decode only the last token is sent to the workers);
 *   - the decode kernel is the engine's paged-attention kernel
 *     ("A vLLM engine small enough to read in one sitting", What it does /
 *     Key highlights: paged attention for decoding).
 *
 * Layouts (all row-major, contiguous, bf16 = IEEE bfloat16):
 *   q            [num_seqs, num_q_heads, head_dim]                 bf16
 *   k, v         [num_tokens, num_kv_heads, head_dim]              bf16
 *   k_cache,
 *   v_cache      [num_blocks, block_size, num_kv_heads, head_dim]  bf16
 *   slot_mapping [num_tokens] int64; slot = block * block_size + offset, -1 = skip
 *   block_tables [num_seqs, max_blocks_per_seq] int32 physical block ids
 *   context_lens [num_seqs] int32, tokens of each sequence, counting the one
 *                just stored
 *   out          [num_seqs, num_q_heads, head_dim]                 bf16
 * Query head h reads KV head h / (num_q_heads / num_kv_heads). The *_layout
 * calls also take the head-major pool [num_blocks, num_kv_heads, block_size,
 * head_dim]; pa_decode_multi and pa_prefill take their q and out shapes as
 * described at each call.
 *
 * Ownership: every pointer is caller-owned memory on the current CUDA device
 * (the workspace included). The library allocates nothing and keeps no data
 * between calls; its only process-wide state is the NVTX domain handle (see
 * Tracing), the static scratch of pa_decode_noalloc, the test hooks, and per
 * device the SM count and the decode's worker counts, computed on the first
 * call on that device. Calls are
 * asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 * stream) and return once the kernels are queued.
 *
 * Tracing: every call that launches work (and pa_take_device_error) opens one
 * NVTX range named after itself, in the NVTX domain "libpagedattn", for as
 * long as it runs on the host; the kernels it queues carry that range in
 * Nsight tools (e.g. `ncu --nvtx --nvtx-include "libpagedattn@pa_decode/"`).
 * pa_decode_noalloc shows as pa_decode. With no tool attached a range costs a
 * test of a function pointer.
 *
 * Errors: argument problems are found on the host, before anything is
 * launched, and returned as a status. Index values the kernels read on the
 * device (slots, block ids, lengths) are never trusted for addressing: a slot
 * outside [-1, num_blocks * block_size) writes nothing, a block id outside
 * [0, num_blocks) reads as zero rows (keys that score 0 and add a zero value),
 * a length is clamped to [0, max_blocks_per_seq * block_size]. Such inputs
 * never touch memory outside the buffers passed in, and the first two are
 * recorded on the device for pa_take_device_error.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer */
    PA_ERR_UNSUPPORTED = 2,   /* head_dim != 128, block_size, group size   */
    PA_ERR_WORKSPACE = 3,     /* workspace missing or too small            */
    PA_ERR_CUDA = 4           /* a CUDA call or launch failed              */
} pa_status_t;

/* KV pool layouts. Token-major is the default of every call that takes no
 * layout argument. */
typedef enum {
    PA_LAYOUT_TOKEN_MAJOR = 0,  /* [num_blocks, block_size, num_kv_heads, head_dim] */
    PA_LAYOUT_HEAD_MAJOR = 1    /* [num_blocks, num_kv_heads, block_size, head_dim] */
} pa_layout_t;

/* Human-readable name of a status. Never NULL. */
PA_API const char *pa_status_string(pa_status_t status);

/*
 * Store new K/V rows into the paged cache.
 *
 * For every i < num_tokens with slot_mapping[i] != -1:
 *   k_cache viewed as [num_blocks * block_size, num_kv_heads * head_dim],
 *   row slot_mapping[i], becomes k[i]; the same for v / v_cache.
 * Rows with slot -1 (batch padding) write nothing. The copy is bit-exact.
 * Two rows with the same slot: the value left there is unspecified.
 *
 * This is how a decode step puts the token it has just projected into the
 * block its sequence's block_table names (the write side of the paged KV
 * cache, "A vLLM engine small enough to read in one sitting": paged KV cache
 * management).
 *
 * Requirements: head_dim == 128; block_size a power of two in [16, 256];
 * all pointers 16-byte aligned (non-null unless num_tokens == 0).
 */
PA_API pa_status_t pa_store_kvcache(const void *k, const void *v,
                             void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int64_t num_tokens,
                             int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks, void *stream);

/*
 * Bytes of device workspace pa_decode needs on the current device for this
 * head configuration, with num_partitions = 0 (automatic) or a forced count
 * (see pa_decode_splitk). Returns 0 for an unsupported configuration.
 */
PA_API size_t pa_decode_workspace_size(int num_q_heads, int num_kv_heads, int head_dim,
                                int num_partitions);

/*
 * Single-token decode attention over the paged cache.
 *
 * For each sequence s and query head h, with L = context_lens[s],
 * kvh = h / (num_q_heads / num_kv_heads) and, for t < L,
 *   K_t = k_cache[block_tables[s][t / block_size]][t % block_size][kvh]
 *   V_t = v_cache[ ... same ... ]:
 *   out[s][h] = sum_t softmax_t(scale * q[s][h] . K_t) V_t
 * computed in fp32 from the bf16 inputs and rounded to bf16. L == 0 gives 0.
 * Only the first ceil(L / block_size) entries of a table row are read, and
 * within the last block only its first L - (blocks - 1) * block_size rows.
 *
 * The work is cut into contiguous, equal shares of all sequences' 16-token
 * tiles (split-K / flash-decoding); a (sequence, KV head) whose tiles span
 * several shares is finished by a log-sum-exp combine launched after the main
 * kernel on the same stream. The workspace holds those partial results; its
 * contents need no initialisation and are garbage after the call.
 *
 * Requirements: head_dim == 128; num_q_heads % num_kv_heads == 0 with group
 * size num_q_heads / num_kv_heads <= 16; block_size a power of two in
 * [16, 256]; q, k_cache, v_cache, out 16-byte aligned; workspace of at least
 * pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim, 0) bytes,
 * 16-byte aligned; num_blocks * block_size and num_blocks * num_kv_heads
 * below 2^31 (the tile copies address pool rows with 32-bit coordinates;
 * PA_ERR_UNSUPPORTED otherwise).
 */
PA_API pa_status_t pa_decode(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, float scale, void *out,
                      int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int64_t num_blocks,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_decode with the number of partitions (split-K shares) forced to
 * num_partitions >= 1 instead of chosen from the device; num_partitions == 0
 * is pa_decode. For tests of the combine path and for tuning. The workspace
 * must hold pa_decode_workspace_size(..., num_partitions) bytes.
 */
PA_API pa_status_t pa_decode_splitk(const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, float scale, void *out,
                             int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int64_t num_blocks,
                             void *workspace, size_t workspace_bytes,
                             int num_partitions, void *stream);

/*
 * Decode for callers that cannot allocate device memory. The pages have no
 * counterpart of this call.
 *
 * pa_decode needs a caller-provided workspace. Some callers cannot provide
 * one: they may not call cudaMalloc (or any allocator) on their path, for
 * example because the call sits in a loop that must not block on the
 * allocator, or because device memory belongs to a host framework that only
 * passes in the input and output buffers. This entry point takes the same
 * inputs and output as pa_decode and allocates nothing: its scratch (the
 * split-K partial results and combine tasks) is one file-scope array of
 * PA_NOALLOC_SCRATCH_BYTES bytes in device global memory, which every GPU
 * that loads the library holds until the process exits.
 *
 * - The first call on a device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture. The cached address belongs to the CUDA context that was
 *   current then: after cudaDeviceReset (or any reset of the device's
 *   primary context) the library's module is loaded again at a new address,
 *   so this call is not supported after such a reset in the same process.
 * - Every call shares the one array. Nothing in it needs to start at zero
 *   (each call writes every word it later reads), but calls that overlap on
 *   the GPU (on different streams, or from different threads) race on it
 *   and give wrong results: serialise them.
 * - A head configuration whose scratch would exceed the array
 *   (pa_decode_workspace_size(...) > PA_NOALLOC_SCRATCH_BYTES; on a 152-SM
 *   GB300 that is a group size above 8) returns PA_ERR_WORKSPACE and
 *   launches nothing.
 * Argument checks and their statuses are pa_decode's (an empty batch
 * returns PA_OK without touching a device); a failed device query returns
 * PA_ERR_CUDA. Results are bit-identical to pa_decode's for the same inputs
 * on the same device.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
PA_API pa_status_t pa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, int max_blocks_per_seq,
                                     const int32_t *context_lens, float scale, void *out,
                                     int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int64_t num_blocks,
                                     void *stream);

/*
 * Decode of several new tokens per sequence at once: the verification pass of
 * speculative decoding, where the target model checks q_len draft tokens of
 * each sequence in one step ("Implementation Details", Speculative Decoding --
 * EAGLE Proposer: draft tokens proposed, then verified by the target model).
 *
 * q and out are [num_seqs, q_len, num_q_heads, head_dim] bf16. context_lens[s]
 * counts all q_len new tokens (they are stored in the cache before the call,
 * e.g. with pa_store_kvcache); query token i sits at position
 * context_lens[s] - q_len + i and attends causally to tokens
 * t <= context_lens[s] - q_len + i, gathered as in pa_decode. A query token
 * with no such token outputs zero. q_len = 1 is pa_decode.
 *
 * Requirements: as pa_decode, plus 1 <= q_len and q_len * (num_q_heads /
 * num_kv_heads) <= 16; the workspace must hold
 * pa_decode_multi_workspace_size(q_len, ...) bytes. Always the tensor-core path.
 */
PA_API size_t pa_decode_multi_workspace_size(int q_len, int num_q_heads, int num_kv_heads,
                                             int head_dim);
PA_API pa_status_t pa_decode_multi(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *context_lens, int q_len, float scale,
                                   void *out, int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_blocks,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_store_kvcache and pa_decode_splitk for a pool in either layout. In the
 * head-major layout a block keeps each KV head's block_size rows together,
 * so a 16-token K (or V) tile of one head is one contiguous 4 KB run instead
 * of 16 rows of 256 B spread num_kv_heads rows apart; slots and block tables
 * mean the same in both layouts (slot = block * block_size + offset), and the
 * results are identical. num_partitions = 0 chooses the share count from the
 * device, as pa_decode. The pages fix no layout; the token-major one is the
 * plainest reading of a slot_mapping store, the head-major one is offered for
 * its contiguous tiles.
 */
PA_API pa_status_t pa_store_kvcache_layout(const void *k, const void *v,
                                           void *k_cache, void *v_cache,
                                           const int64_t *slot_mapping, int64_t num_tokens,
                                           int num_kv_heads, int head_dim, int block_size,
                                           int64_t num_blocks, pa_layout_t layout, void *stream);
PA_API pa_status_t pa_decode_layout(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_tables, int max_blocks_per_seq,
                                    const int32_t *context_lens, float scale, void *out,
                                    int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int64_t num_blocks,
                                    pa_layout_t layout, void *workspace, size_t workspace_bytes,
                                    int num_partitions, void *stream);
/* pa_decode_multi for a pool in either layout (same workspace size). */
PA_API pa_status_t pa_decode_multi_layout(const void *q, const void *k_cache, const void *v_cache,
                                          const int32_t *block_tables, int max_blocks_per_seq,
                                          const int32_t *context_lens, int q_len, float scale,
                                          void *out, int num_seqs, int num_q_heads,
                                          int num_kv_heads, int head_dim, int block_size,
                                          int64_t num_blocks, pa_layout_t layout, void *workspace,
                                          size_t workspace_bytes, void *stream);

/*
 * One decode step in one call: the store of the step's new K/V rows
 * (pa_store_kvcache_layout with k, v, slot_mapping, num_tokens), then
 * single-token decode attention over the updated cache (pa_decode_layout
 * with num_partitions = 0), on `stream`. This is how the engine the pages
 * describe runs a decode step: the token just projected is written into its
 * sequence's block, then attention reads the whole sequence back through the
 * block table ("A vLLM engine small enough to read in one sitting": paged KV
 * cache management and paged attention for decoding).
 *
 * The results are exactly those of the two calls made one after the other.
 * What the single call adds: the decode kernel's only predecessor is then
 * this store, which writes the caches and nothing else, so the decode plans
 * its split of the work (from context_lens) while the store still runs and
 * waits for the store only before its first cache read. context_lens,
 * block_tables and q must therefore not overlap k_cache or v_cache.
 *
 * Every argument of both parts is checked before anything is launched; the
 * statuses are those of the two calls (the store's checks first). With
 * num_tokens == 0 only the decode runs; with num_seqs == 0 only the store.
 * The workspace is pa_decode's (pa_decode_workspace_size(..., 0)).
 */
PA_API pa_status_t pa_decode_step(const void *k, const void *v, const int64_t *slot_mapping,
                                  int64_t num_tokens, const void *q, void *k_cache,
                                  void *v_cache, const int32_t *block_tables,
                                  int max_blocks_per_seq, const int32_t *context_lens,
                                  float scale, void *out, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int64_t num_blocks, pa_layout_t layout, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * Paged prefill (chunked prefill): a chunk of new tokens per sequence attends
 * causally to the sequence's tokens in the paged cache, as in the engine's
 * prefill phase ("A vLLM engine small enough to read in one sitting": prefill
 * and decode over the paged KV cache, flash attention for prefill).
 *
 * q and out are [total_q, num_q_heads, head_dim] bf16, rows packed sequence
 * after sequence: sequence s owns rows [query_start_loc[s],
 * query_start_loc[s + 1]) (query_start_loc: int32 [num_seqs + 1] on the device,
 * starting at 0 and non-decreasing). With n_s rows and L = context_lens[s]
 * counting them (their K/V already stored, e.g. by pa_store_kvcache), row i of
 * sequence s is the token at position L - n_s + i and, for query head h,
 *   out = sum_{t <= L - n_s + i} softmax_t(scale * q . K_t) V_t
 * with K_t, V_t of KV head h / (num_q_heads / num_kv_heads) gathered through the
 * block table. A row with no visible token outputs zero. max_query_len is a
 * host-side hint for the grid (the largest n_s; a smaller value is still
 * correct, only slower). Token-major pool layout; group size <= 16; head_dim
 * 128; num_seqs and num_kv_heads at most 65535; the pool-size limit of
 * pa_decode. Computes in fp32 on the tensor cores, output bf16. Allocates
 * nothing.
 */
PA_API pa_status_t pa_prefill(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, const int32_t *query_start_loc,
                              int max_query_len, float scale, void *out, int num_seqs,
                              int total_q, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int64_t num_blocks, void *stream);

/*
 * pa_prefill on a pool in either layout: PA_LAYOUT_TOKEN_MAJOR
 * [NB, bs, Hkv, head_dim] (what pa_prefill takes) or PA_LAYOUT_HEAD_MAJOR
 * [NB, Hkv, bs, head_dim] (the layout pa_store_kvcache_layout and
 * pa_decode_layout also take). Same results for the same values in either
 * layout; PA_ERR_INVALID_ARG for another layout value.
 */
PA_API pa_status_t pa_prefill_layout(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, int max_blocks_per_seq,
                                     const int32_t *context_lens, const int32_t *query_start_loc,
                                     int max_query_len, float scale, void *out, int num_seqs,
                                     int total_q, int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, int64_t num_blocks, pa_layout_t layout,
                                     void *stream);

/*
 * Device-side error record. The kernels do not fault or hang on their inputs:
 * an index outside its range is handled in a defined way, and every mbarrier
 * wait is bounded (the prefill kernel's hand-offs between its warps, about
 * 2 s; a decode warp's wait for its own tile copies, about 1 s). Each such
 * event is recorded on the device, the first code of each kernel kind kept,
 * without any synchronization in the calls themselves.
 * This call synchronizes `stream`, stores the smallest recorded code in *code
 * and clears every record:
 *   0  none;
 *   1  pa_prefill: shared memory not 1024-byte aligned; the launch's outputs
 *      are undefined;
 *   2  pa_prefill, or any decode call: a bounded wait ran out; the launch's
 *      outputs are undefined;
 *   3  pa_store_kvcache: a slot outside [-1, num_blocks * block_size) was
 *      skipped; nothing is written for that row;
 *   4  pa_decode / pa_decode_multi / pa_prefill: a block-table entry that
 *      covers context tokens lies outside [0, num_blocks); its rows are read
 *      as zeros, so each of those keys scores 0 and adds a zero value.
 * Entries past a sequence's last block are never read and never reported.
 */
PA_API pa_status_t pa_take_device_error(int32_t *code, void *stream);

/*
 * Test hook for the error path above, off by default: with mode 1, later
 * pa_prefill / pa_prefill_layout launches (tcgen05 kernel) hold back one
 * barrier arrival of their V producer, so that a wait runs out after about 2 s
 * and the launch records code 2 and returns, its outputs undefined; mode 0
 * restores normal launches. Process-wide; for tests only.
 */
PA_API pa_status_t pa_debug_prefill_fault(int mode);

/*
 * Test hook, off by default: run the comparison kernels the library keeps
 * for testing instead of the product kernels. flags is 0 (the product
 * kernels) or an OR of
 *   PA_VARIANT_DECODE_SIMT  decode tiles on the CUDA cores instead of the
 *                           tensor cores (single-token decode, group size
 *                           <= 8; other calls keep the tensor cores);
 *   PA_VARIANT_PREFILL_MMA  pa_prefill on the mma.sync kernel instead of the
 *                           tcgen05 kernel.
 * Both compute the same results within the tolerance of the product kernels;
 * the tests use them as a second parity path. Process-wide, read at each
 * call; PA_ERR_INVALID_ARG for an unknown bit. Not for production use.
 */
#define PA_VARIANT_DECODE_SIMT 1
#define PA_VARIANT_PREFILL_MMA 2
PA_API pa_status_t pa_debug_kernel_variant(int flags);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */

// Internal launchers behind the C ABI (not part of the public header).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/pagedattn.h"

namespace pa {

constexpr int kHeadDimPublic = 128;   // head_dim the ABI accepts
constexpr int kDefaultMinTiles = 4;   // automatic shares hold at least this many 16-token tiles

// Tile computation inside the decode worker: tensor cores (mma.sync) or CUDA cores.
enum class DecodeKernel { kMma = 0, kSimt = 1 };

// Everything one paged-decode launch needs. Pointers are device memory.
struct DecodeArgs {
    const void *q;              // bf16 [S, Hq, 128]
    const void *k_cache;        // bf16 [NB, bs, Hkv, 128]
    const void *v_cache;
    const int32_t *block_tables;  // [S, max_blocks_per_seq]
    const int32_t *context_lens;  // [S]
    void *out;                  // bf16 [S, Hq, 128]
    float *part_o;              // [2P, GP, 128] unnormalised partial outputs
    float *part_ml;             // [2P, GP, 2]   (running max in log2 units, sum)
    int4 *tasks;                // [P] combine task of each worker
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;                  // Hq / Hkv
    int q_len;                  // query tokens per sequence (1: plain decode)
    int cols;                   // q_len * group: (query token, head) columns per KV head
    int block_size_log2;
    int head_major;             // pool layout: 0 [NB, bs, Hkv, D], 1 [NB, Hkv, bs, D]
    int max_blocks_per_seq;
    int64_t num_blocks;
    float scale_log2;           // scale * log2(e)
    int num_workers;            // P: contiguous shares of the tile space
    int min_tiles;              // fewest tiles a share may hold (1 = exactly P shares)
    int plan_early;             // the previous kernel writes only the caches: plan before waiting on it
};

// Host-side argument checks of the store entry points (no CUDA call); PA_OK
// with *nothing_to_do set for an empty batch.
pa_status_t store_check_args(const void *k, const void *v, const void *k_cache,
                             const void *v_cache, const int64_t *slot_mapping, int64_t num_tokens,
                             int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                             int layout, bool *nothing_to_do);

// Host-side argument checks of every decode entry point, in the order the
// calls apply them (pointers, sizes, layout, head_dim, block size, group
// size; no CUDA call). PA_OK with *nothing_to_do set for an empty batch.
pa_status_t decode_check_args(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int q_len, float scale,
                              const void *out, int num_seqs, int num_q_heads, int num_kv_heads,
                              int head_dim, int block_size, int64_t num_blocks, int layout,
                              int num_partitions, bool *nothing_to_do);

// Padded group size the kernels are instantiated for (power of two >= group,
// at most 16), or 0 when unsupported.
int decode_group_pad(int group);

// Workers (shares) per device when the caller does not force a count.
int decode_default_workers(int group_pad, DecodeKernel k, int sm_count);

// Workspace bytes for P workers at padded group size GP.
size_t decode_workspace_bytes(int group_pad, int num_workers);

// Carve the workspace into DecodeArgs' part_o / part_ml / tasks.
void decode_carve_workspace(DecodeArgs &a, void *workspace, int group_pad);

cudaError_t launch_decode(const DecodeArgs &a, int group_pad, DecodeKernel k, cudaStream_t stream);

// One paged-prefill launch (pointers are device memory).
struct PrefillArgs {
    const void *q;                  // bf16 [total_q, Hq, 128], rows packed per sequence
    const void *k_cache;            // bf16 [NB, bs, Hkv, 128]
    const void *v_cache;
    const int32_t *block_tables;    // [S, max_blocks_per_seq]
    const int32_t *context_lens;    // [S], counting each sequence's new tokens
    const int32_t *query_start_loc; // [S + 1]
    void *out;                      // bf16 [total_q, Hq, 128]
    int num_seqs;
    int total_q;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int block_size_log2;
    int max_blocks_per_seq;
    int head_major;                 // pool layout [NB, Hkv, bs, 128] instead of [NB, bs, Hkv, 128]
    int fault_hold_v;               // test hook, normally 0: see set_prefill_fault
    int64_t num_blocks;
    float scale_log2;
};

// Test hook for the bounded waits of the tcgen05 prefill kernel: with mode 1
// its V producer leaves the first tile's v_full barrier without its arrival,
// so the MMA warp's wait for it runs out (about 2 s), the kernel records error
// 2 and every warp exits. Mode 0 (the default) turns it off.
void set_prefill_fault(int mode);
int prefill_fault();

cudaError_t launch_prefill(const PrefillArgs &a, int group_pad, int max_query_len,
                           cudaStream_t stream);
// The same on tcgen05 (TMEM accumulators); records device-side errors
// (1 = misaligned shared memory, 2 = an mbarrier wait ran out) for
// take_prefill_error.
cudaError_t launch_prefill_tc(const PrefillArgs &a, int group_pad, int max_query_len,
                              cudaStream_t stream);
// Each synchronizes the stream, returns the first code its kernels recorded
// (DeviceError in common.cuh; 0 = none) and clears it.
cudaError_t take_prefill_error(cudaStream_t stream, int *code);
cudaError_t take_prefill_mma_error(cudaStream_t stream, int *code);
cudaError_t take_decode_error(cudaStream_t stream, int *code);
cudaError_t take_store_error(cudaStream_t stream, int *code);

// cuTensorMapEncodeTiled from the driver (nullptr if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// TMA tensor map over a K or V pool (either layout) whose box is one 16-token
// tile of one KV head, 64 head dims wide, 128-byte swizzle; two boxes (x = 0
// and x = 64) make a whole tile. Coordinates: token-major (x, KV head,
// block * bs + offset); head-major (x, offset, block * Hkv + KV head).
bool make_pool_map(CUtensorMap *m, const void *pool, int64_t num_blocks, int block_size,
                   int num_kv_heads, bool head_major);

// TMA tensor map over a K or V pool whose one box is a whole 16-token tile of
// one KV head (both 64-dim halves, the same landing layout as two boxes of
// make_pool_map's map). Coordinates: token-major (0, block * bs + offset, 0,
// KV head); head-major (0, offset, 0, block * Hkv + KV head).
bool make_tile_map(CUtensorMap *m, const void *pool, int64_t num_blocks, int block_size,
                   int num_kv_heads, bool head_major);

cudaError_t launch_store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache,
                                 const int64_t *slot_mapping, int64_t num_tokens,
                                 int num_kv_heads, int head_dim, int block_size_log2,
                                 int64_t num_slots, int head_major, int sm_count,
                                 cudaStream_t stream);

}  // namespace pa

// store_kvcache: scatter new K/V rows into the paged cache through slot_mapping.
//
// Write side of the paged KV cache ("A vLLM engine small enough to read in one
// sitting", paged KV cache management): row i of k/v goes to cache slot
// slot_mapping[i] = block * block_size + offset, where block comes from the
// sequence's block_table ("Building a minimal vLLM implementation",
// sequence.py). One warp copies one row of num_kv_heads * head_dim bf16 for K
// and the same for V with 16-byte loads and stores; -1 rows are skipped.
#include "common.cuh"
#include "kernels.h"

namespace pa {

__device__ int g_store_error;        // first device-side error of a store launch

namespace {

constexpr int kStoreWarps = 8;

template <bool HEAD_MAJOR>
__global__ void __launch_bounds__(kStoreWarps * 32)
store_kvcache_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                     const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                     int num_kv_heads, int head_chunks, int block_size_log2, int64_t num_slots) {
    // let a decode launched as a programmatic dependent start its launch now;
    // it still waits for this grid to finish before reading the cache
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int row_chunks = num_kv_heads * head_chunks;     // 16-byte chunks per row
    const int64_t first = (int64_t)blockIdx.x * kStoreWarps + (threadIdx.x >> 5);
    const int64_t stride = (int64_t)gridDim.x * kStoreWarps;
    for (int64_t i = first; i < num_tokens; i += stride) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0 || slot >= num_slots) {          // -1 padding, or out of range
            if (slot != -1 && lane == 0) atomicCAS(&g_store_error, 0, kErrBadSlot);
            continue;
        }
        const uint4 *ks = k + i * row_chunks;
        const uint4 *vs = v + i * row_chunks;
        for (int c = lane; c < row_chunks; c += 32) {
            // token-major: the row is contiguous at the slot; head-major: head
            // h's part goes to row (block, h, off) of the [NB][Hkv][bs][D] pool
            int64_t dst = slot * row_chunks + c;
            if (HEAD_MAJOR) {
                const int64_t block = slot >> block_size_log2;
                const int64_t off = slot & ((1 << block_size_log2) - 1);
                const int h = c / head_chunks;
                dst = (((block * num_kv_heads + h) << block_size_log2) + off) * head_chunks +
                      (c - h * head_chunks);
            }
            const uint4 a = __ldg(ks + c);
            const uint4 b = __ldg(vs + c);
            k_cache[dst] = a;
            v_cache[dst] = b;
        }
    }
}

}  // namespace

cudaError_t take_store_error(cudaStream_t stream, int *code) {
    return take_device_word(g_store_error, stream, code);
}

cudaError_t launch_store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache,
                                 const int64_t *slot_mapping, int64_t num_tokens,
                                 int num_kv_heads, int head_dim, int block_size_log2,
                                 int64_t num_slots, int head_major, int sm_count,
                                 cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    int64_t blocks = (num_tokens + kStoreWarps - 1) / kStoreWarps;
    const int64_t cap = (int64_t)sm_count * 16;
    if (blocks > cap) blocks = cap;
    auto kernel = head_major ? store_kvcache_kernel<true> : store_kvcache_kernel<false>;
    kernel<<<(unsigned)blocks, kStoreWarps * 32, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v),
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping, num_tokens,
        num_kv_heads, head_dim / 8, block_size_log2, num_slots);
    return cudaGetLastError();
}

}  // namespace pa

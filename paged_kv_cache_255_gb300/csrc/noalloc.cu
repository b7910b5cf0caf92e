// pa_decode_noalloc: pa_decode for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that must
// not call cudaMalloc (a real-time loop that may not block, a host runtime
// whose allocator is owned by someone else, a plugin that only receives
// input and output pointers). For them the decode's scratch lives in one
// statically sized array in device global memory, created when the CUDA
// module is loaded; this entry point allocates nothing.
#include <mutex>

#include "../../include/pagedattn.h"
#include "kernels.h"

namespace {

// Scratch for the split-K partial results and combine tasks of pa_decode.
// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = PA_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current, and cached. The cache assumes the
// device's context is never reset in this process (a reset reloads the module
// at another address); the header states that limit.
pa_status_t scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status_t pa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, int max_blocks_per_seq,
                                         const int32_t *context_lens, float scale, void *out,
                                         int num_seqs, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, int64_t num_blocks,
                                         void *stream) {
    // pa_decode's own argument checks first, so that both calls answer bad
    // arguments and empty batches with the same status
    bool nothing_to_do = false;
    const pa_status_t chk = pa::decode_check_args(
        q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, 1, scale, out,
        num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
        PA_LAYOUT_TOKEN_MAJOR, 0, &nothing_to_do);
    if (chk != PA_OK || nothing_to_do) return chk;
    // the configuration is valid, so a zero size means the device query failed
    const size_t need = pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim, 0);
    if (need == 0) return PA_ERR_CUDA;
    if (need > kNoAllocScratchBytes) return PA_ERR_WORKSPACE;   // beyond the static scratch
    void *scratch = nullptr;
    const pa_status_t st = scratch_on_current_device(&scratch);
    if (st != PA_OK) return st;
    // Nothing in the scratch needs to start at zero: each call writes every
    // word of it that the same call later reads.
    return pa_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, scale,
                     out, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                     scratch, kNoAllocScratchBytes, stream);
}

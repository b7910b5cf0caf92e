// C ABI of libpagedattn: argument checks on the host, then kernel launches.
// The public contract is in include/pagedattn.h.
#include <atomic>
#include <cmath>
#include <cstdint>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pagedattn.h"
#include "kernels.h"

namespace {

// One NVTX range per public call, named after the entry point, in the domain
// "libpagedattn": a timeline, or an Nsight Compute run filtered with --nvtx,
// shows which call launched each kernel. With no tool attached a push or a pop
// is a test of a function pointer.
nvtxDomainHandle_t trace_domain() {
    static const nvtxDomainHandle_t d = nvtxDomainCreateA("libpagedattn");
    return d;
}

class TraceRange {
  public:
    explicit TraceRange(const char *name) {
        nvtxEventAttributes_t a{};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(trace_domain(), &a);
    }
    ~TraceRange() { nvtxDomainRangePop(trace_domain()); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The TMA tile copies address the pool's rows with int32 coordinates: token
// rows (num_blocks * block_size) in the token-major map, (block, KV head)
// rows (num_blocks * num_kv_heads) in the head-major one.
bool pool_rows_fit(int64_t num_blocks, int block_size, int num_kv_heads) {
    return num_blocks * block_size < ((int64_t)1 << 31) &&
           num_blocks * num_kv_heads < ((int64_t)1 << 31);
}

int log2_exact(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return (1 << l) == x ? l : -1;
}

bool block_size_ok(int bs) { return bs >= 16 && bs <= 256 && log2_exact(bs) >= 0; }

// Per-device values the calls need on every launch, computed on a device's
// first call and kept: its SM count, and the decode's worker count for each
// padded group size (1, 2, 4, 8, 16) and tile kind (both depend only on the
// device and the kernels' resources). A racing first call computes the same
// value twice.
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_workers[kMaxDevices][5][2];

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int current_sm_count() {
    const int dev = current_device();
    if (dev < 0) return 0;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Comparison kernels kept for tests (pa_debug_kernel_variant); 0 = the
// product kernels. Read once per call, so a test that flips it between
// calls sees the change at the next call.
std::atomic<int> g_kernel_variant{0};

// Tile computation for decode: tensor cores, unless the test hook asks for
// the CUDA-core variant (single-token decode, group size <= 8).
pa::DecodeKernel decode_kernel_choice(int group_pad, int q_len) {
    if ((g_kernel_variant.load(std::memory_order_relaxed) & PA_VARIANT_DECODE_SIMT) &&
        group_pad <= 8 && q_len == 1)
        return pa::DecodeKernel::kSimt;
    return pa::DecodeKernel::kMma;
}

// Shares of the tile space for a call: forced, or from the device.
int plan_workers(int group_pad, pa::DecodeKernel k, int num_partitions) {
    if (num_partitions > 0) return num_partitions;
    const int dev = current_device();
    if (dev < 0) return 0;
    int gi = 0;
    while ((1 << gi) < group_pad && gi < 4) ++gi;
    std::atomic<int> &slot = g_workers[dev][gi][k == pa::DecodeKernel::kSimt ? 1 : 0];
    int P = slot.load(std::memory_order_relaxed);
    if (P > 0) return P;
    const int sms = current_sm_count();
    P = sms > 0 ? pa::decode_default_workers(group_pad, k, sms) : 0;
    if (P > 0) slot.store(P, std::memory_order_relaxed);
    return P;
}

pa_status_t decode_impl(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, int q_len, float scale, void *out,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int64_t num_blocks, int layout, void *workspace,
                        size_t workspace_bytes, int num_partitions, void *stream,
                        bool plan_early = false) {
    bool nothing_to_do = false;
    const pa_status_t chk = pa::decode_check_args(
        q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, q_len, scale, out,
        num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, layout,
        num_partitions, &nothing_to_do);
    if (chk != PA_OK || nothing_to_do) return chk;
    const int group = num_q_heads / num_kv_heads;
    const int gp = pa::decode_group_pad(group * q_len);

    const pa::DecodeKernel kind = decode_kernel_choice(gp, q_len);
    const int P = plan_workers(gp, kind, num_partitions);
    if (P <= 0) return PA_ERR_CUDA;
    if (!workspace || !aligned16(workspace) || workspace_bytes < pa::decode_workspace_bytes(gp, P))
        return PA_ERR_WORKSPACE;

    pa::DecodeArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = out;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = group;
    a.q_len = q_len;
    a.cols = group * q_len;
    a.block_size_log2 = log2_exact(block_size);
    a.head_major = layout == PA_LAYOUT_HEAD_MAJOR ? 1 : 0;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);   // scale * log2(e)
    a.num_workers = P;
    a.min_tiles = num_partitions > 0 ? 1 : pa::kDefaultMinTiles;
    a.plan_early = plan_early ? 1 : 0;
    pa::decode_carve_workspace(a, workspace, gp);
    const cudaError_t e = pa::launch_decode(a, gp, kind, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status_t store_impl(const void *k, const void *v, void *k_cache, void *v_cache,
                       const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads,
                       int head_dim, int block_size, int64_t num_blocks, int layout,
                       void *stream) {
    bool nothing_to_do = false;
    const pa_status_t chk = pa::store_check_args(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                                 num_kv_heads, head_dim, block_size, num_blocks,
                                                 layout, &nothing_to_do);
    if (chk != PA_OK || nothing_to_do) return chk;
    const int sms = current_sm_count();
    if (sms <= 0) return PA_ERR_CUDA;
    const cudaError_t e = pa::launch_store_kvcache(
        k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
        log2_exact(block_size), num_blocks * block_size, layout == PA_LAYOUT_HEAD_MAJOR ? 1 : 0,
        sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status_t prefill_impl(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, const int32_t *query_start_loc,
                         int max_query_len, float scale, void *out, int num_seqs, int total_q,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks, int layout, void *stream) {
    if (layout != PA_LAYOUT_TOKEN_MAJOR && layout != PA_LAYOUT_HEAD_MAJOR) return PA_ERR_INVALID_ARG;
    if (num_seqs < 0 || total_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_blocks < 0 || max_blocks_per_seq < 0 || max_query_len < 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (head_dim != pa::kHeadDimPublic || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    const int group = num_q_heads / num_kv_heads;
    const int gp = pa::decode_group_pad(group);
    if (gp == 0) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || total_q == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start_loc || !out)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return PA_ERR_INVALID_ARG;
    if (max_blocks_per_seq == 0 || num_blocks == 0) return PA_ERR_INVALID_ARG;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!pool_rows_fit(num_blocks, block_size, num_kv_heads)) return PA_ERR_UNSUPPORTED;
    pa::PrefillArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start_loc = query_start_loc;
    a.out = out;
    a.num_seqs = num_seqs;
    a.total_q = total_q;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = group;
    a.block_size_log2 = log2_exact(block_size);
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.head_major = layout == PA_LAYOUT_HEAD_MAJOR ? 1 : 0;
    a.fault_hold_v = pa::prefill_fault();
    a.num_blocks = num_blocks;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    const int mql = max_query_len > 0 ? max_query_len : 1;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool mma = g_kernel_variant.load(std::memory_order_relaxed) & PA_VARIANT_PREFILL_MMA;
    const cudaError_t e = mma ? pa::launch_prefill(a, gp, mql, st)
                              : pa::launch_prefill_tc(a, gp, mql, st);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

namespace pa {

pa_status_t store_check_args(const void *k, const void *v, const void *k_cache,
                             const void *v_cache, const int64_t *slot_mapping, int64_t num_tokens,
                             int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                             int layout, bool *nothing_to_do) {
    *nothing_to_do = false;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (layout != PA_LAYOUT_TOKEN_MAJOR && layout != PA_LAYOUT_HEAD_MAJOR) return PA_ERR_INVALID_ARG;
    if (head_dim != kHeadDimPublic || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) {
        *nothing_to_do = true;
        return PA_OK;
    }
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

pa_status_t decode_check_args(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int q_len, float scale,
                              const void *out, int num_seqs, int num_q_heads, int num_kv_heads,
                              int head_dim, int block_size, int64_t num_blocks, int layout,
                              int num_partitions, bool *nothing_to_do) {
    *nothing_to_do = false;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks < 0 ||
        max_blocks_per_seq < 0 || num_partitions < 0 || q_len < 1 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (layout != PA_LAYOUT_TOKEN_MAJOR && layout != PA_LAYOUT_HEAD_MAJOR) return PA_ERR_INVALID_ARG;
    if (head_dim != kHeadDimPublic || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    const int group = num_q_heads / num_kv_heads;
    if (q_len > 16) return PA_ERR_UNSUPPORTED;
    if (decode_group_pad(group * q_len) == 0) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) {
        *nothing_to_do = true;
        return PA_OK;
    }
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return PA_ERR_INVALID_ARG;
    if (max_blocks_per_seq == 0 || num_blocks == 0) return PA_ERR_INVALID_ARG;
    if (!pool_rows_fit(num_blocks, block_size, num_kv_heads)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

}  // namespace pa

extern "C" {

const char *pa_status_string(pa_status_t status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
    }
    return "PA_ERR_UNKNOWN";
}

pa_status_t pa_store_kvcache_layout(const void *k, const void *v, void *k_cache, void *v_cache,
                                    const int64_t *slot_mapping, int64_t num_tokens,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int64_t num_blocks, pa_layout_t layout, void *stream) {
    TraceRange r("pa_store_kvcache_layout");
    return store_impl(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                      block_size, num_blocks, layout, stream);
}

pa_status_t pa_store_kvcache(const void *k, const void *v, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int64_t num_blocks, void *stream) {
    TraceRange r("pa_store_kvcache");
    return store_impl(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                      block_size, num_blocks, PA_LAYOUT_TOKEN_MAJOR, stream);
}

size_t pa_decode_workspace_size(int num_q_heads, int num_kv_heads, int head_dim,
                                int num_partitions) {
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        head_dim != pa::kHeadDimPublic || num_partitions < 0)
        return 0;
    const int gp = pa::decode_group_pad(num_q_heads / num_kv_heads);
    if (gp == 0) return 0;
    // sized for the larger of the two variants' default share counts
    int P = plan_workers(gp, pa::DecodeKernel::kMma, num_partitions);
    if (num_partitions == 0 && gp <= 8) {
        const int Ps = plan_workers(gp, pa::DecodeKernel::kSimt, 0);
        P = Ps > P ? Ps : P;
    }
    if (P <= 0) return 0;
    return pa::decode_workspace_bytes(gp, P);
}

pa_status_t pa_decode(const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, float scale, void *out, int num_seqs,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int64_t num_blocks, void *workspace, size_t workspace_bytes,
                      void *stream) {
    TraceRange r("pa_decode");
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, 1,
                       scale, out, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, PA_LAYOUT_TOKEN_MAJOR, workspace, workspace_bytes, 0, stream);
}

pa_status_t pa_decode_splitk(const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, float scale, void *out, int num_seqs,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks, void *workspace, size_t workspace_bytes,
                             int num_partitions, void *stream) {
    TraceRange r("pa_decode_splitk");
    if (num_partitions < 0) return PA_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, 1,
                       scale, out, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, PA_LAYOUT_TOKEN_MAJOR, workspace, workspace_bytes,
                       num_partitions, stream);
}

size_t pa_decode_multi_workspace_size(int q_len, int num_q_heads, int num_kv_heads,
                                      int head_dim) {
    if (q_len < 1 || q_len > 16 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || head_dim != pa::kHeadDimPublic)
        return 0;
    const int gp = pa::decode_group_pad(num_q_heads / num_kv_heads * q_len);
    if (gp == 0) return 0;
    const int P = plan_workers(gp, pa::DecodeKernel::kMma, 0);
    return P > 0 ? pa::decode_workspace_bytes(gp, P) : 0;
}

pa_status_t pa_decode_layout(const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, float scale, void *out, int num_seqs,
                             int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks, pa_layout_t layout, void *workspace,
                             size_t workspace_bytes, int num_partitions, void *stream) {
    TraceRange r("pa_decode_layout");
    if (num_partitions < 0) return PA_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, 1,
                       scale, out, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, layout, workspace, workspace_bytes, num_partitions, stream);
}

pa_status_t pa_decode_multi(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int q_len, float scale, void *out,
                            int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, void *workspace,
                            size_t workspace_bytes, void *stream) {
    TraceRange r("pa_decode_multi");
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       q_len, scale, out, num_seqs, num_q_heads, num_kv_heads, head_dim,
                       block_size, num_blocks, PA_LAYOUT_TOKEN_MAJOR, workspace,
                       workspace_bytes, 0, stream);
}

pa_status_t pa_decode_multi_layout(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *context_lens, int q_len, float scale, void *out,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int64_t num_blocks, pa_layout_t layout,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    TraceRange r("pa_decode_multi_layout");
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       q_len, scale, out, num_seqs, num_q_heads, num_kv_heads, head_dim,
                       block_size, num_blocks, layout, workspace, workspace_bytes, 0, stream);
}

pa_status_t pa_decode_step(const void *k, const void *v, const int64_t *slot_mapping,
                           int64_t num_tokens, const void *q, void *k_cache, void *v_cache,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, float scale, void *out, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int64_t num_blocks, pa_layout_t layout, void *workspace,
                           size_t workspace_bytes, void *stream) {
    TraceRange r("pa_decode_step");
    // every argument of both calls is checked before anything is launched
    bool no_store = false, no_decode = false;
    pa_status_t chk = pa::store_check_args(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                           num_kv_heads, head_dim, block_size, num_blocks, layout,
                                           &no_store);
    if (chk != PA_OK) return chk;
    chk = pa::decode_check_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, 1, scale, out, num_seqs, num_q_heads, num_kv_heads,
                                head_dim, block_size, num_blocks, layout, 0, &no_decode);
    if (chk != PA_OK) return chk;
    if (!no_decode) {
        const int gp = pa::decode_group_pad(num_q_heads / num_kv_heads);
        const int P = plan_workers(gp, decode_kernel_choice(gp, 1), 0);
        if (P <= 0) return PA_ERR_CUDA;
        if (!workspace || !aligned16(workspace) ||
            workspace_bytes < pa::decode_workspace_bytes(gp, P))
            return PA_ERR_WORKSPACE;
    }
    chk = store_impl(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                     block_size, num_blocks, layout, stream);
    if (chk != PA_OK) return chk;
    // with the store just queued, the decode plans its split while the store runs
    return decode_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, 1,
                       scale, out, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, layout, workspace, workspace_bytes, 0, stream, !no_store);
}

pa_status_t pa_prefill(const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *context_lens, const int32_t *query_start_loc,
                       int max_query_len, float scale, void *out, int num_seqs, int total_q,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       int64_t num_blocks, void *stream) {
    TraceRange r("pa_prefill");
    return prefill_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        query_start_loc, max_query_len, scale, out, num_seqs, total_q,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                        PA_LAYOUT_TOKEN_MAJOR, stream);
}

pa_status_t pa_prefill_layout(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, const int32_t *query_start_loc,
                              int max_query_len, float scale, void *out, int num_seqs,
                              int total_q, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int64_t num_blocks, pa_layout_t layout,
                              void *stream) {
    TraceRange r("pa_prefill_layout");
    return prefill_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        query_start_loc, max_query_len, scale, out, num_seqs, total_q,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, layout,
                        stream);
}

pa_status_t pa_debug_kernel_variant(int flags) {
    if (flags & ~(PA_VARIANT_DECODE_SIMT | PA_VARIANT_PREFILL_MMA)) return PA_ERR_INVALID_ARG;
    g_kernel_variant.store(flags, std::memory_order_relaxed);
    return PA_OK;
}

pa_status_t pa_debug_prefill_fault(int mode) {
    if (mode != 0 && mode != 1) return PA_ERR_INVALID_ARG;
    pa::set_prefill_fault(mode);
    return PA_OK;
}

pa_status_t pa_take_device_error(int32_t *code, void *stream) {
    TraceRange r("pa_take_device_error");
    if (!code) return PA_ERR_INVALID_ARG;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t (*const take[])(cudaStream_t, int *) = {
        pa::take_prefill_error, pa::take_prefill_mma_error, pa::take_decode_error,
        pa::take_store_error};
    int first = 0;
    for (auto f : take) {   // every word is read and cleared; the smallest code is reported
        int v = 0;
        if (f(st, &v) != cudaSuccess) return PA_ERR_CUDA;
        if (v != 0 && (first == 0 || v < first)) first = v;
    }
    *code = first;
    return PA_OK;
}

}  // extern "C"

// Paged prefill on the 5th-generation tensor cores (tcgen05): the same
// attention as prefill.cu (chunk rows of a sequence attend causally to its
// tokens in the paged KV cache; "A vLLM engine small enough to read in one
// sitting": prefill and decode run over the paged KV cache, flash attention
// for prefill), computed in the flash-attention order with the two
// contractions on tcgen05.mma and both accumulators in tensor memory.
//
// A CTA of 4 warps owns 128 rows of one (sequence, KV head): 128 / G query
// tokens x the G query heads of the group (G = group size rounded up to a
// power of two); thread t owns row t, which is TMEM lane t. Per 64-key tile j:
//   S = Q K_j^T   M 128, N 64, K 128: Q and K_j in shared memory, S in TMEM
//   softmax       each thread reads its row of S (tcgen05.ld), masks it
//                 causally, updates its running max / sum and writes P (bf16)
//                 to shared memory
//   O += P V_j    M 128, N 128, K 64: P and V_j in shared memory, O in TMEM
// The running max is raised only when a tile's max exceeds it by more than
// 2^8 (in exp2 units); otherwise the stale max is kept, which changes nothing
// in O / l but the rounding, and saves reading and writing O back. When it is
// raised, the warp rescales its rows of O in TMEM.
//
// Thread 0 issues the MMAs; tcgen05.commit signals their completion on two
// mbarriers (S done, PV done). K and V tiles are gathered through the block
// table by 16-byte cp.async into two-stage rings, written in the 128-byte
// swizzled layout the MMA descriptors name. K_{j+2} is fetched as soon as
// S_j has finished with K_j's stage, V_{j+1} as soon as PV_{j-1} has finished
// with its stage. Two CTAs share an SM (115 KB shared memory and 256 TMEM
// columns each), so one CTA's softmax overlaps the other's MMAs.
//
// Every mbarrier wait is bounded (about 2 s); a CTA whose wait runs out
// records an error, stops at the next CTA-wide barrier (all threads learn of it
// there through __syncthreads_or), waits for its copies, frees its TMEM and
// exits.
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pa {

__device__ int g_prefill_error;      // first device-side error of a prefill launch

namespace {

constexpr int kRows = 128;
constexpr int kKeys = 64;
constexpr int kThreads = 128;
constexpr uint32_t kQBytes = kRows * kRowBytes;         // 32 KB: 2 K-halves of [128][128 B]
constexpr uint32_t kQHalf = kRows * 128;                // 16 KB
constexpr uint32_t kKVBytes = kKeys * kRowBytes;        // 16 KB: 2 halves of [64][128 B]
constexpr uint32_t kKVHalf = kKeys * 128;               // 8 KB
constexpr uint32_t kPBytes = kRows * kKeys * 2;         // 16 KB: [128][128 B]
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;             // 2 stages
constexpr uint32_t kOffV = kOffK + 2 * kKVBytes;        // 2 stages
constexpr uint32_t kOffP = kOffV + 2 * kKVBytes;
constexpr uint32_t kOffCtl = kOffP + kPBytes;           // mbarriers, TMEM base, abort flag
constexpr uint32_t kSmemBytes = kOffCtl + 64;
constexpr uint32_t kTmemCols = 256;                     // S: columns 0-63, O: 128-255
constexpr uint32_t kColO = 128;
constexpr uint32_t kIdescS = tc::idesc_bf16(128, kKeys, false);
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, true);
constexpr float kRescaleSlack = 8.f;                    // log2 units

enum : int { kErrSmemAlign = 1, kErrTimeout = 2 };

__device__ __forceinline__ void set_error(int code) { atomicCAS(&g_prefill_error, 0, code); }

// cp.async of K or V rows of keys [k0, k0 + 64) of (sequence s, KV head kvh)
// into a stage: key r, 16-byte chunk c (dims 8c..8c+7) goes to half c / 8,
// row r, chunk position (c % 8) ^ (r % 8). Keys at or past kend are zero.
__device__ __forceinline__ void load_kv(const PrefillArgs &a, const void *cache, int s, int kvh,
                                        int k0, int kend, uint32_t stage) {
    const int bs_mask = (1 << a.block_size_log2) - 1;
    const char *base = static_cast<const char *>(cache);
#pragma unroll
    for (int i = 0; i < (kKeys * 16) / kThreads; ++i) {
        const int c = threadIdx.x + i * kThreads;
        const int key = c >> 4, chunk = c & 15;
        const int t = k0 + key;
        bool ok = t < kend;
        int64_t row = 0;
        if (ok) {
            const int bid = __ldg(a.block_tables + (int64_t)s * a.max_blocks_per_seq +
                                  (t >> a.block_size_log2));
            ok = bid >= 0 && (int64_t)bid < a.num_blocks;
            row = (((int64_t)bid << a.block_size_log2) + (t & bs_mask)) * a.num_kv_heads + kvh;
        }
        const uint32_t dst = stage + (chunk >> 3) * kKVHalf + key * 128 +
                             ((((uint32_t)chunk & 7) ^ ((uint32_t)key & 7)) << 4);
        cp_async_16(dst, base + (ok ? row * kRowBytes + chunk * 16 : 0), ok ? 16 : 0);
    }
}

template <int G>
__global__ void __launch_bounds__(kThreads, 2) prefill_tc_kernel(const PrefillArgs a) {
    constexpr int BT = kRows / G;               // query tokens per CTA tile
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int s = blockIdx.y, kvh = blockIdx.z;
    const int g = a.group;

    int q0 = __ldg(a.query_start_loc + s);
    int q1 = __ldg(a.query_start_loc + s + 1);
    q0 = q0 < 0 ? 0 : (q0 > a.total_q ? a.total_q : q0);
    q1 = q1 < q0 ? q0 : (q1 > a.total_q ? a.total_q : q1);
    const int n = q1 - q0;
    // heaviest tiles (last rows of the chunk see the most keys) first
    const int qt_first = gridDim.x - 1 - blockIdx.x;
    if (qt_first * BT >= n) return;

    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {                        // the swizzle atoms need 1024-byte alignment
        if (tid == 0) set_error(kErrSmemAlign);
        return;
    }
    int L = __ldg(a.context_lens + s);
    {
        const int64_t max_len = (int64_t)a.max_blocks_per_seq << a.block_size_log2;
        L = L < 0 ? 0 : ((int64_t)L > max_len ? (int)max_len : L);
    }
    const uint32_t sQ = sbase + kOffQ, sK = sbase + kOffK, sV = sbase + kOffV, sP = sbase + kOffP;
    const uint32_t bar_s = sbase + kOffCtl, bar_pv = bar_s + 8;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + kOffCtl + 16);

    if (tid == 0) {
        tc::mbar_init(bar_s, 1);
        tc::mbar_init(bar_pv, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(sbase + kOffCtl + 16, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane = (uint32_t)(warp * 32) << 16;       // this warp's TMEM lane quarter
    const uint32_t tS = tmem, tO = tmem + kColO;
    uint32_t ph_s = 0, ph_pv = 0;
    bool aborted = false;          // CTA-uniform: set from __syncthreads_or
    int timed_out = 0;             // this thread's waits

    const uint16_t *qg = static_cast<const uint16_t *>(a.q);
    char *outg = static_cast<char *>(a.out);

#pragma unroll 1
    for (int qt = qt_first; qt * BT < n && !aborted; qt += gridDim.x) {
        const int tok0 = qt * BT;
        const int tok = tok0 + tid / G, head = tid % G;
        const bool rv = tok < n && head < g;
        int lim = 0;
        if (rv) {
            const int l = L - n + tok + 1;
            lim = l < 0 ? 0 : (l > L ? L : l);
        }
        const int last_tok = (tok0 + BT < n ? tok0 + BT : n) - 1;
        int kend = L - n + last_tok + 1;
        kend = kend < 0 ? 0 : (kend > L ? L : kend);
        const int ntiles = (kend + kKeys - 1) / kKeys;
        const int64_t row_elem = ((int64_t)q0 + tok) * a.num_q_heads + (int64_t)kvh * g + head;

        // Q row -> shared (K-major, swizzled), K_0 / V_0, then K_1
        {
            const char *src = reinterpret_cast<const char *>(qg + (rv ? row_elem : 0) * kHeadDim);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint32_t dst = sQ + (c >> 3) * kQHalf + tid * 128 +
                                     ((((uint32_t)c & 7) ^ ((uint32_t)tid & 7)) << 4);
                cp_async_16(dst, src + (rv ? c * 16 : 0), rv ? 16 : 0);
            }
        }
        if (ntiles > 0) {
            load_kv(a, a.k_cache, s, kvh, 0, kend, sK);
            load_kv(a, a.v_cache, s, kvh, 0, kend, sV);
        }
        cp_async_commit();
        if (ntiles > 1) load_kv(a, a.k_cache, s, kvh, kKeys, kend, sK + kKVBytes);
        cp_async_commit();
        cp_async_wait<1>();
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();

        auto issue_s = [&](int stage) {
            tc::fence_after_sync();
#pragma unroll
            for (int k = 0; k < kHeadDim / 16; ++k) {
                const uint32_t off = (k & 3) * 32;
                tc::mma_ss(tS, tc::sw128_desc(sQ + (k >> 2) * kQHalf + off, 16, 1024),
                           tc::sw128_desc(sK + stage * kKVBytes + (k >> 2) * kKVHalf + off, 16, 1024),
                           kIdescS, k > 0);
            }
            tc::commit(bar_s);
        };
        auto issue_pv = [&](int stage, bool acc) {
            tc::fence_after_sync();
#pragma unroll
            for (int k = 0; k < kKeys / 16; ++k)
                tc::mma_ss(tO, tc::sw128_desc(sP + k * 32, 16, 1024),
                           tc::sw128_desc(sV + stage * kKVBytes + k * 2048, kKVHalf, 1024),
                           kIdescPV, acc || k > 0);
            tc::commit(bar_pv);
        };
        if (tid == 0 && ntiles > 0) issue_s(0);

        float m = -INFINITY, lsum = 0.f;
        const float sc = a.scale_log2;
#pragma unroll 1
        for (int j = 0; j < ntiles; ++j) {
            // 1. this row of S_j
            if (!tc::mbar_wait(bar_s, ph_s)) { set_error(kErrTimeout); timed_out = 1; }
            ph_s ^= 1;
            tc::fence_after_sync();
            uint32_t sr[2][32];
            tc::tmem_ld32(tS + lane, sr[0]);
            tc::tmem_ld32(tS + lane + 32, sr[1]);
            tc::tmem_ld_wait();
            // K_j's stage is free: fetch K_{j+2} into it
            if (j + 2 < ntiles) load_kv(a, a.k_cache, s, kvh, (j + 2) * kKeys, kend, sK + (j & 1) * kKVBytes);
            cp_async_commit();

            // 2. scores in exp2 units, causal mask, running max (raised
            // lazily), P = 2^(S sc - m)
            const int kb = j * kKeys;
            float mt = -INFINITY;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float v = __uint_as_float(sr[h][c]) * sc;
                    if (kb + h * 32 + c >= lim) v = -INFINITY;
                    sr[h][c] = __float_as_uint(v);
                    mt = fmaxf(mt, v);
                }
            bool rescale = false;
            float alpha = 1.f;
            if (mt > m + kRescaleSlack) {
                rescale = m != -INFINITY;
                alpha = rescale ? ex2(m - mt) : 1.f;
                lsum *= alpha;
                m = mt;
            }
            const float mb = m == -INFINITY ? 0.f : m;
            uint32_t pw[32];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float p0 = ex2(__uint_as_float(sr[h][2 * c]) - mb);
                    const float p1 = ex2(__uint_as_float(sr[h][2 * c + 1]) - mb);
                    const uint32_t w = pack_bf16x2(p0, p1);
                    lsum += bf16_lo(w) + bf16_hi(w);
                    pw[h * 16 + c] = w;
                }

            // 3. PV_{j-1} done: O is stable, P and V_{j-1}'s stage are free
            if (j > 0) {
                if (!tc::mbar_wait(bar_pv, ph_pv)) { set_error(kErrTimeout); timed_out = 1; }
                ph_pv ^= 1;
                tc::fence_after_sync();
            }
            if (j + 1 < ntiles) load_kv(a, a.v_cache, s, kvh, (j + 1) * kKeys, kend, sV + ((j + 1) & 1) * kKVBytes);
            cp_async_commit();

            // 4. rescale this warp's rows of O if any of them raised its max
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t o[32];
                    tc::tmem_ld32(tO + lane + ch * 32, o);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tc::tmem_st32(tO + lane + ch * 32, o);
                }
                tc::tmem_st_wait();
            }

            // 5. P_j -> shared (row tid, K-major, swizzled)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t dst = sP + tid * 128 + ((((uint32_t)c) ^ ((uint32_t)tid & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst),
                             "r"(pw[4 * c]), "r"(pw[4 * c + 1]), "r"(pw[4 * c + 2]), "r"(pw[4 * c + 3])
                             : "memory");
            }
            // 6. K_{j+1} and V_j have landed (two newer groups may be pending)
            cp_async_wait<2>();
            tc::fence_proxy_async();
            tc::fence_before_sync();
            if (__syncthreads_or(timed_out)) { aborted = true; break; }
            // 7. O += P_j V_j, then S_{j+1} = Q K_{j+1}^T
            if (tid == 0) {
                issue_pv(j & 1, j > 0);
                if (j + 1 < ntiles) issue_s((j + 1) & 1);
            }
        }
        if (aborted) break;

        // epilogue: O / l -> bf16 rows
        if (ntiles > 0) {
            if (!tc::mbar_wait(bar_pv, ph_pv)) { set_error(kErrTimeout); timed_out = 1; }
            ph_pv ^= 1;
            tc::fence_after_sync();
        }
        float lt = lsum;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        uint4 *orow = reinterpret_cast<uint4 *>(outg + row_elem * kRowBytes);
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
            uint32_t o[32];
            if (ntiles > 0) {
                tc::tmem_ld32(tO + lane + ch * 32, o);
                tc::tmem_ld_wait();
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = 0u;
            }
            if (rv) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv);
                    orow[ch * 4 + c] = w;
                }
            }
        }
        cp_async_wait<0>();
        tc::fence_before_sync();
        // next tile rewrites Q, K/V, S and O
        if (__syncthreads_or(timed_out)) aborted = true;
    }

    cp_async_wait<0>();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int G>
cudaError_t launch_g(const PrefillArgs &a, int max_query_len, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    constexpr int BT = kRows / G;
    int gx = (max_query_len + BT - 1) / BT;
    gx = gx < 1 ? 1 : (gx > 65535 ? 65535 : gx);
    prefill_tc_kernel<G><<<dim3(gx, a.num_seqs, a.num_kv_heads), kThreads, kSmemBytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a, int group_pad, int max_query_len,
                              cudaStream_t stream) {
    switch (group_pad) {
        case 1: return launch_g<1>(a, max_query_len, stream);
        case 2: return launch_g<2>(a, max_query_len, stream);
        case 4: return launch_g<4>(a, max_query_len, stream);
        case 8: return launch_g<8>(a, max_query_len, stream);
        case 16: return launch_g<16>(a, max_query_len, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t take_prefill_error(cudaStream_t stream, int *code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_prefill_error, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    *code = v;
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_prefill_error, &zero, sizeof(int), 0,
                                    cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace pa

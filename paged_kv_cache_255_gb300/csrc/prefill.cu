// Paged prefill: a chunk of new tokens per sequence attends causally to the
// sequence's tokens in the paged KV cache (the prompt phase of the engine,
// "A vLLM engine small enough to read in one sitting": prefill and decode both
// run over the paged KV cache; flash attention for the prefill side).
//
// What it computes: the rows of q are packed sequence after sequence;
// sequence s owns rows [qsl[s], qsl[s + 1]). With n of them and L =
// context_lens[s] (counting the chunk, already stored in the cache), row i is
// the token at position L - n + i and, for query head h of KV head h / g,
//   out = sum_{t <= L - n + i} softmax_t(scale * q . K_t) V_t,
// with K_t, V_t gathered through the sequence's block table.
//
// How (GB300 design): a contraction, so the tensor cores do it, in the
// flash-attention order. A CTA of 4 warps owns 64 rows of one (sequence, KV
// head): 64 / G query tokens x the G query heads of the group (G = group size
// rounded up to a power of two), so every K/V tile fetched serves the whole
// group. Each warp holds 16 rows: S = Q K^T on mma.sync m16n8k16 (bf16 in,
// fp32 accumulate) against 64-key tiles, causal mask per row, online softmax
// on the accumulator fragments, P (bf16) reused in registers as the A operand
// of O += P V. K/V tiles are gathered through the block table into a
// double-buffered, chunk-swizzled shared-memory ring by 16-byte cp.async
// (rows past the visible range are zero-filled, never read).
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace pa {

__device__ int g_prefill_mma_error;  // first device-side error of a launch of this kernel

namespace {

constexpr int kPfRows = 64;                    // query rows per CTA
constexpr int kPfKeys = 64;                    // keys per K/V tile
constexpr int kPfThreads = 128;
constexpr int kPfTileBytes = kPfKeys * kRowBytes;          // 16 KB
constexpr int kPfStageBytes = 2 * kPfTileBytes;            // K then V
constexpr int kPfSmemBytes = 2 * kPfStageBytes;            // double buffer: 64 KB
constexpr float kPfNegInf = -INFINITY;

__device__ __forceinline__ int pf_clamp_len(const PrefillArgs &a, int s) {
    int L = __ldg(a.context_lens + s);
    const int64_t max_len = (int64_t)a.max_blocks_per_seq << a.block_size_log2;
    L = L < 0 ? 0 : L;
    return (int64_t)L > max_len ? (int)max_len : L;
}

// cp.async of the K and V rows of keys [k0, k0 + 64) of (sequence s, KV head
// kvh) into `stage`; keys at or past kend are zero-filled. Token-major pool:
// row (slot * Hkv + kvh); head-major: ((block * Hkv + kvh) * bs + offset).
__device__ __forceinline__ void pf_load_tile(const PrefillArgs &a, int s, int kvh, int k0,
                                             int kend, uint8_t *stage) {
    const uint32_t dst = smem_u32(stage);
    const int bs_mask = (1 << a.block_size_log2) - 1;
#pragma unroll
    for (int i = 0; i < (kPfKeys * 16) / kPfThreads; ++i) {
        const int c = threadIdx.x + i * kPfThreads;
        const int key = c >> 4, chunk = c & 15;
        const int t = k0 + key;
        bool ok = t < kend;
        int64_t row = 0;
        if (ok) {
            const int bid = __ldg(a.block_tables + (int64_t)s * a.max_blocks_per_seq +
                                  (t >> a.block_size_log2));
            ok = bid >= 0 && (int64_t)bid < a.num_blocks;
            if (!ok) atomicCAS(&g_prefill_mma_error, 0, kErrBadBlock);   // read as zeros
            row = a.head_major
                      ? (((int64_t)bid * a.num_kv_heads + kvh) << a.block_size_log2) + (t & bs_mask)
                      : ((((int64_t)bid << a.block_size_log2) + (t & bs_mask)) * a.num_kv_heads + kvh);
        }
        const int pos = chunk ^ (key & 7);
        const char *ks = static_cast<const char *>(a.k_cache) + (ok ? row * kRowBytes + chunk * 16 : 0);
        const char *vs = static_cast<const char *>(a.v_cache) + (ok ? row * kRowBytes + chunk * 16 : 0);
        cp_async_16(dst + key * kRowBytes + pos * 16, ks, ok ? 16 : 0);
        cp_async_16(dst + kPfTileBytes + key * kRowBytes + pos * 16, vs, ok ? 16 : 0);
    }
}

template <int G>
__global__ void __launch_bounds__(kPfThreads)
prefill_kernel(const PrefillArgs a) {
    constexpr int BT = kPfRows / G;             // query tokens per CTA
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int i7 = lane & 7, mi = lane >> 3;
    const int s = blockIdx.y, kvh = blockIdx.z;
    const int g = a.group;

    // rows outside [0, total_q) are never touched, whatever query_start_loc holds
    int q0 = __ldg(a.query_start_loc + s);
    int q1 = __ldg(a.query_start_loc + s + 1);
    q0 = q0 < 0 ? 0 : (q0 > a.total_q ? a.total_q : q0);
    q1 = q1 < q0 ? q0 : (q1 > a.total_q ? a.total_q : q1);
    const int n = q1 - q0;
    const int L = pf_clamp_len(a, s);
    const uint16_t *qg = static_cast<const uint16_t *>(a.q);
    uint32_t *outg = static_cast<uint32_t *>(a.out);

#pragma unroll 1
    for (int qt = blockIdx.x; qt * BT < n; qt += gridDim.x) {
        const int tok0 = qt * BT;
        // this lane's two rows (gid and gid + 8 of the warp's 16)
        int tok[2], head[2], lim[2];
        bool rv[2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = warp * 16 + gid + hr * 8;
            tok[hr] = tok0 + r / G;
            head[hr] = r % G;
            rv[hr] = tok[hr] < n && head[hr] < g;
            const int l = L - n + tok[hr] + 1;
            lim[hr] = rv[hr] ? (l < 0 ? 0 : (l > L ? L : l)) : 0;
        }
        // keys any row of the CTA may see
        const int last_tok = (tok0 + BT < n ? tok0 + BT : n) - 1;
        int kend = L - n + last_tok + 1;
        kend = kend < 0 ? 0 : (kend > L ? L : kend);
        const int ntiles = (kend + kPfKeys - 1) / kPfKeys;

        // Q fragments (A operand): rows gid / gid + 8, dims 16 kk + 2 tig (+ 8)
        uint32_t qa[8][4];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
#pragma unroll
            for (int x = 0; x < 4; ++x) qa[kk][x] = 0u;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            if (rv[hr]) {
                const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                    qg + (((int64_t)q0 + tok[hr]) * a.num_q_heads + (int64_t)kvh * g + head[hr]) *
                             kHeadDim);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    qa[kk][hr] = __ldg(qrow + kk * 8 + tig);
                    qa[kk][hr + 2] = __ldg(qrow + kk * 8 + 4 + tig);
                }
            }
        }

        float o[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int x = 0; x < 4; ++x) o[nt][x] = 0.f;
        float m[2] = {kPfNegInf, kPfNegInf}, l[2] = {0.f, 0.f};

        if (ntiles > 0) pf_load_tile(a, s, kvh, 0, kend, smem);
        cp_async_commit();
#pragma unroll 1
        for (int kt = 0; kt < ntiles; ++kt) {
            if (kt + 1 < ntiles)
                pf_load_tile(a, s, kvh, (kt + 1) * kPfKeys, kend,
                             smem + ((kt + 1) & 1) * kPfStageBytes);
            cp_async_commit();
            cp_async_wait<1>();
            __syncthreads();
            const uint32_t kbase = smem_u32(smem + (kt & 1) * kPfStageBytes);
            const uint32_t vbase = kbase + kPfTileBytes;

            // S = Q K^T for 64 keys: 8 column tiles of 8 keys
            float sc[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int x = 0; x < 4; ++x) sc[nt][x] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t krow = kbase + (16 * j + i7 + 8 * (mi >> 1)) * kRowBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    uint32_t b[4];
                    ldmatrix_x4(krow + (((2 * kk + (mi & 1)) ^ i7) << 4), b);
                    mma_bf16_16816(sc[2 * j], qa[kk], b[0], b[1]);
                    mma_bf16_16816(sc[2 * j + 1], qa[kk], b[2], b[3]);
                }
            }

            // causal mask, online softmax per row (rows gid, gid + 8)
            const int kb = kt * kPfKeys + 2 * tig;
            float mx[2] = {kPfNegInf, kPfNegInf};
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int hr = x >> 1;
                    const int key = kb + nt * 8 + (x & 1);
                    const float v = key < lim[hr] ? sc[nt][x] * a.scale_log2 : kPfNegInf;
                    sc[nt][x] = v;
                    mx[hr] = fmaxf(mx[hr], v);
                }
            }
            float alpha[2], ms[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
                mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
                const float mn = fmaxf(m[hr], mx[hr]);
                ms[hr] = mn == kPfNegInf ? 0.f : mn;
                alpha[hr] = ex2(m[hr] - ms[hr]);
                m[hr] = mn;
                l[hr] *= alpha[hr];
            }
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                o[nt][0] *= alpha[0];
                o[nt][1] *= alpha[0];
                o[nt][2] *= alpha[1];
                o[nt][3] *= alpha[1];
            }
            // P (bf16) as the A operand of P V, 16 keys per k-step; the sums
            // add the same rounded weights
            uint32_t pa_[4][4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int nt = 2 * k2 + half;
                    const uint32_t lo = pack_bf16x2(ex2(sc[nt][0] - ms[0]), ex2(sc[nt][1] - ms[0]));
                    const uint32_t hi = pack_bf16x2(ex2(sc[nt][2] - ms[1]), ex2(sc[nt][3] - ms[1]));
                    l[0] += bf16_lo(lo) + bf16_hi(lo);
                    l[1] += bf16_lo(hi) + bf16_hi(hi);
                    pa_[k2][2 * half] = lo;
                    pa_[k2][2 * half + 1] = hi;
                }
            }
            // O += P V: B = V (keys x dims) by ldmatrix.trans
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
                const uint32_t ap[4] = {pa_[k2][0], pa_[k2][1], pa_[k2][2], pa_[k2][3]};
                const uint32_t vrow = vbase + (16 * k2 + i7 + 8 * (mi & 1)) * kRowBytes;
#pragma unroll
                for (int dt = 0; dt < 8; ++dt) {
                    uint32_t b[4];
                    ldmatrix_x4_trans(vrow + (((2 * dt + (mi >> 1)) ^ i7) << 4), b);
                    mma_bf16_16816(o[2 * dt], ap, b[0], b[1]);
                    mma_bf16_16816(o[2 * dt + 1], ap, b[2], b[3]);
                }
            }
            __syncthreads();   // the stage is refilled by the next iteration's load
        }
        cp_async_wait<0>();

        // normalise and write: lane holds dims 8 nt + 2 tig, + 1 of its two rows
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            float lt = l[hr];
            lt += __shfl_xor_sync(0xffffffffu, lt, 1);
            lt += __shfl_xor_sync(0xffffffffu, lt, 2);
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            if (rv[hr]) {
                uint32_t *orow = outg + (((int64_t)q0 + tok[hr]) * a.num_q_heads +
                                         (int64_t)kvh * g + head[hr]) * (kHeadDim / 2);
#pragma unroll
                for (int nt = 0; nt < 16; ++nt)
                    orow[nt * 4 + tig] = pack_bf16x2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
            }
        }
        __syncthreads();       // next query tile reuses the ring
    }
}

template <int G>
cudaError_t launch_prefill_g(const PrefillArgs &a, int max_query_len, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPfSmemBytes);
    if (e != cudaSuccess) return e;
    constexpr int BT = kPfRows / G;
    int gx = (max_query_len + BT - 1) / BT;
    gx = gx < 1 ? 1 : (gx > 65535 ? 65535 : gx);
    prefill_kernel<G><<<dim3(gx, a.num_seqs, a.num_kv_heads), kPfThreads, kPfSmemBytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t take_prefill_mma_error(cudaStream_t stream, int *code) {
    return take_device_word(g_prefill_mma_error, stream, code);
}

cudaError_t launch_prefill(const PrefillArgs &a, int group_pad, int max_query_len,
                           cudaStream_t stream) {
    switch (group_pad) {
        case 1: return launch_prefill_g<1>(a, max_query_len, stream);
        case 2: return launch_prefill_g<2>(a, max_query_len, stream);
        case 4: return launch_prefill_g<4>(a, max_query_len, stream);
        case 8: return launch_prefill_g<8>(a, max_query_len, stream);
        case 16: return launch_prefill_g<16>(a, max_query_len, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa

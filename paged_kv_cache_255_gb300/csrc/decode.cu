// Paged decode attention: one query token per sequence, K/V gathered through
// the sequence's block table from a pool of fixed-size blocks.
//
// What it computes: for sequence s, query head h, KV head kvh = h / g,
//   out[s][h] = sum_t softmax_t(scale * q[s][h] . K_t) V_t,  t < context_lens[s],
// where token t sits in physical block block_tables[s][t / bs], row t % bs
// ("Building a minimal vLLM implementation", sequence.py block_table;
// config.py kvcache_block_size). This is the engine's decode-side paged
// attention ("A vLLM engine small enough to read in one sitting").
//
// How the work is cut (GB300 design):
//   * A sequence's tokens form 16-token tiles; a (sequence, KV head) pair is a
//     unit of max(1, ceil(L / 16)) tiles. All units, sequence-major, form one
//     flat tile space of W tiles.
//   * P workers (one warp each, persistent: P = SMs x resident CTAs x warps)
//     take equal contiguous shares [w W / P, (w + 1) W / P) of that space, so
//     every SM streams the same number of bytes whatever the length mix. Every
//     CTA plans the split from context_lens in its prologue (before waiting on
//     the previous kernel when that is the same step's store).
//   * A worker streams its tiles through a private kStages-deep ring in shared
//     memory. One lane fills a stage with two TMA boxes (the K tile and the
//     V tile, each 16 rows x 128 head dims landing as two 64-dim halves,
//     128-byte swizzle) counted on the stage's mbarrier; every lane then waits on that barrier. A
//     tile with no tokens, or with a block id outside the pool, is
//     zero-filled by the warp instead, and the V rows of a sequence's last,
//     partly used tile are zeroed after they land. Per query head of its KV
//     head's group the worker keeps an online softmax (running max in log2
//     units, running sum) and an fp32 accumulator of P.V.
// Two interchangeable tile computations sit inside the same worker loop:
//   * MmaTile: q.K^T and P.V on the tensor cores with mma.sync m16n8k16 bf16
//     (fp32 accumulate): 16 tokens x 8 (or 16) query heads x 128 dims per
//     tile; the default.
//   * SimtTile: the same on the CUDA cores, lane l owning dims [4l, 4l + 4);
//     kept as the comparison and a second parity path, selected only by the
//     test hook pa_debug_kernel_variant.
// The kernels never wait on one another inside a launch; a warp waits only on
// its own copies, and every such wait is bounded (1 s, then the launch records
// code 2 and the warp exits).
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pa {

__device__ int g_decode_error;       // first device-side error of a decode launch

namespace {

constexpr int kWarps = 4;      // workers per CTA
// Ring depth: one tile in flight while the warp works on the other. With the
// ring this shallow, three CTAs fit an SM (12 warps), which measured faster
// than two CTAs of three-stage rings.
constexpr int kStages = 2;
constexpr int kBoxBytes = kTileBytes / 2;     // one half of a tile: 16 rows x 128 B (64 head dims)
constexpr int kStageBytes = 2 * kTileBytes;   // K tile then V tile
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kCombineBatch = 8;              // pieces a combine warp loads at once
constexpr float kNegInf = -INFINITY;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // bounded waits give up after 1 s

// Byte offset, inside a K or V tile in shared memory, of the 16-byte chunk
// holding head dims [8c, 8c + 8) of token row r. The tile lands as two halves
// (dims 0-63, then 64-127) of 16 rows x 128 B in the 128-byte swizzle: chunk
// k of a 128-byte row r sits at position k ^ (r % 8).
__device__ __forceinline__ uint32_t chunk_off(int r, int c) {
    return (uint32_t)((c >> 3) * kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// The warp waits until the phase of `bar` with the given parity completes.
// It first polls (every lane tests, a vote answers, __syncwarp orders the
// lanes that saw the completion before the rest; a suspended waiter would
// resume late), then lane 0 waits with a time limit. False when the limit
// ran out.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int lane) {
    for (int i = 0; i < 4096; ++i)
        if (__any_sync(0xffffffffu, tc::mbar_test_wait(bar, parity))) {
            __syncwarp();
            return true;
        }
    bool ok = true;
    if (lane == 0) {
        const uint64_t t0 = tc::globaltimer_ns();
        while (!tc::mbar_try_wait(bar, parity)) {
            if (tc::globaltimer_ns() - t0 > kWaitLimitNs) {
                ok = false;
                break;
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}

__device__ __forceinline__ int clamp_len(const int32_t *cl, int s, int max_len) {
    int L = __ldg(cl + s);
    L = L < 0 ? 0 : L;
    return L > max_len ? max_len : L;
}

// Tiles of a unit: a zero-length sequence still owns one (empty) tile so that
// some worker writes its zero output.
__device__ __forceinline__ int unit_tiles(int L) { return L > 0 ? (L + 15) >> 4 : 1; }

// Position in the flat tile space: sequence, KV head, tile within the unit.
struct Cursor {
    int s, kvh, j, nt, L;
};

__device__ __forceinline__ void cursor_advance(Cursor &c, const DecodeArgs &a, int max_len) {
    if (++c.j == c.nt) {
        c.j = 0;
        if (++c.kvh == a.num_kv_heads) {
            c.kvh = 0;
            if (++c.s < a.num_seqs) {
                c.L = clamp_len(a.context_lens, c.s, max_len);
                c.nt = unit_tiles(c.L);
            }
        }
    }
}

__device__ __forceinline__ int tile_valid(const Cursor &c) {
    int v = c.L - (c.j << 4);
    return v < 0 ? 0 : (v > 16 ? 16 : v);
}

// Physical block of the tile under the cursor (0 when the tile has no tokens).
__device__ __forceinline__ int tile_block(const Cursor &c, const DecodeArgs &a) {
    if (tile_valid(c) == 0) return 0;
    return __ldg(a.block_tables + (int64_t)c.s * a.max_blocks_per_seq +
                 ((c.j << 4) >> a.block_size_log2));
}

// Fill `stage` with the K tile and the V tile under cursor c (physical block
// bid): one TMA box each, issued by one elected lane and counted in bytes on `bar`.
// A tile with no tokens, or whose block id lies outside the pool, is written
// with zeros by the warp instead (each of its keys then scores 0 and adds a
// zero value) and `bar` gets a plain arrival. The stage's previous contents
// must have been read by every lane (the __syncwarp below orders that).
__device__ __forceinline__ void issue_tile(const Cursor &c, int bid, uint8_t *stage, uint32_t bar,
                                           const DecodeArgs &a, const CUtensorMap *mk,
                                           const CUtensorMap *mv, int lane) {
    const int valid = tile_valid(c);
    const bool bad = bid < 0 || (int64_t)bid >= a.num_blocks;   // never address outside the pool
    if (valid > 0 && bad && lane == 0) atomicCAS(&g_decode_error, 0, kErrBadBlock);
    __syncwarp();
    if (valid > 0 && !bad) {
        // one lane, chosen by elect.sync (the branch is warp-uniform): issued
        // from an elected lane rather than under lane == 0 the step measured
        // 1-5 % faster
        if (tc::elect_one()) {
            // token-major pool: (0, block * bs + offset, 0, KV head);
            // head-major pool: (0, offset, 0, block * Hkv + KV head)
            const int off = (c.j << 4) & ((1 << a.block_size_log2) - 1);
            const int row = a.head_major ? off : (bid << a.block_size_log2) + off;
            const int outer = a.head_major ? bid * a.num_kv_heads + c.kvh : c.kvh;
            const uint32_t dst = smem_u32(stage);
            mbar_arrive_expect_tx(bar, kStageBytes);
            tc::tma_load_4d(dst, mk, 0, row, 0, outer, bar);               // K tile
            tc::tma_load_4d(dst + kTileBytes, mv, 0, row, 0, outer, bar);  // V tile
        }
    } else {
        uint4 *z = reinterpret_cast<uint4 *>(stage);
#pragma unroll
        for (int i = 0; i < kStageBytes / 16 / 32; ++i) z[i * 32 + lane] = make_uint4(0u, 0u, 0u, 0u);
        tc::fence_proxy_async();    // a later TMA into this stage lands after these stores
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
    }
}

// Zero rows [valid, 16) of a V tile that has landed: keys past the sequence
// end get zero weight, but 0 x NaN would still be NaN. Chunk i of the tile is
// box i / 128, row (i / 8) % 16.
__device__ __forceinline__ void zero_v_tail(uint8_t *vtile, int valid, int lane) {
    uint4 *z = reinterpret_cast<uint4 *>(vtile);
#pragma unroll
    for (int k = 0; k < kTileBytes / 16 / 32; ++k) {
        const int i = k * 32 + lane;
        if (((i >> 3) & 15) >= valid) z[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_proxy_async();
    __syncwarp();
}

// Element offset of the q (and out) row of column c of a (sequence, KV head)
// unit. Columns are (query token i, head h of the group) pairs, c = i g + h;
// single-token decode has one query token, so columns are the group's heads.
__device__ __forceinline__ int64_t col_row(const DecodeArgs &a, int s, int kvh, int c) {
    const int g = a.group;
    const int i = c / g, h = c - i * g;
    return (((int64_t)s * a.q_len + i) * a.num_q_heads + (int64_t)kvh * g + h) * kHeadDim;
}

// Tokens column c may see in a sequence of L tokens: query token i of the
// q_len new ones sits at position L - q_len + i and sees t <= that position.
__device__ __forceinline__ int col_limit(const DecodeArgs &a, int L, int c) {
    const int lim = L - a.q_len + c / a.group + 1;
    return c < a.cols ? (lim > 0 ? lim : 0) : 0;
}

// ---------------------------------------------------------------------------
// Tile computation on the tensor cores.
//
// Scores as S^T = K Q^T: A = the K tile (16 tokens x 16 dims per k-step,
// ldmatrix from the swizzled stage), B = Q^T (16 dims x 8 heads, kept in
// registers for the unit), C = 16 tokens x 8 heads in fp32. Lane (gid =
// lane / 4, tig = lane % 4) holds tokens gid and gid + 8 of heads 2 tig and
// 2 tig + 1, so the per-head max over tokens is a 3-step xor reduction.
// P^T (bf16) becomes the B operand of O^T += V^T P^T through one movmatrix
// transpose per 8x8 half; A = V^T comes from the V tile by ldmatrix.trans.
// O^T (128 dims x 8 heads, fp32) lives in 8 m-tiles of 4 registers.
template <int GP>
struct MmaTile {
    static constexpr int NT = GP > 8 ? 2 : 1;      // 8-head column tiles
    static constexpr int kScratchFloats = 0;
    uint32_t qb[NT][8][2];
    float o[NT][8][4];
    float m[NT][2], l[NT][2];
    int lim[NT][2];     // tokens visible to this lane's two score columns per column tile

    __device__ __forceinline__ void begin(const DecodeArgs &a, const Cursor &cur, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        const uint16_t *qg = static_cast<const uint16_t *>(a.q);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int h = nt * 8 + gid;          // this lane's column of the Q^T operand
            lim[nt][0] = col_limit(a, cur.L, nt * 8 + 2 * tig);
            lim[nt][1] = col_limit(a, cur.L, nt * 8 + 2 * tig + 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t w0 = 0u, w1 = 0u;
                if (h < a.cols) {
                    const uint32_t *p = reinterpret_cast<const uint32_t *>(
                        qg + col_row(a, cur.s, cur.kvh, h) + kk * 16 + tig * 2);
                    w0 = __ldg(p);
                    w1 = __ldg(p + 4);
                }
                qb[nt][kk][0] = w0;
                qb[nt][kk][1] = w1;
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) o[nt][mt][i] = 0.f;
            m[nt][0] = m[nt][1] = kNegInf;
            l[nt][0] = l[nt][1] = 0.f;
        }
    }

    __device__ __forceinline__ void tile(const uint8_t *stage, int t0, float scale_log2,
                                         float *, int lane) {
        const uint32_t base = smem_u32(stage);
        const int i7 = lane & 7, mi = lane >> 3;
        const int gid = lane >> 2;

        float s[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
        // lane supplies row i7 + 8 (mi & 1), dim chunk 2 kk + (mi >> 1) of the K tile
        const uint32_t krow = base + (i7 + 8 * (mi & 1)) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a[4];
            ldmatrix_x4(krow + (kk >> 2) * kBoxBytes + ((((2 * kk + (mi >> 1)) & 7) ^ i7) << 4), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(s[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
        }

        // token t0 + gid (and + 8) is visible to a column below its limit
        const int r0 = t0 + gid, r1 = t0 + gid + 8;
        uint32_t pb0[NT], pb1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float s0 = r0 < lim[nt][0] ? s[nt][0] * scale_log2 : kNegInf;
            const float s1 = r0 < lim[nt][1] ? s[nt][1] * scale_log2 : kNegInf;
            const float s2 = r1 < lim[nt][0] ? s[nt][2] * scale_log2 : kNegInf;
            const float s3 = r1 < lim[nt][1] ? s[nt][3] * scale_log2 : kNegInf;
            float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
            for (int x = 4; x <= 16; x <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
            }
            const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
            const float ms0 = mn0 == kNegInf ? 0.f : mn0, ms1 = mn1 == kNegInf ? 0.f : mn1;
            // a column whose running max did not move keeps its scale exactly
            const float al0 = mn0 == m[nt][0] ? 1.f : ex2(m[nt][0] - ms0);
            const float al1 = mn1 == m[nt][1] ? 1.f : ex2(m[nt][1] - ms1);
            const uint32_t w0 = pack_bf16x2(ex2(s0 - ms0), ex2(s1 - ms1));   // token gid
            const uint32_t w1 = pack_bf16x2(ex2(s2 - ms0), ex2(s3 - ms1));   // token gid + 8
            // the running sum adds the same bf16-rounded weights the tensor cores use
            l[nt][0] = fmaf(l[nt][0], al0, bf16_lo(w0) + bf16_lo(w1));
            l[nt][1] = fmaf(l[nt][1], al1, bf16_hi(w0) + bf16_hi(w1));
            m[nt][0] = mn0;
            m[nt][1] = mn1;
            pb0[nt] = movmatrix_trans(w0);
            pb1[nt] = movmatrix_trans(w1);
            // rescale the accumulators only when some column's max moved
            // (rare once a long sequence's first tiles have been seen)
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    o[nt][mt][0] *= al0;
                    o[nt][mt][1] *= al1;
                    o[nt][mt][2] *= al0;
                    o[nt][mt][3] *= al1;
                }
            }
        }

        // lane supplies row i7 + 8 (mi >> 1), dim chunk 2 mt + (mi & 1) of the V tile
        const uint32_t vrow = base + kTileBytes + (i7 + 8 * (mi >> 1)) * 128;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t a[4];
            ldmatrix_x4_trans(vrow + (mt >> 2) * kBoxBytes + ((((2 * mt + (mi & 1)) & 7) ^ i7) << 4), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[nt][mt], a, pb0[nt], pb1[nt]);
        }
    }

    // Leave o[h][4 lane .. 4 lane + 3] (unnormalised) in `oc`, and the per-head
    // running max and total sum in sm_m / sm_l. `scr` is a free 8 KB stage.
    __device__ __forceinline__ void finish(float *scr, float *sm_m, float *sm_l, float (&oc)[GP][4],
                                           int lane) {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float lt0 = l[nt][0], lt1 = l[nt][1];
#pragma unroll
            for (int x = 4; x <= 16; x <<= 1) {
                lt0 += __shfl_xor_sync(0xffffffffu, lt0, x);
                lt1 += __shfl_xor_sync(0xffffffffu, lt1, x);
            }
            const int h0 = nt * 8 + 2 * tig;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int d0 = mt * 16 + gid;
                if (h0 < GP) {
                    scr[h0 * kHeadDim + d0] = o[nt][mt][0];
                    scr[h0 * kHeadDim + d0 + 8] = o[nt][mt][2];
                }
                if (h0 + 1 < GP) {
                    scr[(h0 + 1) * kHeadDim + d0] = o[nt][mt][1];
                    scr[(h0 + 1) * kHeadDim + d0 + 8] = o[nt][mt][3];
                }
            }
            if (gid == 0) {
                if (h0 < GP) {
                    sm_m[h0] = m[nt][0];
                    sm_l[h0] = lt0;
                }
                if (h0 + 1 < GP) {
                    sm_m[h0 + 1] = m[nt][1];
                    sm_l[h0 + 1] = lt1;
                }
            }
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            const float4 v = reinterpret_cast<const float4 *>(scr + h * kHeadDim)[lane];
            oc[h][0] = v.x;
            oc[h][1] = v.y;
            oc[h][2] = v.z;
            oc[h][3] = v.w;
        }
    }
};

// ---------------------------------------------------------------------------
// Tile computation on the CUDA cores: lane l owns head dims [4l, 4l + 4) of
// every query head of the group.

// Sum NV per-lane values across the 32 lanes, halving the set at each of the
// five xor steps: afterwards lane l holds max(1, NV / 32) fully reduced
// values, originally at indices l * NV / 32 + i (NV >= 32) or l >> 1 (NV = 16).
template <int NV>
__device__ __forceinline__ void butterfly_sum(float (&v)[NV], int lane) {
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int mask = 16 >> step;
        const int n = NV >> step;
        if (n >= 2) {
            const bool upper = lane & mask;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
                const float send = upper ? v[i] : v[i + n / 2];
                const float keep = upper ? v[i + n / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
            }
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
        }
    }
}

template <int GP>
struct SimtTile {
    static constexpr int HP = GP >= 2 ? GP / 2 : 1;     // heads whose scores a lane holds
    static constexpr int kScratchFloats = 16 * GP + GP;  // p[16][GP], alpha[GP]
    float qf[GP][4], o[GP][4], m_run[HP], l_run[HP];
    int L_;             // tokens of the unit's sequence (one query token per sequence)

    __device__ __forceinline__ void begin(const DecodeArgs &a, const Cursor &cur, int lane) {
        const uint16_t *qg = static_cast<const uint16_t *>(a.q);
        L_ = cur.L;
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            uint2 u = make_uint2(0u, 0u);
            if (h < a.cols)
                u = __ldg(reinterpret_cast<const uint2 *>(qg + col_row(a, cur.s, cur.kvh, h)) + lane);
            qf[h][0] = bf16_lo(u.x);
            qf[h][1] = bf16_hi(u.x);
            qf[h][2] = bf16_lo(u.y);
            qf[h][3] = bf16_hi(u.y);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[h][i] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < HP; ++c) {
            m_run[c] = kNegInf;
            l_run[c] = 0.f;
        }
    }

    __device__ __forceinline__ void tile(const uint8_t *stage, int t0, float scale_log2,
                                         float *scratch, int lane) {
        const int valid = L_ - t0 < 0 ? 0 : (L_ - t0 > 16 ? 16 : L_ - t0);
        const uint8_t *sk = stage;
        const uint8_t *sv = stage + kTileBytes;
        float *sp = scratch;              // p[16][GP]
        float *sa = scratch + 16 * GP;    // alpha[GP]
        const int t_lane = lane >> 1;
        const int hb = GP >= 2 ? (lane & 1) * HP : 0;

        float part[16 * GP];
        // lane l reads dims [4l, 4l + 4): half of 16-byte chunk l / 2 of each row
        const uint32_t lane_half = (lane & 1) * 8;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const uint2 u = *reinterpret_cast<const uint2 *>(sk + chunk_off(t, lane >> 1) + lane_half);
            const float k0 = bf16_lo(u.x), k1 = bf16_hi(u.x), k2 = bf16_lo(u.y), k3 = bf16_hi(u.y);
#pragma unroll
            for (int h = 0; h < GP; ++h)
                part[t * GP + h] = fmaf(qf[h][3], k3, fmaf(qf[h][2], k2, fmaf(qf[h][1], k1, qf[h][0] * k0)));
        }
        butterfly_sum<16 * GP>(part, lane);

        const bool tok_ok = t_lane < valid;
#pragma unroll
        for (int c = 0; c < HP; ++c) {
            const float s = tok_ok ? part[c] * scale_log2 : kNegInf;
            float mx = s;
#pragma unroll
            for (int x = 2; x <= 16; x <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, x));
            const float m_new = fmaxf(m_run[c], mx);
            const float ms = m_new == kNegInf ? 0.f : m_new;
            const float alpha = ex2(m_run[c] - ms);
            const float p = ex2(s - ms);
            l_run[c] = fmaf(l_run[c], alpha, p);
            m_run[c] = m_new;
            sp[t_lane * GP + hb + c] = p;
            if (t_lane == 0) sa[hb + c] = alpha;
        }
        __syncwarp();

#pragma unroll
        for (int h = 0; h < GP; ++h) {
            const float al = sa[h];
#pragma unroll
            for (int i = 0; i < 4; ++i) o[h][i] *= al;
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const uint2 u = *reinterpret_cast<const uint2 *>(sv + chunk_off(t, lane >> 1) + lane_half);
            const float v0 = bf16_lo(u.x), v1 = bf16_hi(u.x), v2 = bf16_lo(u.y), v3 = bf16_hi(u.y);
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                const float p = sp[t * GP + h];
                o[h][0] = fmaf(p, v0, o[h][0]);
                o[h][1] = fmaf(p, v1, o[h][1]);
                o[h][2] = fmaf(p, v2, o[h][2]);
                o[h][3] = fmaf(p, v3, o[h][3]);
            }
        }
        __syncwarp();
    }

    __device__ __forceinline__ void finish(float *, float *sm_m, float *sm_l, float (&oc)[GP][4],
                                           int lane) {
        const int t_lane = lane >> 1;
        const int hb = GP >= 2 ? (lane & 1) * HP : 0;
#pragma unroll
        for (int c = 0; c < HP; ++c) {
            float x = l_run[c];
#pragma unroll
            for (int msk = 2; msk <= 16; msk <<= 1) x += __shfl_xor_sync(0xffffffffu, x, msk);
            if (t_lane == 0) {
                sm_m[hb + c] = m_run[c];
                sm_l[hb + c] = x;
            }
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < GP; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) oc[h][i] = o[h][i];
    }
};

// Shared memory of a CTA, from a 1024-byte aligned start (the 128-byte swizzle
// of the TMA boxes repeats every 1024 bytes): every warp's ring, then per warp
// its stage barriers, the tile scratch and m / l per head.
template <class Tile, int GP>
struct Layout {
    static constexpr int kSmallFloats = Tile::kScratchFloats + 2 * GP;
    static constexpr int kSmallBytes = ((8 * kStages + kSmallFloats * 4 + 127) / 128) * 128;
    static constexpr int kCtaBytes = 1024 + kWarps * (kRingBytes + kSmallBytes);   // + alignment slack
};

// CTA prologue: the total tile count W, the share count actually used, and
// the position (sequence, KV head, tile) of this warp's first tile.
__device__ __forceinline__ void plan_share(const DecodeArgs &a, int max_len, int64_t &W,
                                           int &p_eff, int64_t &T0, int64_t &T1, Cursor &c) {
    __shared__ long long s_wsum[kWarps];
    __shared__ long long s_scan[kWarps * 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.num_seqs, Hkv = a.num_kv_heads;

    // pass 1: total tiles
    long long local = 0;
    for (int s = threadIdx.x; s < S; s += kWarps * 32)
        local += unit_tiles(clamp_len(a.context_lens, s, max_len));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) local += __shfl_xor_sync(0xffffffffu, local, m);
    if (lane == 0) s_wsum[warp] = local;
    __syncthreads();
    long long total = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) total += s_wsum[i];
    __syncthreads();
    W = total * Hkv;

    int64_t pe = W / (a.min_tiles > 0 ? a.min_tiles : 1);
    if (pe < 1) pe = 1;
    if (pe > a.num_workers) pe = a.num_workers;
    p_eff = (int)pe;
    const int w = blockIdx.x * kWarps + warp;
    if (w < p_eff) {
        T0 = (int64_t)w * W / p_eff;
        T1 = (int64_t)(w + 1) * W / p_eff;
    } else {
        T0 = T1 = W;
    }

    // pass 2: chunked inclusive scan of tiles per sequence; each warp finds
    // the sequence holding tile T0
    bool found = T0 >= T1;
    long long base = 0;
    for (int c0 = 0; c0 < S; c0 += kWarps * 32) {
        const int s = c0 + threadIdx.x;
        long long v = s < S ? unit_tiles(clamp_len(a.context_lens, s, max_len)) : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long n = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += n;
        }
        if (lane == 31) s_wsum[warp] = v;
        __syncthreads();
        long long woff = base;
        for (int i = 0; i < warp; ++i) woff += s_wsum[i];
        s_scan[threadIdx.x] = v + woff;
        __syncthreads();
        const long long chunk_end = s_scan[kWarps * 32 - 1];
        if (!found && T0 < chunk_end * Hkv) {
            int hit_i = -1;
            for (int i0 = 0; i0 < kWarps * 32 && hit_i < 0; i0 += 32) {
                const unsigned msk = __ballot_sync(0xffffffffu, s_scan[i0 + lane] * Hkv > T0);
                if (msk) hit_i = i0 + __ffs(msk) - 1;
            }
            const long long excl = hit_i == 0 ? base : s_scan[hit_i - 1];
            const long long nt = s_scan[hit_i] - excl;
            const long long rem = T0 - excl * Hkv;
            c.s = c0 + hit_i;
            c.kvh = (int)(rem / nt);
            c.j = (int)(rem % nt);
            c.nt = (int)nt;
            c.L = clamp_len(a.context_lens, c.s, max_len);
            found = true;
        }
        base = chunk_end;
        __syncthreads();
    }
}

// L2 prefetch of context_lens, block_tables and q, in 128-byte lines spread
// over every thread of the grid.
__device__ __forceinline__ void prefetch_inputs(const DecodeArgs &a) {
    const int64_t n_cl = ((int64_t)a.num_seqs * 4 + 127) >> 7;
    const int64_t n_bt = ((int64_t)a.num_seqs * a.max_blocks_per_seq * 4 + 127) >> 7;
    const int64_t n_q = ((int64_t)a.num_seqs * a.num_q_heads * kRowBytes + 127) >> 7;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_cl + n_bt + n_q;
         i += stride) {
        const char *p = i < n_cl ? reinterpret_cast<const char *>(a.context_lens) + (i << 7)
                      : i < n_cl + n_bt
                          ? reinterpret_cast<const char *>(a.block_tables) + ((i - n_cl) << 7)
                          : static_cast<const char *>(a.q) + ((i - n_cl - n_bt) << 7);
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
    }
}

template <class Tile, int GP>
__global__ void __launch_bounds__(kWarps * 32)
decode_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v) {
    using Lay = Layout<Tile, GP>;
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *ring = smem + warp * kRingBytes;
    uint8_t *small = smem + kWarps * kRingBytes + warp * Lay::kSmallBytes;
    const uint32_t bar0 = smem_u32(small);                      // kStages mbarriers
    float *scratch = reinterpret_cast<float *>(small + 8 * kStages);
    float *sm_m = scratch + Tile::kScratchFloats;
    float *sm_l = sm_m + GP;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kStages; ++i) tc::mbar_init(bar0 + 8 * i, 1);
        tc::fence_mbar_init();
    }
    __syncwarp();

    // Launched as a programmatic dependent of the previous kernel in the
    // stream (normally the store of this step's K/V rows). While that kernel
    // may still run, pull this launch's small inputs (lengths, tables, q) into
    // L2; a prefetch reads nothing into registers, and L2 is the point of
    // coherence, so a later write by that kernel still wins. Then wait until
    // it has finished and its writes are visible before reading anything, and
    // let the combine launch queue up behind this grid. When the previous
    // kernel is known to be this step's store (plan_early), which writes the
    // caches only, the split of the work is planned from the lengths first.
    prefetch_inputs(a);
    if (!a.plan_early) {
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    }

    const int max_len = (int)min((int64_t)a.max_blocks_per_seq << a.block_size_log2,
                                 (int64_t)0x7fffffff);
    int64_t W, T0, T1;
    int p_eff;
    Cursor cc{0, 0, 0, 1, 0};
    plan_share(a, max_len, W, p_eff, T0, T1, cc);
    if (a.plan_early) {
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    }
    const int w = blockIdx.x * kWarps + warp;
    if (w >= a.num_workers) return;
    if (T0 >= T1) {
        if (lane == 0) a.tasks[w] = make_int4(-1, 0, 0, 0);
        return;
    }

    uint32_t *outg = static_cast<uint32_t *>(a.out);
    uint32_t phase = 0;      // bit i: parity of stage i's next barrier phase
    uint32_t pending = 0;    // bit i: stage i has been filled and not yet waited for

    // producer: runs kStages - 1 tiles ahead of the consumer
    Cursor pc = cc;
    int64_t Tp = T0;
    int p_bid = tile_block(pc, a);
    int stage_p = 0;
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) {
        if (Tp < T1) {
            issue_tile(pc, p_bid, ring + stage_p * kStageBytes, bar0 + 8 * stage_p, a, &tmap_k,
                       &tmap_v, lane);
            pending |= 1u << stage_p;
            cursor_advance(pc, a, max_len);
            ++Tp;
            p_bid = Tp < T1 ? tile_block(pc, a) : 0;
        }
        stage_p = stage_p + 1 == kStages ? 0 : stage_p + 1;
    }

    Tile tl;
    int stage_c = 0;
    int piece = 0;              // index of the current piece within this share
    bool fresh = true;          // next tile starts a piece
    int64_t piece_T = T0;       // flat index of the piece's first tile
    int piece_j0 = 0;
    int4 task = make_int4(-1, 0, 0, 0);
    bool failed = false;

    for (int64_t T = T0; T < T1; ++T) {
        if (Tp < T1) {
            issue_tile(pc, p_bid, ring + stage_p * kStageBytes, bar0 + 8 * stage_p, a, &tmap_k,
                       &tmap_v, lane);
            pending |= 1u << stage_p;
            cursor_advance(pc, a, max_len);
            ++Tp;
            p_bid = Tp < T1 ? tile_block(pc, a) : 0;
        }
        stage_p = stage_p + 1 == kStages ? 0 : stage_p + 1;

        if (fresh) {
            fresh = false;
            piece_T = T;
            piece_j0 = cc.j;
            tl.begin(a, cc, lane);
        }

        if (!warp_wait(bar0 + 8 * stage_c, (phase >> stage_c) & 1u, lane)) {
            failed = true;
            break;
        }
        phase ^= 1u << stage_c;
        pending &= ~(1u << stage_c);
        uint8_t *stage = ring + stage_c * kStageBytes;
        const int valid = tile_valid(cc);
        if (valid > 0 && valid < 16) zero_v_tail(stage + kTileBytes, valid, lane);
        tl.tile(stage, cc.j << 4, a.scale_log2, scratch, lane);
        stage_c = stage_c + 1 == kStages ? 0 : stage_c + 1;

        const bool unit_end = cc.j == cc.nt - 1;
        if (unit_end || T == T1 - 1) {
            // the stage just consumed is refilled only at the next iteration:
            // it serves as transpose scratch here
            float oc[GP][4];
            __syncwarp();
            tl.finish(reinterpret_cast<float *>(stage), sm_m, sm_l, oc, lane);
            tc::fence_proxy_async();     // the TMA that refills the stage lands after these stores
            __syncwarp();
            if (piece_j0 == 0 && unit_end) {
                // the whole unit is in this share: normalise and write bf16
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    if (h < a.cols) {
                        const float l = sm_l[h];
                        const float inv = l > 0.f ? 1.f / l : 0.f;
                        uint2 pk;
                        pk.x = pack_bf16x2(oc[h][0] * inv, oc[h][1] * inv);
                        pk.y = pack_bf16x2(oc[h][2] * inv, oc[h][3] * inv);
                        reinterpret_cast<uint2 *>(outg + col_row(a, cc.s, cc.kvh, h) / 2)[lane] = pk;
                    }
                }
            } else {
                // a piece of a unit that other shares continue
                const int slot = 2 * w + (piece == 0 ? 0 : 1);
                float *po = a.part_o + (int64_t)slot * GP * kHeadDim;
#pragma unroll
                for (int h = 0; h < GP; ++h)
                    reinterpret_cast<float4 *>(po + h * kHeadDim)[lane] =
                        make_float4(oc[h][0], oc[h][1], oc[h][2], oc[h][3]);
                if (lane < GP)
                    reinterpret_cast<float2 *>(a.part_ml)[(int64_t)slot * GP + lane] =
                        make_float2(sm_m[lane], sm_l[lane]);
                if (piece_j0 == 0) {
                    // this share holds the unit's first tile: it owns the combine
                    const int64_t unit_end_T = piece_T + cc.nt;
                    const int w_last = (int)((unit_end_T * p_eff - 1) / W);
                    task = make_int4(cc.s, cc.kvh, slot, w_last);
                }
            }
            __syncwarp();
            ++piece;
            fresh = true;
        }
        cursor_advance(cc, a, max_len);
    }
    if (failed) {
        // a copy did not land in time: record it, give the copies still in
        // flight into this warp's ring a bounded chance to land, own no
        // combine task, and stop (the launch's outputs are undefined)
        if (lane == 0) atomicCAS(&g_decode_error, 0, kErrTimeout);
        for (int i = 0; i < kStages; ++i)
            if ((pending >> i) & 1u && i != stage_c) warp_wait(bar0 + 8 * i, (phase >> i) & 1u, lane);
        task = make_int4(-1, 0, 0, 0);
    }
    if (lane == 0) a.tasks[w] = task;
}

// Log-sum-exp merge of the pieces of each split unit. Block (x, y) holds
// four warps, one per worker task 4x .. 4x + 3, all on column y; lane l
// handles dims [4l, 4l + 4). One online pass over the pieces: each piece's
// (max, sum, o) is folded in with weights 2^(m_i - M). The pieces are read
// in batches whose loads are all issued before the batch is merged, so that
// a unit cut into n pieces costs about n / kCombineBatch memory round trips.
template <int GP>
__global__ void __launch_bounds__(128) combine_kernel(const DecodeArgs a) {
    // programmatic dependent of the decode grid: wait for all of it (and its
    // writes) before reading any task or partial result
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = blockIdx.x * 4 + warp;
    const int h = blockIdx.y;
    if (w >= a.num_workers || h >= a.cols) return;
    const int4 task = a.tasks[w];
    if (task.x < 0) return;
    const int n = 1 + task.w - w;
    const float2 *ml = reinterpret_cast<const float2 *>(a.part_ml);
    float M = kNegInf, L = 0.f, acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    // pieces in batches: a batch's loads are all in flight before its merge
    for (int i0 = 0; i0 < n; i0 += kCombineBatch) {
        float2 eb[kCombineBatch];
        float4 ob[kCombineBatch];
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {
            const int i = i0 + k;
            if (i < n) {
                const int slot = i == 0 ? task.z : 2 * (w + i);
                eb[k] = ml[(int64_t)slot * GP + h];
                ob[k] = reinterpret_cast<const float4 *>(a.part_o + ((int64_t)slot * GP + h) * kHeadDim)[lane];
            }
        }
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {
            if (i0 + k >= n) break;
            const float2 e = eb[k];
            const float4 po = ob[k];
            if (e.x == kNegInf) continue;    // no visible token of this column in the piece
            const float Mn = fmaxf(M, e.x);
            const float a_old = ex2(M - Mn), a_new = ex2(e.x - Mn);
            L = L * a_old + e.y * a_new;
            acc0 = acc0 * a_old + po.x * a_new;
            acc1 = acc1 * a_old + po.y * a_new;
            acc2 = acc2 * a_old + po.z * a_new;
            acc3 = acc3 * a_old + po.w * a_new;
            M = Mn;
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(acc0 * inv, acc1 * inv);
    pk.y = pack_bf16x2(acc2 * inv, acc3 * inv);
    reinterpret_cast<uint2 *>(static_cast<uint32_t *>(a.out) + col_row(a, task.x, task.y, h) / 2)[lane] = pk;
}

template <class Tile, int GP>
struct Launcher {
    using Lay = Layout<Tile, GP>;
    static cudaError_t prepare() {
        return cudaFuncSetAttribute(decode_kernel<Tile, GP>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kCtaBytes);
    }
    static int ctas_per_sm() {
        if (prepare() != cudaSuccess) return 0;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<Tile, GP>, kWarps * 32,
                                                          Lay::kCtaBytes) != cudaSuccess)
            return 0;
        return n;
    }
    // Both kernels go out as programmatic dependent launches: each may be
    // scheduled while the kernel before it in the stream is still running, and
    // waits for it (griddepcontrol.wait) before touching its results.
    static cudaError_t launch_pdl(const void *fn, dim3 grid, unsigned block, size_t smem,
                                  void **args, cudaStream_t st) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(block);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelExC(&cfg, fn, args);
    }
    static cudaError_t launch(const DecodeArgs &a, cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        CUtensorMap mk, mv;
        const int bs = 1 << a.block_size_log2;
        if (!make_tile_map(&mk, a.k_cache, a.num_blocks, bs, a.num_kv_heads, a.head_major != 0) ||
            !make_tile_map(&mv, a.v_cache, a.num_blocks, bs, a.num_kv_heads, a.head_major != 0))
            return cudaErrorInvalidValue;
        const unsigned grid = (a.num_workers + kWarps - 1) / kWarps;
        DecodeArgs args_copy = a;
        void *dargs[] = {&args_copy, &mk, &mv};
        e = launch_pdl(reinterpret_cast<const void *>(&decode_kernel<Tile, GP>), dim3(grid),
                       kWarps * 32, Lay::kCtaBytes, dargs, st);
        if (e != cudaSuccess) return e;
        void *cargs[] = {&args_copy};
        e = launch_pdl(reinterpret_cast<const void *>(&combine_kernel<GP>),
                       dim3((a.num_workers + 3) / 4, a.cols), 128, 0, cargs, st);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
};

template <int GP>
int ctas_per_sm_for(DecodeKernel k) {
    return k == DecodeKernel::kSimt ? Launcher<SimtTile<GP>, GP>::ctas_per_sm()
                                    : Launcher<MmaTile<GP>, GP>::ctas_per_sm();
}

template <int GP>
cudaError_t launch_for(const DecodeArgs &a, DecodeKernel k, cudaStream_t st) {
    return k == DecodeKernel::kSimt ? Launcher<SimtTile<GP>, GP>::launch(a, st)
                                    : Launcher<MmaTile<GP>, GP>::launch(a, st);
}

// The CUDA-core tile keeps 16 x GP partial scores per lane: GP = 16 does not fit.
template <>
int ctas_per_sm_for<16>(DecodeKernel) {
    return Launcher<MmaTile<16>, 16>::ctas_per_sm();
}
template <>
cudaError_t launch_for<16>(const DecodeArgs &a, DecodeKernel, cudaStream_t st) {
    return Launcher<MmaTile<16>, 16>::launch(a, st);
}

}  // namespace

cudaError_t take_decode_error(cudaStream_t stream, int *code) {
    return take_device_word(g_decode_error, stream, code);
}

int decode_group_pad(int group) {
    if (group < 1) return 0;
    int gp = 1;
    while (gp < group) gp <<= 1;
    return gp <= 16 ? gp : 0;
}

int decode_default_workers(int group_pad, DecodeKernel k, int sm_count) {
    int per_sm = 0;
    switch (group_pad) {
        case 1: per_sm = ctas_per_sm_for<1>(k); break;
        case 2: per_sm = ctas_per_sm_for<2>(k); break;
        case 4: per_sm = ctas_per_sm_for<4>(k); break;
        case 8: per_sm = ctas_per_sm_for<8>(k); break;
        case 16: per_sm = ctas_per_sm_for<16>(k); break;
        default: return 0;
    }
    if (per_sm < 1) return 0;
    return sm_count * per_sm * kWarps;
}

size_t decode_workspace_bytes(int group_pad, int num_workers) {
    const size_t P = (size_t)num_workers;
    return 2 * P * group_pad * kHeadDim * sizeof(float)   // part_o
           + 2 * P * group_pad * 2 * sizeof(float)         // part_ml
           + P * sizeof(int4);                             // tasks
}

void decode_carve_workspace(DecodeArgs &a, void *workspace, int group_pad) {
    const size_t P = (size_t)a.num_workers;
    char *p = static_cast<char *>(workspace);
    a.part_o = reinterpret_cast<float *>(p);
    p += 2 * P * group_pad * kHeadDim * sizeof(float);
    a.part_ml = reinterpret_cast<float *>(p);
    p += 2 * P * group_pad * 2 * sizeof(float);
    a.tasks = reinterpret_cast<int4 *>(p);
}

cudaError_t launch_decode(const DecodeArgs &a, int group_pad, DecodeKernel k, cudaStream_t stream) {
    switch (group_pad) {
        case 1: return launch_for<1>(a, k, stream);
        case 2: return launch_for<2>(a, k, stream);
        case 4: return launch_for<4>(a, k, stream);
        case 8: return launch_for<8>(a, k, stream);
        case 16: return launch_for<16>(a, k, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa

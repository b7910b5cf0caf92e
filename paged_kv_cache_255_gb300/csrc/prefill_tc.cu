// Paged prefill on the 5th-generation tensor cores (tcgen05): the same
// attention as prefill.cu (chunk rows of a sequence attend causally to its
// tokens in the paged KV cache; "A vLLM engine small enough to read in one
// sitting": prefill and decode run over the paged KV cache, flash attention
// for prefill), computed in the flash-attention order with both contractions
// on tcgen05.mma, S, P and O in tensor memory.
//
// One CTA per SM works through items: an item is two 128-row query tiles A
// and B of one (sequence, KV head); a tile is 128 / G query tokens x the G
// query heads of the group (G = group size rounded up to a power of two), so
// every K/V tile fetched serves 256 rows. Keys go in tiles of 128. TMEM (512
// columns): S_A 0-127, O_A 128-255, S_B 256-383, O_B 384-511; P_t (bf16, two
// per column) overwrites the first 64 columns of S_t.
//
// Work is handed out by grid cell (KV head, pair slot, sequence rank; heaviest
// first in launch order). A CTA runs its own cell, then, through cluster
// launch control, takes over cells whose CTAs have not been launched yet and
// runs them too, keeping its TMEM, barriers and pipelines: the next item's Q
// and first K/V tiles load while the current item finishes, and the cells are
// still walked in launch order with a dynamic balance. Warp roles:
//   warps 0-3, 4-7   softmax of tile A, B: thread t of the warpgroup owns row
//                    t (TMEM lane t). Per key tile j it reads its row of S_j
//                    (tcgen05.ld, two passes: the max, then P), masks it
//                    causally on the tiles that reach its limit, keeps a
//                    running max (raised only when a tile's max exceeds it by
//                    more than 2^8 in exp2 units; then it rescales its row of
//                    O in TMEM) and sum, and writes P_j (tcgen05.st).
//   warps 8, 9       K and V producers: per tile, 16 lanes each fetch one
//                    box of 16 tokens x 64 dims of one KV head by TMA through
//                    a 3-D tensor map over the pool (either layout),
//                    landing in the 128-byte swizzled layout the MMA
//                    descriptors name, into 3 K stages and 2 V stages. V rows
//                    of a partly used 16-token group at the end of the keys
//                    are copied (rows past the end zeroed) by the lanes. The
//                    V producer also loads each item's two query tiles by TMA
//                    (a 3-D tensor map over q: dims x heads x tokens) once the
//                    previous item's MMAs are done with the Q buffers (a warp
//                    of its own for Q made the other roles' code measurably
//                    slower). The K producer publishes the next cell once it
//                    has issued the current one's last K tile.
//   warp 10          issues the MMAs (converged warp, one elected lane):
//                      S_t(j)  = Q_t K_j^T      M 128, N 128, K 16 x 8 (smem, smem)
//                      O_t    += P_t(j) V_j     M 128, N 128, K 16 x 8 (TMEM, smem)
//                    as soon as their inputs are ready; S_t(j + 1) follows
//                    PV_t(j) in issue order, so the tensor core has read P_t(j)
//                    before S_t(j + 1) overwrites it, and a softmax warp that
//                    sees S_t(j + 1) knows PV_t(j) has finished (O is stable).
//                    16-token V groups wholly past the end of the keys are
//                    left out of PV.
//
// Hand-offs are mbarriers: k_full / v_full complete when the TMA bytes have
// landed and the producer warp has arrived (after fencing its own
// shared-memory writes to the async proxy); q_full when the Q copies have
// landed; unit_full / unit_empty hand the next cell's descriptor from the K
// producer to the other warps; tcgen05.commit arrives on s_full, pv_done,
// k_empty and v_empty; the softmax warps arrive on p_ready once P is in TMEM
// (and O rescaled), and on o_free once the epilogue has read O. Every wait is
// bounded (about 2 s) and also gives up once any thread of the CTA has
// recorded a failed wait; then every role skips to the end, where the CTA
// frees its TMEM and exits.
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pa {

__device__ int g_prefill_error;      // first device-side error of a prefill launch

namespace {

constexpr int kRows = 128;                              // rows per query tile
constexpr int kKeys = 128;                              // keys per K/V tile
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kSoftmaxThreads = 256;
constexpr int kKWarp = kSoftmaxThreads / 32;             // 8
constexpr int kVWarp = kKWarp + 1;                       // 9
constexpr int kMmaWarp = kKWarp + 2;                     // 10
constexpr int kThreads = kSoftmaxThreads + 3 * 32;
constexpr int kGroup = 16;                               // tokens per TMA box
constexpr int kGroups = kKeys / kGroup;                  // 8
constexpr uint32_t kQBytes = kRows * kRowBytes;         // 32 KB: 2 K-halves of [128][128 B]
constexpr uint32_t kQHalf = kRows * 128;                // 16 KB
constexpr uint32_t kKVBytes = kKeys * kRowBytes;        // 32 KB: 2 halves of [128][128 B]
constexpr uint32_t kKVHalf = kKeys * 128;               // 16 KB
constexpr uint32_t kOffQ = 0;                           // Q_A, Q_B
constexpr uint32_t kOffK = kOffQ + 2 * kQBytes;         // K stages
constexpr uint32_t kOffV = kOffK + kKStages * kKVBytes; // V stages
constexpr uint32_t kOffCtl = kOffV + kVStages * kKVBytes;
// control block: mbarriers (8 B each), then the TMEM base and the abort flag
constexpr uint32_t kBarQFull = 0;
constexpr uint32_t kBarQEmpty = 1;
constexpr uint32_t kBarKFull = 2;                        // + stage
constexpr uint32_t kBarKEmpty = kBarKFull + kKStages;    // + stage
constexpr uint32_t kBarVFull = kBarKEmpty + kKStages;    // + stage
constexpr uint32_t kBarVEmpty = kBarVFull + kVStages;    // + stage
constexpr uint32_t kBarSFull = kBarVEmpty + kVStages;    // + query tile (A 0, B 1)
constexpr uint32_t kBarPReady = kBarSFull + 2;
constexpr uint32_t kBarPVDone = kBarPReady + 2;
constexpr uint32_t kBarOFree = kBarPVDone + 2;
constexpr uint32_t kBarUnitFull = kBarOFree + 2;         // + unit ring slot
constexpr uint32_t kBarUnitEmpty = kBarUnitFull + 2;     // + unit ring slot
constexpr uint32_t kBarClc = kBarUnitEmpty + 2;          // launch-control responses
constexpr uint32_t kNumBars = kBarClc + 1;
constexpr uint32_t kOffTmemSlot = kOffCtl + 8 * kNumBars;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
// heavy-first sequence order (up to kRankMaxSeqs sequences): their lengths,
// query starts and the sequence of each rank, staged once per CTA
constexpr int kRankMaxSeqs = 256;
constexpr uint32_t kOffSeqLens = kOffCtl + 256;
constexpr uint32_t kOffSeqStarts = kOffSeqLens + 4 * kRankMaxSeqs;
constexpr uint32_t kOffRankSeq = kOffSeqStarts + 4 * (kRankMaxSeqs + 1);       // uint16 per rank
constexpr uint32_t kOffUnits = (kOffRankSeq + 2 * kRankMaxSeqs + 15) & ~15u;  // 2 UnitDesc
constexpr uint32_t kOffClcResp = kOffUnits + 64;                              // 16 B, 16-aligned
constexpr uint32_t kSmemBytes = kOffClcResp + 16;
static_assert(kOffAbort + 4 <= kOffSeqLens, "control block");
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr int kUnitReaders = kThreads / 32;              // every warp reads each unit
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescS = tc::idesc_bf16(128, kKeys, false);
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, true);
constexpr float kRescaleSlack = 8.f;                    // log2 units
constexpr int kPairsPerCta = 1;                         // query-tile pairs per CTA (grid sizing)

__device__ __forceinline__ void set_error(int code) { atomicCAS(&g_prefill_error, 0, code); }

// Three-input max / min (one instruction on sm_100-family parts).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// Bounded wait that also gives up once the CTA's abort flag is set.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer_ns();
    for (;;) {
        if (tc::mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (*abort) return false;
        if (tc::globaltimer_ns() - t0 > 2000000000ull) {
            set_error(kErrTimeout);
            *abort = 1;
            return false;
        }
    }
}

// Warp-level hand-offs: one lane waits (or arrives) for the whole warp, the
// others are ordered with it by __syncwarp. With `spin` (the waits on the
// per-tile chain), the warp first polls: every lane tests the barrier (one
// shared-memory access, no divergent branch), a vote gives one answer and
// __syncwarp orders the lanes that saw the phase complete before the rest.
// A thread that try_wait has suspended resumes some hundreds of cycles after
// the phase completes, which those hand-offs cannot afford.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          bool spin = false) {
    if (spin) {
        for (int i = 0; i < 256; ++i)
            if (__any_sync(0xffffffffu, tc::mbar_test_wait(bar, parity))) {
                __syncwarp();
                return true;
            }
    }
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort);
    const bool r = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return r;
}
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Physical row (token slot) of key t of sequence s in the pool, or -1.
__device__ __forceinline__ int64_t key_row(const PrefillArgs &a, int s, int t) {
    const int bid = __ldg(a.block_tables + (int64_t)s * a.max_blocks_per_seq + (t >> a.block_size_log2));
    if (bid < 0 || (int64_t)bid >= a.num_blocks) {   // the rows read as zeros
        set_error(kErrBadBlock);
        return -1;
    }
    return ((int64_t)bid << a.block_size_log2) + (t & ((1 << a.block_size_log2) - 1));
}

// The V rows of the 16-token group starting at key t0 (which holds the end
// kend of the keys) into its place in a V stage, by the 32 lanes of a warp;
// rows at or past kend are zero. Plain loads and shared stores.
__device__ __forceinline__ void copy_v_tail(const PrefillArgs &a, int s, int kvh, int t0, int kend,
                                            uint32_t vdst, int lane) {
    const int chunk = lane & 15;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (lane >> 4) + 2 * i;          // row of the group
        const int t = t0 + r;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (t < kend) {
            const int64_t slot = key_row(a, s, t);
            if (slot >= 0) {
                const int lb = a.block_size_log2;
                const int64_t row = a.head_major
                    ? (((slot >> lb) * a.num_kv_heads + kvh) << lb) + (slot & ((1 << lb) - 1))
                    : slot * a.num_kv_heads + kvh;
                w = __ldg(reinterpret_cast<const uint4 *>(
                    static_cast<const char *>(a.v_cache) + row * kRowBytes + chunk * 16));
            }
        }
        const int key = (t0 & (kKeys - 1)) + r;     // row in the tile
        const uint32_t dst = vdst + (chunk >> 3) * kKVHalf + key * 128 +
                             ((((uint32_t)chunk & 7) ^ ((uint32_t)key & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(w.x), "r"(w.y),
                     "r"(w.z), "r"(w.w)
                     : "memory");
    }
}

// 16-token groups of the tile at k0 that hold keys (first key < kend), and
// those wholly below kend.
__device__ __forceinline__ int groups_used(int k0, int kend) {
    const int n = (kend - k0 + kGroup - 1) / kGroup;
    return n < 0 ? 0 : (n > kGroups ? kGroups : n);
}
__device__ __forceinline__ int groups_full(int k0, int kend) {
    const int n = (kend - k0) / kGroup;
    return n < 0 ? 0 : (n > kGroups ? kGroups : n);
}

// A unit of work is one grid cell: KV head x, pair slot y of the sequence of
// rank z. A CTA starts with its own cell and then takes over cells whose CTAs
// have not been launched yet (cluster launch control), so the persistent CTAs
// walk the grid in its launch order. The descriptors of the current and the
// next unit sit in a two-entry ring in shared memory.
struct UnitDesc {
    int valid;      // 0: no unit (the end of this CTA's walk)
    int kvh, y, s;  // KV head, pair slot, sequence
    int q0, n, L;   // first query row, query rows, context length
    int np;         // query-tile pairs of the sequence's chunk
};
static_assert(sizeof(UnitDesc) == 32, "unit descriptor");

// Work item: a pair of query tiles (2 x 128 / G tokens) of one (sequence, KV
// head). Every role walks the same items and computes the same bounds.
struct Item {
    int tok0;       // first token of tile A
    int kend;       // keys the pair reads: L - n + (its last token) + 1
    int nt;         // K/V tiles (the more of the two query tiles' counts)
    int nta, ntb;   // key tiles query tile A, B reads (B: 0 when the chunk ends in A)
};

// Pair index of the i-th item of CTA b of the g CTAs of a (sequence, KV
// head), or -1 past the last: the np pairs, heaviest first (the last rows of
// the chunk see the most keys), are dealt in boustrophedon order b, 2g-1-b,
// 2g+b, ... so that each CTA's pairs add up to about the same work. Over b in
// [0, g) the positions cover [0, np) once each, whatever g is.
__device__ __forceinline__ int pair_of(int i, int b, int g, int np) {
    const int pos = 2 * g * (i >> 1) + ((i & 1) ? 2 * g - 1 - b : b);
    return pos < np ? np - 1 - pos : -1;
}

template <int G>
__device__ __forceinline__ Item make_item(int qp, int n, int L) {
    constexpr int BT = kRows / G;
    Item it;
    it.tok0 = qp * 2 * BT;
    const int last_tok = (it.tok0 + 2 * BT < n ? it.tok0 + 2 * BT : n) - 1;
    int kend = L - n + last_tok + 1;
    it.kend = kend < 0 ? 0 : (kend > L ? L : kend);
    it.nt = (it.kend + kKeys - 1) / kKeys;
    // tile A's own last token may need one key tile fewer; tile B holds tokens
    // only if the chunk reaches past tile A
    const int last_a = (it.tok0 + BT < n ? it.tok0 + BT : n) - 1;
    int kend_a = L - n + last_a + 1;
    kend_a = kend_a < 0 ? 0 : (kend_a > L ? L : kend_a);
    it.nta = (kend_a + kKeys - 1) / kKeys;
    it.ntb = it.tok0 + BT < n ? it.nt : 0;
    return it;
}

// The unit of grid cell (x, y, z), from the staged sequence tables (or from
// global memory beyond kRankMaxSeqs sequences, where z is the sequence).
template <int G>
__device__ __forceinline__ UnitDesc decode_unit(const PrefillArgs &a, const uint8_t *smem, int x,
                                                int y, int z, int64_t max_len) {
    constexpr int BT = kRows / G;
    UnitDesc u;
    int q0, q1, L;
    if (a.num_seqs <= kRankMaxSeqs) {
        const int *lens = reinterpret_cast<const int *>(smem + kOffSeqLens);
        const int *starts = reinterpret_cast<const int *>(smem + kOffSeqStarts);
        const uint16_t *rank_seq = reinterpret_cast<const uint16_t *>(smem + kOffRankSeq);
        u.s = rank_seq[z];
        q0 = starts[u.s];
        q1 = starts[u.s + 1];
        L = lens[u.s];
    } else {
        u.s = z;
        q0 = __ldg(a.query_start_loc + z);
        q1 = __ldg(a.query_start_loc + z + 1);
        const int64_t l = __ldg(a.context_lens + z);
        L = (int)(l < 0 ? 0 : (l > max_len ? max_len : l));
    }
    q0 = q0 < 0 ? 0 : (q0 > a.total_q ? a.total_q : q0);
    q1 = q1 < q0 ? q0 : (q1 > a.total_q ? a.total_q : q1);
    u.kvh = x;
    u.y = y;
    u.q0 = q0;
    u.n = q1 - q0;
    u.L = L;
    u.np = (u.n + 2 * BT - 1) / (2 * BT);
    u.valid = pair_of(0, y, gridDim.y, u.np) >= 0 ? 1 : 0;
    return u;
}

// Cluster launch control: ask to take over a CTA of this grid that has not
// been launched yet. The 16-byte response lands at `resp` and completes a
// phase of `bar` (the caller has armed it for 16 bytes).
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
        "[%0], [%1];\n" ::"r"(resp),
        "r"(bar)
        : "memory");
}
// Decode a response: true and the taken CTA's index when a CTA was taken.
__device__ __forceinline__ bool clc_taken(uint32_t resp, int &x, int &y, int &z) {
    uint32_t ok, cx = 0, cy = 0, cz = 0;
    asm volatile(
        "{\n .reg .b128 h;\n .reg .pred p;\n ld.shared.b128 h, [%4];\n"
        " clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, h;\n"
        " selp.u32 %0, 1, 0, p;\n"
        " @p clusterlaunchcontrol.query_cancel.get_first_ctaid.v4.b32.b128 {%1, %2, %3, _}, h;\n}\n"
        : "=r"(ok), "+r"(cx), "+r"(cy), "+r"(cz)
        : "r"(resp)
        : "memory");
    x = (int)cx;
    y = (int)cy;
    z = (int)cz;
    return ok != 0;
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_q) {
    constexpr int BT = kRows / G;               // query tokens per query tile
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int g = a.group;
    const int64_t max_len = (int64_t)a.max_blocks_per_seq << a.block_size_log2;

    // Grid (KV head x, pair slot y, sequence rank z). The block scheduler
    // starts CTAs in grid order (x fastest, z slowest), so with few enough
    // sequences slice z takes the one of rank z by context length (longest
    // first, ties by index), every KV head of its heaviest pair first: the
    // longest work of the whole launch starts first and the last wave holds
    // the shortest. Every CTA ranks the same staged lengths. A CTA that runs
    // out of work takes over the next CTA not launched yet, so the grid order
    // is also the order in which the persistent CTAs walk the cells.
    if (a.num_seqs <= kRankMaxSeqs) {
        int *lens = reinterpret_cast<int *>(smem + kOffSeqLens);
        int *starts = reinterpret_cast<int *>(smem + kOffSeqStarts);
        uint16_t *rank_seq = reinterpret_cast<uint16_t *>(smem + kOffRankSeq);
        if (tid < a.num_seqs) {
            const int64_t l = __ldg(a.context_lens + tid);
            lens[tid] = (int)(l < 0 ? 0 : (l > max_len ? max_len : l));
        }
        if (tid <= a.num_seqs) starts[tid] = __ldg(a.query_start_loc + tid);
        __syncthreads();
        if (tid < a.num_seqs) {
            const int lj = lens[tid];
            int rank = 0;
            for (int i = 0; i < a.num_seqs; ++i) {
                const int li = lens[i];
                rank += (li > lj || (li == lj && i < tid)) ? 1 : 0;
            }
            rank_seq[rank] = (uint16_t)tid;
        }
        __syncthreads();
    }
    UnitDesc *units = reinterpret_cast<UnitDesc *>(smem + kOffUnits);
    {
        const UnitDesc u0 = decode_unit<G>(a, smem, blockIdx.x, blockIdx.y, blockIdx.z, max_len);
        if (!u0.valid) return;                  // this cell holds no pair
        if (tid == 0) units[0] = u0;
    }

    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {                        // the swizzle atoms need 1024-byte alignment
        if (tid == 0) set_error(kErrSmemAlign);
        return;
    }

    const uint32_t ctl = sbase + kOffCtl;
    auto bar = [&](uint32_t i) { return ctl + 8 * i; };
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kOffAbort);
    if (tid == 0) {
        tc::mbar_init(bar(kBarQFull), 1);
        tc::mbar_init(bar(kBarQEmpty), 1);
        for (int i = 0; i < kKStages; ++i) {
            tc::mbar_init(bar(kBarKFull + i), 1);
            tc::mbar_init(bar(kBarKEmpty + i), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            tc::mbar_init(bar(kBarVFull + i), 1);
            tc::mbar_init(bar(kBarVEmpty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(kBarSFull + i), 1);
            tc::mbar_init(bar(kBarPReady + i), kRows / 32);
            tc::mbar_init(bar(kBarPVDone + i), 1);
            tc::mbar_init(bar(kBarOFree + i), kRows / 32);
            tc::mbar_init(bar(kBarUnitFull + i), 1);
            tc::mbar_init(bar(kBarUnitEmpty + i), kUnitReaders);
        }
        tc::mbar_init(bar(kBarClc), 1);
        *abort = 0;
        tc::fence_mbar_init();
        mbar_arrive(bar(kBarUnitFull));         // unit 0 (this CTA's own cell) is published
    }
    if (warp == kMmaWarp) tc::tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kOffTmemSlot);

    if (tid < kSoftmaxThreads) {
        // ---------------- softmax warpgroups ----------------
        const int wg = tid >> 7, r = tid & 127;
        const uint32_t lane = (uint32_t)(r & ~31) << 16;
        const uint32_t tS = tmem + lane + wg * 256, tO = tS + 128;
        const float sc = a.scale_log2;
        // a masked score for the max: the value that loses whatever the
        // scale's sign (masked keys then get p = 0 directly)
        const float masked = sc >= 0.f ? -INFINITY : INFINITY;
        uint32_t gt = 0;                        // this query tile's key tiles before this item
        bool ok = true;
#pragma unroll 1
        for (int k = 0; ok; ++k) {
        // unit k of this CTA's walk; its fields are read from shared memory
        // where they are used, so none stays live across the tile loop
        const volatile UnitDesc &u = units[k & 1];
        if (!warp_wait(bar(kBarUnitFull + (k & 1)), (k >> 1) & 1, abort)) { ok = false; break; }
        if (!u.valid) break;
#pragma unroll 1
        for (int i = 0; ok; ++i) {
            const int n = u.n, L = u.L;
            const int qp = pair_of(i, u.y, gridDim.y, u.np);
            if (qp < 0) break;
            const Item it = make_item<G>(qp, n, L);
            const int tok = it.tok0 + wg * BT + r / G, head = r % G;
            const bool rv = tok < n && head < g;
            int lim = 0;
            if (rv) {
                const int l = L - n + tok + 1;
                lim = l < 0 ? 0 : (l > L ? L : l);
            }
            const int ntt = wg == 0 ? it.nta : it.ntb;  // key tiles this query tile reads
            float m = -INFINITY, lsum = 0.f;
#pragma unroll 1
            for (int j = 0; j < ntt; ++j) {
                const uint32_t gj = gt + j;
                // S_t(j) done: also PV_t(j - 1) (issued before it), so O is stable
                if (!warp_wait(bar(kBarSFull + wg), gj & 1, abort, true)) { ok = false; break; }
                tc::fence_after_sync();
                const int kb = j * kKeys;
                const bool need_mask = kb + kKeys > lim;
                // the row's 128 scores in registers (one TMEM round trip);
                // the tile's extreme raw score (the max, or the min for a
                // negative scale), four independent running values
                uint32_t sr[4][32];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) tc::tmem_ld32(tS + ch * 32, sr[ch]);
                tc::tmem_ld_wait();
                if (need_mask) {
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        const int nv = lim - (kb + ch * 32);        // valid keys in the chunk
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (c >= nv) sr[ch][c] = __float_as_uint(masked);
                    }
                }
                float e4[4] = {masked, masked, masked, masked};
                if (sc >= 0.f) {
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            e4[0] = fmax3(e4[0], __uint_as_float(sr[ch][c]), __uint_as_float(sr[ch][c + 1]));
                            e4[1] = fmax3(e4[1], __uint_as_float(sr[ch][c + 2]), __uint_as_float(sr[ch][c + 3]));
                            e4[2] = fmax3(e4[2], __uint_as_float(sr[ch][c + 4]), __uint_as_float(sr[ch][c + 5]));
                            e4[3] = fmax3(e4[3], __uint_as_float(sr[ch][c + 6]), __uint_as_float(sr[ch][c + 7]));
                        }
                } else {
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            e4[0] = fmin3(e4[0], __uint_as_float(sr[ch][c]), __uint_as_float(sr[ch][c + 1]));
                            e4[1] = fmin3(e4[1], __uint_as_float(sr[ch][c + 2]), __uint_as_float(sr[ch][c + 3]));
                            e4[2] = fmin3(e4[2], __uint_as_float(sr[ch][c + 4]), __uint_as_float(sr[ch][c + 5]));
                            e4[3] = fmin3(e4[3], __uint_as_float(sr[ch][c + 6]), __uint_as_float(sr[ch][c + 7]));
                        }
                }
                const float ext = sc >= 0.f ? fmax3(fmaxf(e4[0], e4[1]), e4[2], e4[3])
                                            : fmin3(fminf(e4[0], e4[1]), e4[2], e4[3]);
                // every score of the row masked: no new max (also for scale 0)
                const float mt = ext == masked ? -INFINITY : ext * sc;
                bool rescale = false;
                float alpha = 1.f;
                if (mt > m + kRescaleSlack) {
                    rescale = m != -INFINITY;
                    alpha = rescale ? ex2(m - mt) : 1.f;
                    lsum *= alpha;
                    m = mt;
                }
                const float mb = m == -INFINITY ? 0.f : m;
                // P = 2^(S sc - m) in bf16 over the first 64 columns (all of S
                // is in registers already); masked keys get p = 0
                float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t pw[16];
                    const int nv = need_mask ? lim - (kb + ch * 32) : 32;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        float p0 = ex2(fmaf(__uint_as_float(sr[ch][2 * c]), sc, -mb));
                        float p1 = ex2(fmaf(__uint_as_float(sr[ch][2 * c + 1]), sc, -mb));
                        if (need_mask) {
                            p0 = 2 * c < nv ? p0 : 0.f;
                            p1 = 2 * c + 1 < nv ? p1 : 0.f;
                        }
                        l4[c & 3] += p0 + p1;
                        pw[c] = pack_bf16x2(p0, p1);
                    }
                    tc::tmem_st16(tS + ch * 16, pw);
                }
                lsum += (l4[0] + l4[1]) + (l4[2] + l4[3]);
                // rescale this warp's rows of O if any of them raised its max
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t o[32];
                        tc::tmem_ld32(tO + ch * 32, o);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tc::tmem_st32(tO + ch * 32, o);
                    }
                }
                tc::tmem_st_wait();
                tc::fence_before_sync();
                warp_arrive(bar(kBarPReady + wg));
            }
            if (!ok) break;
            // epilogue: O / l -> bf16 rows; then O is free for the next item
            if (ntt > 0) {
                if (!warp_wait(bar(kBarPVDone + wg), (gt + ntt - 1) & 1, abort, true)) { ok = false; break; }
                tc::fence_after_sync();
            }
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            const int64_t row_elem = ((int64_t)u.q0 + tok) * a.num_q_heads + (int64_t)u.kvh * g + head;
            uint4 *orow = reinterpret_cast<uint4 *>(static_cast<char *>(a.out) + row_elem * kRowBytes);
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t o[32];
                if (ntt > 0) {
                    tc::tmem_ld32(tO + ch * 32, o);
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
            tc::fence_before_sync();
            warp_arrive(bar(kBarOFree + wg));
            gt += ntt;
        }
        if (ok) warp_arrive(bar(kBarUnitEmpty + (k & 1)));
        }
    } else if (warp == kKWarp || warp == kVWarp) {
        // ---------------- K and V producers ----------------
        // Per key tile, lane i < 16 loads the box of 16-key group i / 2, half
        // i % 2 by TMA; a box at row -kGroup reads zeros (a bad block id reads
        // as zeros the same way). The block ids of the next tile are read
        // while this one is issued. The V group holding the end of the keys
        // is copied by the warp with the rows past the end zeroed.
        const bool is_v = warp == kVWarp;
        const int nst = is_v ? kVStages : kKStages;
        const int lane = tid & 31;
        const int q = lane >> 1, h = lane & 1;
        const void *map = is_v ? static_cast<const void *>(&tmap_v) : static_cast<const void *>(&tmap_k);
        const uint32_t bar_full = bar(is_v ? kBarVFull : kBarKFull);
        const uint32_t bar_empty = bar(is_v ? kBarVEmpty : kBarKEmpty);
        const uint32_t base = sbase + (is_v ? kOffV : kOffK);
        uint32_t gt = 0;
        uint32_t clc_n = 0;                     // launch-control requests made (K warp)
        int qitem = 0;                          // items whose Q the V warp has loaded
        bool clc_done = false;                  // a request found no CTA left to take
        bool ok = true;
#pragma unroll 1
        for (int k = 0; ok; ++k) {
        if (!warp_wait(bar(kBarUnitFull + (k & 1)), (k >> 1) & 1, abort)) { ok = false; break; }
        const UnitDesc u = units[k & 1];
        if (!u.valid) break;
        const int s = u.s, kvh = u.kvh, n = u.n, L = u.L, q0 = u.q0;
#pragma unroll 1
        for (int i = 0; ok; ++i) {
            const int qp = pair_of(i, u.y, gridDim.y, u.np);
            if (qp < 0) break;
            const Item it = make_item<G>(qp, n, L);
            const int kend = it.kend;
            if (is_v) {
                // the V producer also loads each item's Q tiles, once the
                // previous item's MMAs are done with the Q buffers
                if (qitem > 0 && !warp_wait(bar(kBarQEmpty), (qitem - 1) & 1, abort)) { ok = false; break; }
                if (lane == 0) {
                    tc::mbar_expect_tx(bar(kBarQFull), 2 * kQBytes);
                    for (int t = 0; t < 2; ++t)
                        for (int hh = 0; hh < 2; ++hh)
                            tc::tma_load_3d(sbase + kOffQ + t * kQBytes + hh * kQHalf, &tmap_q, hh * 64,
                                            kvh * g, q0 + it.tok0 + t * BT, bar(kBarQFull));
                }
                warp_arrive(bar(kBarQFull));
                ++qitem;
            }
            // TMA coordinates (dim 1, dim 2) of this lane's box of tile j:
            // token-major (KV head, slot), head-major (offset in the block,
            // block * Hkv + KV head); dim 1 at -kGroup reads zeros (a bad block
            // id reads as zeros that way); x = INT_MIN: no box
            auto box_at = [&](int j) -> int2 {
                const int k0 = j * kKeys;
                const int ng = is_v ? groups_full(k0, kend) : groups_used(k0, kend);
                if (lane >= 2 * kGroups || j >= it.nt || q >= ng) return make_int2(INT_MIN, 0);
                const int64_t slot = key_row(a, s, k0 + q * kGroup);
                if (slot < 0) return a.head_major ? make_int2(-kGroup, 0) : make_int2(kvh, -kGroup);
                if (!a.head_major) return make_int2(kvh, (int)slot);
                const int lb = a.block_size_log2;
                return make_int2((int)(slot & ((1 << lb) - 1)), (int)((slot >> lb) * a.num_kv_heads + kvh));
            };
            int2 box_next = box_at(0);
#pragma unroll 1
            for (int j = 0; j < it.nt; ++j) {
                const int2 box = box_next;
                box_next = box_at(j + 1);
                const uint32_t gj = gt + j;
                const int st = gj % nst;
                if (!warp_wait(bar_empty + 8 * st, ((gj / nst) & 1) ^ 1, abort)) { ok = false; break; }
                const uint32_t dst = base + st * kKVBytes;
                const uint32_t full = bar_full + 8 * st;
                const int k0 = j * kKeys;
                const int nk = groups_used(k0, kend), nf = groups_full(k0, kend);
                if (lane == 0) tc::mbar_expect_tx(full, (uint32_t)(is_v ? nf : nk) * 2 * kGroup * 128);
                __syncwarp();
                if (box.x != INT_MIN)
                    tc::tma_load_3d(dst + h * kKVHalf + q * kGroup * 128, map, h * 64, box.x, box.y, full);
                if (is_v && nk > nf) {
                    copy_v_tail(a, s, kvh, k0 + nf * kGroup, kend, dst, lane);
                    tc::fence_proxy_async();
                }
                // (test hook: the first tile's V arrival held back, see
                // set_prefill_fault)
                if (!(is_v && a.fault_hold_v && gj == 0)) warp_arrive(full);
            }
            gt += it.nt;
        }
        if (!ok) break;
        warp_arrive(bar(kBarUnitEmpty + (k & 1)));
        if (is_v) continue;
        // The K warp publishes unit k + 1 once it has issued unit k's last K
        // tile: it takes over the next CTA of the grid not launched yet
        // (cells with no pair are taken and skipped). Once a request finds no
        // CTA left, no further request is made and the published unit marks
        // the end of the walk.
        UnitDesc nx{};
        nx.valid = 0;
        while (!clc_done) {
            // every lane has read the previous response; the next one is
            // written through the async proxy
            __syncwarp();
            tc::fence_proxy_async();
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(kBarClc), 16);
                clc_try_cancel(sbase + kOffClcResp, bar(kBarClc));
            }
            if (!warp_wait(bar(kBarClc), clc_n & 1, abort)) { ok = false; break; }
            ++clc_n;
            int cx, cy, cz;
            if (!clc_taken(sbase + kOffClcResp, cx, cy, cz)) {
                clc_done = true;
                break;
            }
            nx = decode_unit<G>(a, smem, cx, cy, cz, max_len);
            if (nx.valid) break;
        }
        if (!ok) break;
        // its ring slot held unit k - 1, which every warp has finished
        if (k >= 1 && !warp_wait(bar(kBarUnitEmpty + ((k + 1) & 1)), ((k - 1) >> 1) & 1, abort)) {
            ok = false;
            break;
        }
        if (lane == 0) units[(k + 1) & 1] = nx;
        warp_arrive(bar(kBarUnitFull + ((k + 1) & 1)));
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue ----------------
        // The whole warp runs the issue loop, converged, so that barrier
        // tests and descriptors are warp-uniform; one elected lane executes
        // each tcgen05.mma / commit. Descriptor high word (stride offset
        // 1024 B, version, 128-byte swizzle) is common; the low word is
        // (address >> 4) | leading offset.
        const uint64_t dq = tc::sw128_desc(sbase + kOffQ, 16, 1024);        // K-major (LBO unused)
        const uint64_t dk = tc::sw128_desc(sbase + kOffK, 16, 1024);
        const uint64_t dv = tc::sw128_desc(sbase + kOffV, kKVHalf, 1024);   // MN-major: next 64 dims
        const uint32_t hi = (uint32_t)(dq >> 32);                           // same for all three
        const uint32_t q_lo = (uint32_t)dq, k_lo = (uint32_t)dk, v_lo = (uint32_t)dv;
        auto desc = [hi](uint32_t lo) { return ((uint64_t)hi << 32) | lo; };
        // S_t = Q_t K^T from K stage st. The elected lane issues; the other
        // lanes go on to the next barrier test, whose warp-wide vote waits
        // for it (a __syncwarp after each batch measured 0.4-1.3 % slower).
        auto issue_s = [&](int t, int st, uint32_t release) {
            const uint32_t qd = q_lo + t * (kQBytes >> 4);
            const uint32_t kd = k_lo + st * (kKVBytes >> 4);
            const uint32_t d = tmem + t * 256;
            tc::fence_after_sync();
            if (tc::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk)
                    tc::mma_ss(d, desc(qd + (((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4)),
                               desc(kd + (((kk >> 2) * kKVHalf + (kk & 3) * 32) >> 4)), kIdescS, kk > 0);
                tc::commit(bar(kBarSFull + t));
                if (release) tc::commit(release);
            }
        };
        // O_t += P_t V over the first nv 16-key groups of V stage st (P_t in
        // TMEM, 8 columns per 16 keys; the groups past the end of the keys
        // have P = 0 and no V)
        auto issue_pv = [&](int t, int st, bool acc, int nv, uint32_t release) {
            const uint32_t vd = v_lo + st * (kKVBytes >> 4);
            const uint32_t pa_ = tmem + t * 256;
            const uint32_t d = pa_ + 128;
            tc::fence_after_sync();
            if (tc::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kGroups; ++kk)
                    if (kk < nv)
                        tc::mma_ts(d, pa_ + kk * 8, desc(vd + ((kk * 2048) >> 4)), kIdescPV, acc || kk > 0);
                tc::commit(bar(kBarPVDone + t));
                if (release) tc::commit(release);
            }
        };
        // every lane tests the barrier (one shared-memory access for the
        // warp, no divergent branch) and a vote gives the warp one answer: a
        // completed phase stays completed until this warp issues the work
        // that lets the next one complete, so any lane's yes is the answer;
        // __syncwarp then orders the lanes that saw it before the others
        auto ready = [](uint32_t b, uint32_t parity) {
            const bool r = __any_sync(0xffffffffu, tc::mbar_test_wait(b, parity));
            if (r) __syncwarp();
            return r;
        };
        // Event-driven issue for each query tile t: S_t(x) once K_x has
        // landed and PV_t(x - 1) has been issued; PV_t(y) once P_t(y) is in
        // TMEM and V_y has landed (and, for the first PV of an item, the
        // previous item's O has been read), each tile up to its own count of
        // key tiles. A K stage is released after the last S that reads it
        // (the second, or the only one when the other tile stops short), a V
        // stage after the last PV.
        uint32_t gt = 0;                        // the pair's key tiles before this item (K/V stages)
        uint32_t gq0 = 0, gq1 = 0;              // each query tile's key tiles before this item
        int item = 0;
        bool ok = true;
#pragma unroll 1
        for (int k = 0; ok; ++k) {
        if (!warp_wait(bar(kBarUnitFull + (k & 1)), (k >> 1) & 1, abort)) { ok = false; break; }
        const volatile UnitDesc &u = units[k & 1];
        if (!u.valid) break;
#pragma unroll 1
        for (int i = 0; ok; ++i, ++item) {
            const int qp = pair_of(i, u.y, gridDim.y, u.np);
            if (qp < 0) break;
            const Item it = make_item<G>(qp, u.n, u.L);
            ok = warp_wait(bar(kBarQFull), item & 1, abort);
            int sj0 = 0, sj1 = 0, pj0 = 0, pj1 = 0;     // next S / PV tile of A, B
            uint64_t t_idle = 0;
            uint32_t idle = 0;
#pragma unroll 1
            while (ok && (pj0 < it.nta || pj1 < it.ntb)) {
                bool progress = false;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    int &sj = t == 0 ? sj0 : sj1;
                    int &pj = t == 0 ? pj0 : pj1;
                    const int other_pj = t == 0 ? pj1 : pj0;
                    const int other_sj = t == 0 ? sj1 : sj0;
                    const int my_nt = t == 0 ? it.nta : it.ntb;
                    const int other_nt = t == 0 ? it.ntb : it.nta;
                    const uint32_t my_gq = t == 0 ? gq0 : gq1;
                    if (pj < sj) {
                        const uint32_t gp = gt + pj;
                        const int st = gp % kVStages;
                        bool go = ready(bar(kBarPReady + t), (my_gq + pj) & 1) &&
                                  ready(bar(kBarVFull + st), (gp / kVStages) & 1);
                        if (go && pj == 0 && item > 0) go = ready(bar(kBarOFree + t), (item - 1) & 1);
                        if (go) {
                            // the V stage is released by its last reader
                            issue_pv(t, st, pj > 0, groups_used(pj * kKeys, it.kend),
                                     other_pj > pj || other_nt <= pj ? bar(kBarVEmpty + st) : 0u);
                            ++pj;
                            progress = true;
                        }
                    }
                    if (sj == pj && sj < my_nt) {
                        const uint32_t gs = gt + sj;
                        const int st = gs % kKStages;
                        if (ready(bar(kBarKFull + st), (gs / kKStages) & 1)) {
                            issue_s(t, st, other_sj > sj || other_nt <= sj ? bar(kBarKEmpty + st) : 0u);
                            ++sj;
                            progress = true;
                        }
                    }
                }
                if (progress) {
                    idle = 0;
                    continue;
                }
                // nothing ready: poll again (no back-off: a sleeping issuer
                // reacts late to the next hand-off); the 2 s limit is
                // checked every 256 rounds
                if (++idle == 1) {
                    t_idle = tc::globaltimer_ns();
                } else if ((idle & 255) == 0) {
                    const bool stop = __shfl_sync(0xffffffffu,
                                                  (*abort || tc::globaltimer_ns() - t_idle > 2000000000ull) ? 1 : 0, 0) != 0;
                    if (stop) {
                        if ((threadIdx.x & 31) == 0 && !*abort) {
                            set_error(kErrTimeout);
                            *abort = 1;
                        }
                        ok = false;
                    }
                }
            }
            // Q buffers free once this item's MMAs are done
            if (tc::elect_one()) tc::commit(bar(kBarQEmpty));
            __syncwarp();
            gt += it.nt;
            gq0 += it.nta;
            gq1 += it.ntb;
        }
        if (ok) warp_arrive(bar(kBarUnitEmpty + (k & 1)));
        }
    }

    // teardown: every role is done (or has given up); TMEM is freed
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// q [total_q, Hq, 128] bf16 as a 3-D tensor (128, Hq, total_q) with boxes of
// 64 dims x G heads x 128 / G tokens, 128-byte swizzle: one box is one half
// (64 dims) of a 128-row query tile.
bool make_q_map(CUtensorMap *m, const void *q, int total_q, int num_q_heads, int G) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    const cuuint64_t strides[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)num_q_heads * kRowBytes};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(kRows / G)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G>
cudaError_t launch_g(const PrefillArgs &a, int max_query_len, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    // TMA coordinates are int32
    if ((a.num_blocks << a.block_size_log2) >= (int64_t)1 << 31 ||
        a.num_blocks * a.num_kv_heads >= (int64_t)1 << 31)
        return cudaErrorInvalidValue;
    const int bs = 1 << a.block_size_log2;
    CUtensorMap mk, mv, mq;
    if (!make_pool_map(&mk, a.k_cache, a.num_blocks, bs, a.num_kv_heads, a.head_major != 0) ||
        !make_pool_map(&mv, a.v_cache, a.num_blocks, bs, a.num_kv_heads, a.head_major != 0) ||
        !make_q_map(&mq, a.q, a.total_q, a.num_q_heads, G))
        return cudaErrorInvalidValue;
    constexpr int BT = kRows / G;
    const int pairs = (max_query_len + 2 * BT - 1) / (2 * BT);
    int gy = (pairs + kPairsPerCta - 1) / kPairsPerCta;   // pair slots per (sequence, KV head)
    gy = gy < 1 ? 1 : (gy > 65535 ? 65535 : gy);
    prefill_tc_kernel<G><<<dim3(a.num_kv_heads, gy, a.num_seqs), kThreads, kSmemBytes, st>>>(a, mk, mv, mq);
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

namespace {
std::atomic<int> g_fault_mode{0};
}  // namespace

void set_prefill_fault(int mode) { g_fault_mode.store(mode); }
int prefill_fault() { return g_fault_mode.load(); }

cudaError_t take_prefill_error(cudaStream_t stream, int *code) {
    return take_device_word(g_prefill_error, stream, code);
}

}  // namespace pa

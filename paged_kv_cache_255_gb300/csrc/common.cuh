// Device helpers shared by the libpagedattn kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pa {

constexpr int kHeadDim = 128;                    // the only head size supported
constexpr int kTileTokens = 16;                  // tokens per KV tile
constexpr int kRowBytes = kHeadDim * 2;          // one bf16 K (or V) row: 256 B
constexpr int kTileBytes = kTileTokens * kRowBytes;  // 4 KB

// Device-side error codes. Each kernel file keeps a __device__ int word that
// a kernel sets (first code wins) when it meets one of these and carries on
// in the defined way; pa_take_device_error reads and clears the words.
enum DeviceError : int {
    kErrNone = 0,
    kErrSmemAlign = 1,   // prefill: dynamic shared memory not 1024-byte aligned; CTA skipped
    kErrTimeout = 2,     // prefill or decode: a bounded mbarrier wait ran out; the launch gave up
    kErrBadSlot = 3,     // store: a slot outside [-1, num_blocks * block_size) was skipped
    kErrBadBlock = 4,    // decode / prefill: a block id outside [0, num_blocks) read as zeros
};

// Read the __device__ int `word` (of the calling file) on `stream`, wait for
// it, store it in *code and clear it if it was set.
template <typename Word>
inline cudaError_t take_device_word(Word &word, cudaStream_t stream, int *code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, word, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    *code = v;
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(word, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    return e;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global->shared copy; src_bytes == 0 reads nothing and
// zero-fills the 16 bytes.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// 2^x on the SFU (PTX ex2.approx; flushes denormal results to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// Two bf16 packed in a 32-bit word -> two floats (bf16 is the top half of an
// fp32, so widening is exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// float -> bf16 bits, round to nearest even (via the cvt instruction).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ldmatrix: four 8x8 b16 matrices from shared memory; lane i supplies the
// address of row (i % 8) of matrix (i / 8). Lane l receives, of matrix j,
// row l / 4, columns 2 (l % 4) and 2 (l % 4) + 1 (transposed with .trans).
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D = A B + D, A 16x16 bf16 (row), B 16x8 bf16 (col), D 16x8 fp32.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose an 8x8 b16 matrix held one row-pair per lane (ldmatrix layout).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

}  // namespace pa

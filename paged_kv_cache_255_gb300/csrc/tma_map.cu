// TMA tensor maps over the paged K/V pool, shared by the decode and prefill
// kernels: both fetch a tile of 16 tokens of one KV head as two boxes of 64
// head dims, which land in shared memory as 16 rows of 128 bytes in the
// 128-byte swizzled layout (16-byte chunk c of row r at chunk position
// c ^ (r % 8), given a 1024-byte aligned destination).
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace pa {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Token-major [NB, bs, Hkv, 128] is the 3-D tensor (128, Hkv, NB * bs) with
// box (64, 1, 16); head-major [NB, Hkv, bs, 128] is (128, bs, NB * Hkv) with
// box (64, 16, 1). Coordinates are int32, so the row count must stay below
// 2^31 (checked by the callers).
bool make_pool_map(CUtensorMap *m, const void *pool, int64_t num_blocks, int block_size,
                   int num_kv_heads, bool head_major) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t d1 = head_major ? block_size : num_kv_heads;
    const cuuint64_t d2 = head_major ? num_blocks * num_kv_heads : num_blocks * block_size;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, d1, d2};
    const cuuint64_t strides[2] = {(cuuint64_t)kRowBytes, d1 * kRowBytes};
    const cuuint32_t box[3] = {64, head_major ? (cuuint32_t)kTileTokens : 1u,
                               head_major ? 1u : (cuuint32_t)kTileTokens};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pa

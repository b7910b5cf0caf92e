// TMA tensor maps over the paged K/V pool. Both kernels fetch tiles of 16
// tokens of one KV head that land in shared memory as two halves (head dims
// 0-63, then 64-127) of 16 rows of 128 bytes in the 128-byte swizzled layout
// (16-byte chunk c of row r at chunk position c ^ (r % 8), given a 1024-byte
// aligned destination): the prefill as two boxes per tile (make_pool_map),
// the decode as one (make_tile_map).
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

// The decode's map: one box is a whole 16-token tile of one KV head, landing
// as the same two 16 x 128-byte halves (dims 0-63, then 64-127) that two boxes
// of make_pool_map's map would give, for half the TMA instructions. Its
// dimensions are (64 head dims, token row, half, KV head) for token-major and
// (64 head dims, offset in the block, half, block * Hkv + KV head) for
// head-major; the half's 128-byte stride comes after the row's. Coordinates:
// token-major (0, block * bs + offset, 0, KV head); head-major (0, offset, 0,
// block * Hkv + KV head).
bool make_tile_map(CUtensorMap *m, const void *pool, int64_t num_blocks, int block_size,
                   int num_kv_heads, bool head_major) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t rows = head_major ? (cuuint64_t)block_size : (cuuint64_t)(num_blocks * block_size);
    const cuuint64_t outer = head_major ? (cuuint64_t)(num_blocks * num_kv_heads) : (cuuint64_t)num_kv_heads;
    const cuuint64_t row_stride = head_major ? (cuuint64_t)kRowBytes : (cuuint64_t)num_kv_heads * kRowBytes;
    const cuuint64_t outer_stride = head_major ? (cuuint64_t)block_size * kRowBytes : (cuuint64_t)kRowBytes;
    const cuuint64_t dims[4] = {64, rows, 2, outer};
    const cuuint64_t strides[3] = {row_stride, 128, outer_stride};
    const cuuint32_t box[4] = {64, (cuuint32_t)kTileTokens, 2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pool), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pa

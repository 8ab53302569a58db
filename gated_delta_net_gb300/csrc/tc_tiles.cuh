// tc_tiles.cuh -- shared helpers of the tensor-core verify kernels: bf16 packing,
// the 128-byte-swizzled tile layout the TMA boxes and the MMA descriptors use,
// named barriers, and the token tensor maps.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.cuh"

namespace gdn {
namespace tiles {

constexpr int kD = 128;  // d_k = d_v of the tensor-core kernels

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Byte offset of element (row, k) in a tile of `rows` rows, 128-byte-swizzled bf16:
// column blocks of 64 elements (rows * 128 bytes apart), rows of 128 bytes, 16-byte
// chunks permuted by (row mod 8).  Used K-major (row = M/N index, k = K index)
// and, for the right-hand side, MN-major (row = K index, k = N index).
__device__ __forceinline__ uint32_t sw128_offset(int row, int k, int rows = 128) {
    return (uint32_t)((k >> 6) * rows * 128 + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2);
}

__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// [T][H][128] bf16 viewed as a 3-D tensor (d, head, token); boxes of 64 x 1 x 32,
// 128-byte swizzle.
inline bool encode_tokens(CUtensorMap *map, const void *base, int heads, int total) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)total};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2};
    cuuint32_t box[3] = {64, 1, 32};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace tiles
}  // namespace gdn

// Pieces shared by the two bf16 backward kernels (bwd.cu: dK/dV, bwd_dq.cu: dQ).
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace jfa {

// Stores n fp32 values (n a multiple of 8), each times `mul`, as bf16 to a 16-byte
// aligned global row.
__device__ __forceinline__ void store_bf16_row(__nv_bfloat16* dst, const float* v, int n, float mul) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < n / 8; ++i) {
        uint4 u;
        u.x = pack_bf16x2(v[8 * i + 0] * mul, v[8 * i + 1] * mul);
        u.y = pack_bf16x2(v[8 * i + 2] * mul, v[8 * i + 3] * mul);
        u.z = pack_bf16x2(v[8 * i + 4] * mul, v[8 * i + 5] * mul);
        u.w = pack_bf16x2(v[8 * i + 6] * mul, v[8 * i + 7] * mul);
        d4[i] = u;
    }
}

// Zero-fills n bf16 values (n a multiple of 8) of a 16-byte aligned global row.
__device__ __forceinline__ void zero_bf16_row(__nv_bfloat16* dst, int n) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < n / 8; ++i) d4[i] = make_uint4(0u, 0u, 0u, 0u);
}

// TMEM column, relative to a 128-column score tile, of the 16 bf16 operand values
// of K-step s (16 rows of the contraction) when the tile's compute threads have
// packed their values in place: warpgroup g owns columns [64g, 64g+64) and writes
// its 64 packed values to the first 32 of them.
__device__ __forceinline__ uint32_t packed_col(int s) { return uint32_t(64 * (s >> 2) + 8 * (s & 3)); }

}  // namespace jfa

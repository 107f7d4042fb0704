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

// Writes a warp's 32 x 32 fp32 chunk (lane = row, raw = the row's 32 values as bits),
// each times `mul`, as bf16 to 32 global rows of 64 bytes: row r at dst + r * stride
// (elements; 16-byte aligned), skipped unless bit r of valid is set.  Each lane stores its row's four 16-byte
// pieces in the warp's 2 KB staging buffer `stg` (piece q of row r at slot q ^ ((r >> 1) &
// 3), so that any eight consecutive rows cover all 32 banks), then every global store
// instruction writes eight whole 64-byte rows.  Stored straight from registers, each
// instruction would instead touch 32 rows, one 16-byte piece of each: four times the
// cache-line transactions.
__device__ __forceinline__ void store_chunk_bf16(uint32_t* stg, const uint32_t (&raw)[32], float mul, int lane,
                                                 uint32_t valid, __nv_bfloat16* dst, size_t stride) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16x2(__uint_as_float(raw[8 * q + 0]) * mul, __uint_as_float(raw[8 * q + 1]) * mul);
        u.y = pack_bf16x2(__uint_as_float(raw[8 * q + 2]) * mul, __uint_as_float(raw[8 * q + 3]) * mul);
        u.z = pack_bf16x2(__uint_as_float(raw[8 * q + 4]) * mul, __uint_as_float(raw[8 * q + 5]) * mul);
        u.w = pack_bf16x2(__uint_as_float(raw[8 * q + 6]) * mul, __uint_as_float(raw[8 * q + 7]) * mul);
        *reinterpret_cast<uint4*>(stg + lane * 16 + ((q ^ ((lane >> 1) & 3)) << 2)) = u;
    }
    __syncwarp();
    const int piece = lane & 3;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = (lane >> 2) + 8 * k;
        const uint4 u = *reinterpret_cast<const uint4*>(stg + r * 16 + ((piece ^ ((r >> 1) & 3)) << 2));
        if ((valid >> r) & 1u) *reinterpret_cast<uint4*>(dst + size_t(r) * stride + 8 * piece) = u;
    }
    __syncwarp();
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

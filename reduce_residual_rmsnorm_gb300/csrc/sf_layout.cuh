// Byte offset of NVFP4 scale factor (row m, 16-column block k) in the three
// `QuantizationSFLayout`s of tokenspeed trtllm.py.  The pages name the two
// swizzled layouts without defining them; the offsets below are the tile
// layouts the library documents in include/ts_fused_norm.h.
//
// Every layout splits into a row part and a column part
//   offset(m, k) = sf_row_base(m) + (k / 4) * sf_tile_stride() + k % 4
// with tile strides 4 (LINEAR: consecutive k), 32 (8-row x 4-column tiles)
// and 512 (128-row x 4-column tiles), so a kernel computes the row part once.
#pragma once

#include <cstdint>

#include "launch.h"

namespace tsfn {

__device__ __forceinline__ int sf_tile_stride(const FusedArgs &a)
{
    return a.sf_layout == kSfLinear ? 4 : (a.sf_layout == kSfSwizzled8x4 ? 32 : 512);
}

__device__ __forceinline__ int64_t sf_row_base(const FusedArgs &a, int64_t m)
{
    if (a.sf_layout == kSfLinear)
        return m * (a.H >> 4);
    const int64_t tiles_per_band = a.sf_cols >> 2;
    if (a.sf_layout == kSfSwizzled8x4)  // 32-byte tiles, row-major inside: row m%8 at byte 4*(m%8)
        return (m >> 3) * tiles_per_band * 32 + (m & 7) * 4;
    // 512-byte tiles; inside a tile row m%128 = 32*i + j sits at byte 16*j + 4*i
    return (m >> 7) * tiles_per_band * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4;
}

__device__ __forceinline__ int64_t sf_offset(const FusedArgs &a, int64_t m, int64_t k)
{
    return sf_row_base(a, m) + (k >> 2) * sf_tile_stride(a) + (k & 3);
}

}  // namespace tsfn

// Byte offset of NVFP4 scale factor (row m, 16-column block k) in the three
// `QuantizationSFLayout`s of tokenspeed trtllm.py.  The pages name the two
// swizzled layouts without defining them; the offsets below are the tile
// layouts the library documents in include/ts_fused_norm.h.
#pragma once

#include <cstdint>

#include "launch.h"

namespace tsfn {

__device__ __forceinline__ int64_t sf_offset(const FusedArgs &a, int64_t m, int64_t k)
{
    if (a.sf_layout == kSfLinear)
        return m * (a.H >> 4) + k;
    const int64_t tiles_per_band = a.sf_cols >> 2;
    if (a.sf_layout == kSfSwizzled8x4)  // 32-byte tiles of 8 rows x 4 columns, row-major inside
        return ((m >> 3) * tiles_per_band + (k >> 2)) * 32 + (m & 7) * 4 + (k & 3);
    // 512-byte tiles of 128 rows x 4 columns; inside a tile row m%128 = 32*i + j
    // sits at byte 16*j + 4*i
    return ((m >> 7) * tiles_per_band + (k >> 2)) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4 + (k & 3);
}

}  // namespace tsfn

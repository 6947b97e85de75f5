// Internal interface between the C ABI (api.cu: argument checks) and the
// kernel launchers.  Everything here has already been validated.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace tsfn {

constexpr int kMaxR = 16;

// Kinds of output epilogue; the pattern codes map onto them.
enum class Epilogue : int {
    kAllReduce = 0,  // pattern 0
    kNorm = 1,       // patterns 1, 8
    kFp8Tensor = 2,  // patterns 2, 4
    kFp4 = 3,        // patterns 3, 5
    kFp8Block = 4    // patterns 6, 7
};

struct FusedArgs {
    const uint16_t *partials[kMaxR];
    int R;
    const uint16_t *residual;
    const uint16_t *gamma;
    float eps;
    const float *scale_factor;  // device scalar (sigma or g), may be null
    int64_t T;
    int64_t H;
    uint16_t *allreduce_out;
    uint16_t *residual_out;
    uint16_t *norm_out;
    uint16_t *partial_norm_out;
    int64_t partial_cols;
    uint8_t *quant_out;
    void *scale_out;    // fp32 block scales or uint8 SFs
    int sf_swizzled;    // 1: SWIZZLED_128x4, 0: LINEAR
    int64_t sf_rows;    // rows of the SF buffer (T, or T padded to 128)
    int64_t sf_cols;    // H/16, padded to a multiple of 4 when swizzled
};

struct QKArgs {
    const uint16_t *shards[kMaxR];
    int R;
    int64_t T;
    int64_t row_stride;
    int Q;
    int K;
    const uint16_t *q_weight;
    const uint16_t *k_weight;
    float eps;
    uint16_t *q_out;
    int64_t ldq;
    uint16_t *k_out;
    int64_t ldk;
};

cudaError_t launch_fused(Epilogue ep, const FusedArgs &a, cudaStream_t stream);
cudaError_t launch_qk(const QKArgs &a, cudaStream_t stream);

}  // namespace tsfn

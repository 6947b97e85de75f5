// Internal interface between the C ABI (api.cu: argument checks) and the
// kernel launchers.  Everything here has already been validated.
#pragma once

#include <atomic>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "int_div.h"

namespace tsfn {

constexpr int kMaxR = 16;

// `QuantizationSFLayout` codes.
constexpr int kSfSwizzled128x4 = 0;
constexpr int kSfSwizzled8x4 = 1;
constexpr int kSfLinear = 2;

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
    const uint16_t *add_in;  // optional extra addend before the residual (reduce-scatter "Add")
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
    int sf_layout;      // kSfSwizzled128x4, kSfSwizzled8x4 or kSfLinear
    int64_t sf_rows;    // rows of the SF buffer (T, or T padded to 128 / 8)
    int64_t sf_cols;    // H/16, padded to a multiple of 4 when swizzled
    int64_t prefetch_rows;  // rows ahead whose inputs a CTA prefetches into L2 (0: none)
    int pdl_wait;           // where a PDL launch waits: 0 first, 1 after the first loads, 2 before exit
};

struct QKArgs {
    const uint16_t *shards[kMaxR];
    int R;
    DivMagic div_r;  // division by R (a warp's token and shard)
    int64_t T;
    int64_t row_stride;
    int Q;
    int K;
    // 1/Q, 1/K, 1/R where that count is a power of two (exact), else 0: the
    // kernel then multiplies instead of dividing, with the same rounded result
    float inv_q, inv_k, inv_r;
    const uint16_t *q_weight;
    const uint16_t *k_weight;
    float eps;
    uint16_t *q_out;
    int64_t ldq;
    uint16_t *k_out;
    int64_t ldk;
    int64_t prefetch_tokens;  // tokens ahead whose shard rows a warp prefetches into L2 (0: none)
};

struct AGArgs {
    const uint16_t *inputs[kMaxR];  // rank r's token slice [count_r, hidden]
    int R;
    int64_t T;                      // gathered tokens
    // the token split: ranks below `extra` hold base + 1 rows (gathered rows
    // below `split` = extra * (base + 1)), the others base rows
    uint32_t base, extra, split;
    DivMagic div_hi, div_lo;        // division by base + 1 and by base
    int hidden, q, kv;              // row = x (q) | y (kv) | rope
    const uint16_t *x_gamma;
    const uint16_t *y_gamma;
    float x_eps, y_eps;
    int pattern;                    // AllGatherFusionPattern 0..2
    uint16_t *allgather_out;        // [T, hidden]
    uint16_t *x_norm_out;           // [T, q] (optional in pattern 2)
    uint16_t *y_norm_out;           // [T, kv]
    uint8_t *quant_out;             // [T, q] e4m3 (pattern 2)
    float *scale_out;               // [T, q/128] (pattern 2)
};

// Launch `kernel` on `stream`, with programmatic stream serialisation when
// `pdl` is set (the kernel then overlaps its launch with the previous
// kernel's tail and waits for it in pdl_wait()).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Devices whose properties the launchers cache (ordinals 0..kMaxCachedDevices-1;
// a device beyond that is queried on every call).
constexpr int kMaxCachedDevices = 64;

// Multiprocessor count of the current device, 0 if it cannot be read.  The
// driver is asked once per device; later calls only read the current device
// ordinal (stored in *dev when dev is not null).
inline int current_device_sms(int *dev = nullptr)
{
    static std::atomic<int> cache[kMaxCachedDevices];  // 0: not read yet
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess)
        return 0;
    if (dev != nullptr)
        *dev = d;
    const bool cached = d >= 0 && d < kMaxCachedDevices;
    if (cached) {
        const int v = cache[d].load(std::memory_order_relaxed);
        if (v > 0)
            return v;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || sms < 0)
        return 0;
    if (cached && sms > 0)
        cache[d].store(sms, std::memory_order_relaxed);
    return sms;
}

cudaError_t launch_fused(Epilogue ep, const FusedArgs &a, bool pdl, cudaStream_t stream);
cudaError_t launch_ag(const AGArgs &a, bool pdl, cudaStream_t stream);
// Sharded RMSNorm over one (K == 0) or two (q and k) segments of each shard row.
cudaError_t launch_qk(const QKArgs &a, bool pdl, cudaStream_t stream);

}  // namespace tsfn

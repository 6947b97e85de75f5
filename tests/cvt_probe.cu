// Test-only probe: applies the library's conversion helpers (device_util.cuh)
// to arbitrary fp32 inputs so the GPU conversions can be compared with the
// oracle's encoders on exhaustive sweeps, and sweeps the FP8 1x128 block
// quotient over its whole bf16 domain against the IEEE divide.  Built by
// tests/test_gpu_cvt.py.
#include <cstdint>

#include "device_util.cuh"

namespace {

__global__ void probe_kernel(const float *__restrict__ x, int64_t n, uint16_t *bf16_out, uint8_t *e4m3_out,
                             uint8_t *e2m1_out)
{
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2;
    if (i + 1 >= n + 1)
        return;
    const float lo = x[i];
    const float hi = (i + 1 < n) ? x[i + 1] : 0.0f;
    const uint32_t b = tsfn::pack_bf16x2(lo, hi);
    const uint32_t e8 = tsfn::cvt_e4m3x2(lo, hi);
    const uint32_t e4 = tsfn::cvt_e2m1x2(lo, hi);
    bf16_out[i] = (uint16_t)(b & 0xFFFFu);
    e4m3_out[i] = (uint8_t)(e8 & 0xFFu);
    e2m1_out[i] = (uint8_t)(e4 & 0xFu);
    if (i + 1 < n) {
        bf16_out[i + 1] = (uint16_t)(b >> 16);
        e4m3_out[i + 1] = (uint8_t)(e8 >> 8);
        e2m1_out[i + 1] = (uint8_t)((e4 >> 4) & 0xFu);
    }
}

__global__ void e4m3_value_kernel(float *out)
{
    const uint32_t c = threadIdx.x + blockIdx.x * blockDim.x;
    if (c < 256)
        out[c] = tsfn::e4m3_value(c);
}

// Block blockIdx.x takes amax = the bf16 pattern blockIdx.x + 1 (every
// positive value up to +inf), s = amax/448 as the kernels form it, and every
// bf16 n with |n| <= amax: the E4M3 codes of tsfn::e4m3_block_codes against
// the codes of the IEEE quotients; mismatches counted per amax pattern.
__global__ void block_codes_kernel(uint32_t *mismatch)
{
    const uint32_t ab = blockIdx.x + 1;
    const float amax = __uint_as_float(ab << 16);
    const float s = __fdiv_rn(amax, 448.0f);
    uint32_t bad = 0;
    for (uint32_t g = threadIdx.x; g < 8192; g += blockDim.x) {
        float n[8], qd[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            n[e] = __uint_as_float((g * 8 + e) << 16);
            qd[e] = __fdiv_rn(n[e], s);
        }
        const uint2 got = tsfn::e4m3_block_codes(n, s), want = tsfn::cvt_e4m3x8(qd);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t gw = e < 4 ? got.x : got.y, ww = e < 4 ? want.x : want.y;
            const int sh = 8 * (e & 3);
            if (fabsf(n[e]) <= amax && ((gw >> sh) & 0xFFu) != ((ww >> sh) & 0xFFu))
                ++bad;
        }
    }
    if (bad)
        atomicAdd(&mismatch[ab], bad);
}

// Every non-negative bf16 value a (bit patterns 0 .. 0x7FFF, +inf and NaNs
// included): tsfn::div_const_rn for d = 448 (the 1x128 block scale) and d = 6
// (the NVFP4 scale factor) against the IEEE quotients, bit for bit (NaN
// against NaN).  mismatch[0] counts d = 448, mismatch[1] d = 6.
__global__ void div_const_kernel(uint32_t *mismatch)
{
    const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b > 0x7FFFu)
        return;
    const float a = __uint_as_float(b << 16);
    const float g448 = tsfn::div_const_rn(a, 448.0f, tsfn::kRcp448), w448 = __fdiv_rn(a, 448.0f);
    const float g6 = tsfn::div_const_rn(a, 6.0f, tsfn::kRcp6), w6 = __fdiv_rn(a, 6.0f);
    if (!((isnan(g448) && isnan(w448)) || __float_as_uint(g448) == __float_as_uint(w448)))
        atomicAdd(&mismatch[0], 1u);
    if (!((isnan(g6) && isnan(w6)) || __float_as_uint(g6) == __float_as_uint(w6)))
        atomicAdd(&mismatch[1], 1u);
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int cvt_probe(const float *x, int64_t n, uint16_t *bf16_out, uint8_t *e4m3_out, uint8_t *e2m1_out)
{
    if (n <= 0)
        return 0;
    const int64_t pairs = (n + 1) / 2;
    const int threads = 256;
    probe_kernel<<<(unsigned)((pairs + threads - 1) / threads), threads>>>(x, n, bf16_out, e4m3_out, e2m1_out);
    return (int)cudaGetLastError();
}

extern "C" __attribute__((visibility("default"))) int e4m3_values(float *out)
{
    e4m3_value_kernel<<<1, 256>>>(out);
    return (int)cudaGetLastError();
}

// mismatch: 0x7F81 counters, zeroed by the caller; entry a counts the bf16 n
// whose block-quotient code differs from the IEEE one for amax pattern a.
extern "C" __attribute__((visibility("default"))) int block_codes_probe(uint32_t *mismatch)
{
    block_codes_kernel<<<0x7F80, 256>>>(mismatch);
    return (int)cudaGetLastError();
}

// mismatch: two counters, zeroed by the caller.
extern "C" __attribute__((visibility("default"))) int div_const_probe(uint32_t *mismatch)
{
    div_const_kernel<<<128, 256>>>(mismatch);
    return (int)cudaGetLastError();
}

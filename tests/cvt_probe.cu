// Test-only probe: applies the library's conversion helpers (device_util.cuh)
// to arbitrary fp32 inputs so the GPU conversions can be compared with the
// oracle's encoders on exhaustive sweeps.  Built by tests/test_gpu_cvt.py.
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

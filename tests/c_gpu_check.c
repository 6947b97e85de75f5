/* Plain C99 caller of the library on a GPU: device buffers from the CUDA
 * runtime's C API, one kARResidualRMSNorm call (R=2, T=3, H=256) on the legacy
 * default stream, and the same call on pinned host buffers.  Built and run by
 * tests/test_c_abi.py.  With p0 = 1, p1 = 2, residual = 0.5 and gamma = 1 in
 * every column, x = 3.5 exactly, residual_out = bf16(3.5) = 0x4060 and
 * norm = bf16(3.5 * rsqrt(3.5^2 + 1e-6)) = bf16(0.99999996) = 1.0 = 0x3F80.
 * Prints "ok" and returns 0 when every element is as stated. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ts_fused_norm.h"

enum { R = 2, T = 3, H = 256, N = T * H };

static int check(const char *what, const uint16_t *res_out, const uint16_t *norm_out)
{
    int bad = 0;
    for (int i = 0; i < N; ++i)
        bad += res_out[i] != 0x4060u || norm_out[i] != 0x3F80u;
    if (bad)
        printf("%s: %d wrong elements (first: residual_out 0x%04x, norm_out 0x%04x)\n", what, bad,
               (unsigned)res_out[0], (unsigned)norm_out[0]);
    return bad;
}

static void fill(uint16_t *p, int n, uint16_t v)
{
    for (int i = 0; i < n; ++i)
        p[i] = v;
}

int main(void)
{
    static uint16_t h_p0[N], h_p1[N], h_res[N], h_gamma[H], h_ro[N], h_no[N];
    fill(h_p0, N, 0x3F80u);    /* 1.0 */
    fill(h_p1, N, 0x4000u);    /* 2.0 */
    fill(h_res, N, 0x3F00u);   /* 0.5 */
    fill(h_gamma, H, 0x3F80u); /* 1.0 */
    int failures = 0;

    /* device buffers */
    void *d[6];
    const size_t sizes[6] = {N * 2, N * 2, N * 2, H * 2, N * 2, N * 2};
    for (int i = 0; i < 6; ++i)
        if (cudaMalloc(&d[i], sizes[i]) != cudaSuccess) {
            printf("cudaMalloc failed\n");
            return 1;
        }
    cudaMemcpy(d[0], h_p0, N * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(d[1], h_p1, N * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(d[2], h_res, N * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(d[3], h_gamma, H * 2, cudaMemcpyHostToDevice);
    const void *parts[R] = {d[0], d[1]};
    ts_outs_t outs;
    memset(&outs, 0, sizeof(outs));
    outs.residual_out = d[4];
    outs.norm_out = d[5];
    outs.sf_layout = TS_SF_LINEAR;
    int st = ts_fused_reduce_norm(TS_AR_RES_RMS, parts, R, d[2], d[3], 1e-6f, NULL, T, H, &outs, TS_FLAG_PDL, NULL);
    if (st != TS_OK) {
        printf("device call: %s: %s\n", ts_status_string(st), ts_last_error_detail());
        return 1;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        printf("device call failed on the GPU\n");
        return 1;
    }
    cudaMemcpy(h_ro, d[4], N * 2, cudaMemcpyDeviceToHost);
    cudaMemcpy(h_no, d[5], N * 2, cudaMemcpyDeviceToHost);
    failures += check("device buffers", h_ro, h_no);
    for (int i = 0; i < 6; ++i)
        cudaFree(d[i]);

    /* pinned host buffers, addressed by the kernel across the host link */
    uint16_t *p[6];
    for (int i = 0; i < 6; ++i)
        if (cudaHostAlloc((void **)&p[i], sizes[i], cudaHostAllocDefault) != cudaSuccess) {
            printf("cudaHostAlloc failed\n");
            return 1;
        }
    memcpy(p[0], h_p0, N * 2);
    memcpy(p[1], h_p1, N * 2);
    memcpy(p[2], h_res, N * 2);
    memcpy(p[3], h_gamma, H * 2);
    memset(p[4], 0, N * 2);
    memset(p[5], 0, N * 2);
    const void *hparts[R] = {p[0], p[1]};
    outs.residual_out = p[4];
    outs.norm_out = p[5];
    st = ts_fused_reduce_norm(TS_AR_RES_RMS, hparts, R, p[2], p[3], 1e-6f, NULL, T, H, &outs, 0, NULL);
    if (st != TS_OK) {
        printf("host-buffer call: %s: %s\n", ts_status_string(st), ts_last_error_detail());
        return 1;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        printf("host-buffer call failed on the GPU\n");
        return 1;
    }
    failures += check("pinned host buffers", p[4], p[5]);
    for (int i = 0; i < 6; ++i)
        cudaFreeHost(p[i]);

    if (failures == 0)
        printf("ok\n");
    return failures == 0 ? 0 : 1;
}

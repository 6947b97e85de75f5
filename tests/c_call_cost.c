/* Host time of one call of each C-ABI entry point, from a plain C99 caller.
 *
 * Every call is a small decode-sized launch (16 tokens) on a created stream,
 * with TS_FLAG_PDL.  For each entry point: 50 untimed calls, then 25 batches
 * of 200 calls, each batch timed on the host clock around the calls only (the
 * stream is synchronised after the clock stops, so no batch waits for the
 * GPU: 200 launches stay well inside the launch queue).  The per-call figure
 * is the median batch time / 200, in microseconds.  It is what the library
 * costs the calling thread: argument checks, the launch configuration and
 * cudaLaunchKernelEx.
 *
 * Prints one JSON object and returns 0, or prints the failing call and
 * returns 1.  Built and run by tests/test_gpu_call_cost.py and bench.py. */
#define _POSIX_C_SOURCE 199309L
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <cuda_runtime_api.h>

#include "ts_fused_norm.h"

enum { BATCH = 200, BATCHES = 25, WARM = 50, TOK = 16 };

static double now_us(void)
{
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return (double)ts.tv_sec * 1e6 + (double)ts.tv_nsec * 1e-3;
}

static int cmp_double(const void *a, const void *b)
{
    const double x = *(const double *)a, y = *(const double *)b;
    return (x > y) - (x < y);
}

static void *dev_zeros(size_t bytes)
{
    void *p = NULL;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        printf("cudaMalloc(%zu) failed\n", bytes);
        exit(1);
    }
    cudaMemset(p, 0, bytes);
    return p;
}

typedef int (*call_fn)(void *ctx);

struct fused_ctx {
    int pattern, R;
    const void *parts[16];
    void *res, *gamma, *add;
    const float *scale;
    int64_t T, H;
    ts_outs_t outs;
    cudaStream_t s;
};

static int call_fused(void *p)
{
    struct fused_ctx *c = (struct fused_ctx *)p;
    return ts_fused_reduce_norm(c->pattern, c->parts, c->R, c->res, c->gamma, 1e-6f, c->scale, c->T, c->H,
                                &c->outs, TS_FLAG_PDL, c->s);
}

static int call_rs(void *p)
{
    struct fused_ctx *c = (struct fused_ctx *)p;
    return ts_reducescatter_fused_norm(TS_RS_ADD_RES_RMS, c->parts, c->R, 0, c->add, c->res, c->gamma, 1e-6f,
                                       NULL, c->T, c->H, &c->outs, TS_FLAG_PDL, c->s);
}

struct qk_ctx {
    const void *shards[8];
    void *wq, *wk, *qo, *ko;
    cudaStream_t s;
};

static int call_qk(void *p)
{
    struct qk_ctx *c = (struct qk_ctx *)p;
    return ts_qk_norm_sharded(c->shards, 8, TOK, 1280, 1024, 128, c->wq, c->wk, 1e-6f, c->qo, 8 * 1024, c->ko,
                              8 * 128, TS_FLAG_PDL, c->s);
}

static int call_rms(void *p)
{
    struct qk_ctx *c = (struct qk_ctx *)p;
    return ts_rms_norm_sharded(c->shards, 8, TOK, 1280, 768, c->wq, 1e-6f, c->qo, 8 * 768, TS_FLAG_PDL, c->s);
}

struct ag_ctx {
    const void *inputs[8];
    void *xg, *yg, *ago, *yo, *qo, *so;
    cudaStream_t s;
};

static int call_ag(void *p)
{
    struct ag_ctx *c = (struct ag_ctx *)p;
    return ts_allgather_fused_norm(TS_AG_RMS_FP8_BLOCKWISE, c->inputs, 8, TOK, 2112, 1536, 512, 64, c->xg, c->yg,
                                   1e-6f, 1e-6f, c->ago, NULL, c->yo, c->qo, c->so, TS_FLAG_PDL, c->s);
}

/* median host microseconds per call, or a negative value on a failed call */
static double per_call_us(const char *name, call_fn fn, void *ctx, cudaStream_t s)
{
    double t[BATCHES];
    for (int i = 0; i < WARM; ++i) {
        const int st = fn(ctx);
        if (st != TS_OK) {
            printf("%s: %s: %s\n", name, ts_status_string(st), ts_last_error_detail());
            return -1.0;
        }
    }
    cudaStreamSynchronize(s);
    for (int b = 0; b < BATCHES; ++b) {
        const double t0 = now_us();
        for (int i = 0; i < BATCH; ++i)
            fn(ctx);
        t[b] = (now_us() - t0) / BATCH;
        cudaStreamSynchronize(s);
    }
    if (cudaGetLastError() != cudaSuccess) {
        printf("%s: a launch failed on the GPU\n", name);
        return -1.0;
    }
    qsort(t, BATCHES, sizeof(double), cmp_double);
    return t[BATCHES / 2];
}

int main(void)
{
    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
        printf("cudaStreamCreate failed\n");
        return 1;
    }
    /* fused: R=8, 16 tokens, H=7168 (bf16 norm and FP8 1x128); NVFP4 R=4 H=5120 */
    struct fused_ctx f;
    memset(&f, 0, sizeof(f));
    f.R = 8;
    f.T = TOK;
    f.H = 7168;
    f.s = s;
    for (int r = 0; r < 8; ++r)
        f.parts[r] = dev_zeros(TOK * 7168 * 2);
    f.res = dev_zeros(TOK * 7168 * 2);
    f.add = dev_zeros(TOK * 7168 * 2);
    f.gamma = dev_zeros(7168 * 2);
    float *scale = (float *)dev_zeros(4);
    void *ro = dev_zeros(TOK * 7168 * 2), *no = dev_zeros(TOK * 7168 * 2), *q = dev_zeros(TOK * 7168);
    void *sc = dev_zeros(128 * 7168 / 16 * 4);
    f.outs.residual_out = ro;
    f.outs.sf_layout = TS_SF_LINEAR;

    double us[7];
    f.pattern = TS_AR_RES_RMS;
    f.outs.norm_out = no;
    us[0] = per_call_us("fused pattern 1", call_fused, &f, s);
    f.pattern = TS_AR_RES_RMS_FP8_BLOCKWISE;
    f.outs.norm_out = NULL;
    f.outs.quant_out = q;
    f.outs.scale_out = sc;
    us[1] = per_call_us("fused pattern 6", call_fused, &f, s);
    f.pattern = TS_AR_RES_RMS_FP4;
    f.R = 4;
    f.H = 5120;
    f.scale = scale;
    f.outs.sf_layout = TS_SF_SWIZZLED_128x4;
    us[2] = per_call_us("fused pattern 3", call_fused, &f, s);
    f.R = 8;
    f.H = 7168;
    f.scale = NULL;
    f.outs.quant_out = NULL;
    f.outs.scale_out = NULL;
    f.outs.sf_layout = TS_SF_LINEAR;
    f.outs.norm_out = no;
    us[3] = per_call_us("reduce-scatter 8", call_rs, &f, s);

    struct qk_ctx k;
    memset(&k, 0, sizeof(k));
    k.s = s;
    for (int r = 0; r < 8; ++r)
        k.shards[r] = dev_zeros(TOK * 1280 * 2);
    k.wq = dev_zeros(8 * 1024 * 2);
    k.wk = dev_zeros(8 * 128 * 2);
    k.qo = dev_zeros(TOK * 8 * 1024 * 2);
    k.ko = dev_zeros(TOK * 8 * 128 * 2);
    us[4] = per_call_us("qk", call_qk, &k, s);
    us[5] = per_call_us("rms sharded", call_rms, &k, s);

    struct ag_ctx a;
    memset(&a, 0, sizeof(a));
    a.s = s;
    for (int r = 0; r < 8; ++r)
        a.inputs[r] = dev_zeros(2 * 2112 * 2);
    a.xg = dev_zeros(1536 * 2);
    a.yg = dev_zeros(512 * 2);
    a.ago = dev_zeros(TOK * 2112 * 2);
    a.yo = dev_zeros(TOK * 512 * 2);
    a.qo = dev_zeros(TOK * 1536);
    a.so = dev_zeros(TOK * 12 * 4);
    us[6] = per_call_us("all-gather 2", call_ag, &a, s);

    for (int i = 0; i < 7; ++i)
        if (us[i] < 0.0)
            return 1;
    printf("{\"fused_p1_R8_H7168\": %.3f, \"fused_p6_R8_H7168\": %.3f, \"fused_p3_R4_H5120_swizzled\": %.3f, "
           "\"reducescatter_add_R8_H7168\": %.3f, \"qk_R8\": %.3f, \"rms_sharded_R8\": %.3f, "
           "\"allgather_fp8_R8\": %.3f, \"tokens\": %d, \"unit\": \"host us per call\"}\n",
           us[0], us[1], us[2], us[3], us[4], us[5], us[6], TOK);
    return 0;
}

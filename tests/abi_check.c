/* Plain C99 caller of the library's C ABI (include/ts_fused_norm.h), built and
 * run by tests/test_c_abi.py on a machine without a GPU: every call below
 * either validates and returns before any launch (T == 0) or is rejected on
 * the host, so no kernel runs.  Prints "ok" and returns 0 when every status
 * is the expected one. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ts_fused_norm.h"

static int failures = 0;

static void expect(const char *what, int got, int want)
{
    if (got != want) {
        printf("%s: got %s (%s), want %s\n", what, ts_status_string(got), ts_last_error_detail(),
               ts_status_string(want));
        ++failures;
    }
}

int main(void)
{
    /* fake, aligned, non-overlapping device addresses: never dereferenced */
    uintptr_t base = (uintptr_t)1 << 40;
    const void *partials[2] = {(const void *)base, (const void *)(base + 0x1000000)};
    const void *residual = (const void *)(base + 0x2000000);
    const void *gamma = (const void *)(base + 0x3000000);
    const float *sf = (const float *)(base + 0x4000000);
    ts_outs_t outs;
    memset(&outs, 0, sizeof(outs));
    outs.residual_out = (void *)(base + 0x5000000);
    outs.norm_out = (void *)(base + 0x6000000);
    outs.sf_layout = TS_SF_LINEAR;

    expect("T=0 kARResidualRMSNorm",
           ts_fused_reduce_norm(TS_AR_RES_RMS, partials, 2, residual, gamma, 1e-6f, NULL, 0, 256, &outs, 0, NULL),
           TS_OK);
    expect("T=0 with PDL",
           ts_fused_reduce_norm(TS_AR_RES_RMS, partials, 2, residual, gamma, 1e-6f, NULL, 0, 256, &outs,
                                TS_FLAG_PDL, NULL),
           TS_OK);
    expect("pattern 9",
           ts_fused_reduce_norm(9, partials, 2, residual, gamma, 1e-6f, NULL, 4, 256, &outs, 0, NULL),
           TS_ERR_BAD_PATTERN);
    expect("H % 8",
           ts_fused_reduce_norm(TS_AR_RES_RMS, partials, 2, residual, gamma, 1e-6f, NULL, 4, 250, &outs, 0, NULL),
           TS_ERR_SHAPE);
    expect("FP8 without scale_factor",
           ts_fused_reduce_norm(TS_AR_RES_RMS_FP8, partials, 2, residual, gamma, 1e-6f, NULL, 4, 256, &outs, 0,
                                NULL),
           TS_ERR_NULL);
    (void)sf;
    expect("misaligned partial",
           ts_fused_reduce_norm(TS_AR_RES_RMS, (const void *const[]){(const void *)(base + 2), partials[1]}, 2,
                                residual, gamma, 1e-6f, NULL, 4, 256, &outs, 0, NULL),
           TS_ERR_ALIGN);
    outs.norm_out = (void *)(base + 0x5000010); /* overlaps residual_out */
    expect("overlapping outputs",
           ts_fused_reduce_norm(TS_AR_RES_RMS, partials, 2, residual, gamma, 1e-6f, NULL, 4, 256, &outs, 0, NULL),
           TS_ERR_ALIAS);
    outs.norm_out = (void *)(base + 0x6000000);

    expect("reduce-scatter rank out of range",
           ts_reducescatter_fused_norm(TS_RS_ADD_RES_RMS, partials, 2, 2, residual, residual, gamma, 1e-6f, NULL,
                                       4, 256, &outs, 0, NULL),
           TS_ERR_SHAPE);
    expect("reduce-scatter T=0, all ranks",
           ts_reducescatter_fused_norm(TS_RS_RES_RMS, partials, 2, -1, NULL, residual, gamma, 1e-6f, NULL, 0, 256,
                                       &outs, 0, NULL),
           TS_OK);

    const void *shards[2] = {partials[0], partials[1]};
    expect("QK T=0",
           ts_qk_norm_sharded(shards, 2, 0, 1280, 1024, 128, gamma, residual, 1e-6f, outs.residual_out, 2048,
                              outs.norm_out, 256, 0, NULL),
           TS_OK);
    expect("QK q_shard % 8",
           ts_qk_norm_sharded(shards, 2, 4, 1280, 1020, 128, gamma, residual, 1e-6f, outs.residual_out, 2048,
                              outs.norm_out, 256, 0, NULL),
           TS_ERR_SHAPE);
    expect("single-matrix T=0",
           ts_rms_norm_sharded(shards, 2, 0, 768, 768, gamma, 1e-6f, outs.norm_out, 1536, 0, NULL), TS_OK);
    expect("all-gather hidden mismatch",
           ts_allgather_fused_norm(TS_AG_RMS, shards, 2, 4, 2104, 1536, 512, 64, gamma, residual, 1e-6f, 1e-6f,
                                   outs.residual_out, outs.norm_out, (void *)(base + 0x7000000), NULL, NULL, 0,
                                   NULL),
           TS_ERR_SHAPE);
    if (strcmp(ts_status_string(TS_ERR_LAUNCH), "TS_ERR_LAUNCH") != 0)
        ++failures;
    if (failures == 0)
        printf("ok\n");
    return failures == 0 ? 0 : 1;
}

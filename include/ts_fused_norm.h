/*
 * ts_fused_norm.h: C ABI of the GB300 (sm_103a) fused "reduce R partials ->
 * add residual -> RMSNorm -> optional FP8 / NVFP4 quantise" epilogue and of
 * the tensor-parallel MiniMax QK-RMSNorm, restated for one GPU.
 *
 * What the calls compute is defined by three pages:
 *   - tokenspeed `thirdparty/cuda/trtllm.py`: the `AllReduceFusionPattern`
 *     codes (kept here with the same numbers), `QuantizationSFLayout`, and
 *     `trtllm_allreduce_fusion` (its inputs, its optional outputs
 *     allreduce_out / residual_out / norm_out / partial_norm_out /
 *     quant_out / scale_out, rms_gamma, rms_eps, scale_factor, layout_code).
 *   - tokenspeed `ops/communication/triton.py`: `amd_all_reduce_kernel` and
 *     `amd_allreduce_residual_rmsnorm_kernel`, the executable statement of the
 *     math (fp32 sum over peers in ascending order, + residual, mean of
 *     squares, rsqrt(var + eps), x * scale * weight).
 *   - vLLM `minimax_rms_norm/rms_norm_tp`: `_minimax_qk_norm_tp_eager`,
 *     `_minimax_qk_var_kernel`, `_minimax_rms_apply_kernel`.
 * On one GPU the R rank partials (or the R tensor-parallel shards) are R
 * buffers in this GPU's memory: there is no communication, no workspace and
 * no inter-GPU synchronisation.
 *
 * Conventions for every entry point:
 *   - Every tensor pointer is device-accessible memory owned by the caller:
 *     device memory, or page-locked host memory allocated or registered
 *     through CUDA (cudaHostAlloc, cudaHostRegister), which on a system with
 *     unified addressing a kernel reads and writes at its host address.  With
 *     host buffers the kernel itself moves the bytes across the host link
 *     (NVLink-C2C on a Grace-Blackwell node): no staging copy is needed.  A
 *     pointer to ordinary pageable host memory is outside this contract.  The
 *     library allocates no memory and never synchronises: a call validates
 *     its arguments on the host, enqueues one kernel on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) and returns.  Between
 *     calls it keeps only the calling thread's last error detail and, per
 *     device, the SM count and occupancy figures read on the first call.  Arrays of pointers (`partials`, `qkv_shards`) and the
 *     `ts_outs_t` struct live in HOST memory and are read during the call only.
 *   - bf16 tensors are row-major and contiguous unless a leading dimension is
 *     given.  Tensor base pointers must be 16-byte aligned (128-bit vector
 *     access); fp32 scalars / scale arrays need 4-byte alignment.
 *   - Results are deterministic and per row: a row's (token's) outputs depend
 *     on its own inputs, R, the widths, the pattern and its scalars only, not
 *     on T, on the other rows, on the flags or on where the buffers live, so
 *     the same row gives the same bits in every call (a reduce-scatter slice
 *     equals the matching rows of the all-reduce form).
 *   - Errors: the return value is TS_OK (0) or a negative ts_status_t.  All
 *     argument checks run on the host before anything is launched, so a
 *     rejected call touches no memory.  ts_last_error_detail() returns a
 *     human-readable reason for the last failure on the calling thread.
 *     TS_ERR_LAUNCH reports a CUDA error raised by the launch itself
 *     (the CUDA error name is in the detail string).
 */
#ifndef TS_FUSED_NORM_H
#define TS_FUSED_NORM_H

#include <stdint.h>

#if defined(__GNUC__)
#define TS_API __attribute__((visibility("default")))
#else
#define TS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TS_OK = 0,
    TS_ERR_BAD_PATTERN = -1, /* pattern code outside 0..8, or an unknown SF layout       */
    TS_ERR_NULL = -2,        /* a required pointer is NULL                              */
    TS_ERR_SHAPE = -3,       /* sizes out of range / not multiples the pattern requires  */
    TS_ERR_ALIGN = -4,       /* a pointer is not aligned as required                     */
    TS_ERR_UNSUPPORTED = -5, /* valid request the library does not implement, or an output
                                pointer the pattern does not define                      */
    TS_ERR_ALIAS = -6,       /* overlapping buffers (other than the allowed in-place ones) */
    TS_ERR_LAUNCH = -7       /* the CUDA launch failed                                    */
} ts_status_t;

/* Launch flags (the `flags` argument of the compute calls). */
enum {
    /* Programmatic dependent launch (the pages' `launch_with_pdl`): the kernel
     * is launched with programmatic stream serialisation, so its launch and
     * prologue overlap the tail of the previous kernel in the stream; it waits
     * (griddepcontrol.wait) for that kernel to complete before it touches any
     * memory, and lets the next kernel start launching once its own loads are
     * issued.  Results are identical with and without the flag. */
    TS_FLAG_PDL = 1u,
    /* With TS_FLAG_PDL, for ts_fused_reduce_norm and ts_reducescatter_fused_norm
     * only: the kernel reads the first part of its inputs (partials, residual,
     * add_in) before it waits for the previous kernel in the stream, so that
     * those reads overlap that kernel's last CTAs.  Set it only when the
     * previous kernel writes none of this call's inputs (for example the
     * per-rank calls of one reduce-scatter, or calls on buffers produced
     * earlier); the kernel still waits before it writes any output, so a
     * previous kernel that reads this call's outputs is safe either way.
     * Results are identical with and without the flag.  It takes effect for 2
     * to 8 partials with rows of up to 4096 columns, and with rows of up to
     * 8192 columns when there are more rows than SMs; elsewhere, and without
     * TS_FLAG_PDL, it is accepted and changes nothing.  An extension: the
     * pages have only launch_with_pdl. */
    TS_FLAG_PDL_EARLY_READ = 2u,
    /* With TS_FLAG_PDL, for ts_fused_reduce_norm and ts_reducescatter_fused_norm
     * only: the kernel does all of its work without waiting for the kernels
     * before it in the stream and waits for them only before it finishes, so it
     * still completes after them and any later work in the stream sees every
     * result.  It may therefore run at the same time as the earlier calls of a
     * run of calls made with this flag and as the kernel just before that run
     * (a call made without it waits for its predecessors before it starts and
     * so ends the run).  The caller guarantees that none of those kernels
     * writes this call's inputs or reads or writes its outputs: for example
     * the per-rank calls of one reduce-scatter, which read the same inputs and
     * write disjoint outputs.  Results are identical with and without the flag.
     * It takes effect where TS_FLAG_PDL_EARLY_READ does; elsewhere it is
     * accepted and changes nothing.  An extension: the pages have only
     * launch_with_pdl. */
    TS_FLAG_PDL_INDEPENDENT = 4u
};

/* Codes identical to `AllReduceFusionPattern` (tokenspeed trtllm.py). */
typedef enum {
    TS_AR = 0,                                 /* kAllReduce                                  */
    TS_AR_RES_RMS = 1,                         /* kARResidualRMSNorm                          */
    TS_AR_RES_RMS_FP8 = 2,                     /* kARResidualRMSNormFP8Quant                  */
    TS_AR_RES_RMS_FP4 = 3,                     /* kARResidualRMSNormFP4Quant                  */
    TS_AR_RES_RMS_OUT_FP8 = 4,                 /* kARResidualRMSNormOutFP8Quant               */
    TS_AR_RES_RMS_OUT_FP4 = 5,                 /* kARResidualRMSNormOutFP4Quant               */
    TS_AR_RES_RMS_FP8_BLOCKWISE = 6,           /* kARResidualRMSNormFP8BlockWiseQuant         */
    TS_AR_RES_RMS_PARTIAL_OUT_FP8_BLOCKWISE = 7, /* kARResidualRMSNormPartialOutFP8BlockWiseQuant */
    TS_AR_RES_RMS_PARTIAL_OUT = 8              /* kARResidualRMSNormPartialOut                */
} ts_pattern_t;

/* Codes identical to `QuantizationSFLayout` (tokenspeed trtllm.py). */
typedef enum {
    TS_SF_SWIZZLED_128x4 = 0,
    TS_SF_SWIZZLED_8x4 = 1,
    TS_SF_LINEAR = 2
} ts_sf_layout_t;

/*
 * Output set of ts_fused_reduce_norm.  Which members a pattern writes
 * (R = required, o = optional: written when non-NULL, - = must be NULL):
 *
 *   pattern            allreduce_out residual_out norm_out partial_norm_out quant_out scale_out
 *   0 kAllReduce             R            -          -           -             -         -
 *   1 ResidualRMSNorm        o            R          R           -             -         -
 *   2 ...FP8Quant            o            R          -           -             R         -
 *   3 ...FP4Quant            o            R          -           -             R         R
 *   4 ...OutFP8Quant         o            R          R           -             R         -
 *   5 ...OutFP4Quant         o            R          R           -             R         R
 *   6 ...FP8BlockWise        o            R          -           -             R         R
 *   7 ...PartialOutFP8BW     o            R          -           R             R         R
 *   8 ...PartialOut          o            R          o           R             -         -
 *
 *   allreduce_out     bf16 [T, H]: bf16(sum of partials).  May equal partials[0]
 *                     (in place, as the Triton all_reduce writes its result
 *                     into its input); no other overlap.
 *   residual_out      bf16 [T, H]: bf16(sum + residual).  May equal `residual`.
 *   norm_out          bf16 [T, H]: n = bf16((x * rsqrt(mean(x^2) + eps)) * gamma),
 *                     x the unrounded fp32 sum + residual.
 *   partial_norm_out  bf16 [T, partial_cols]: the first partial_cols columns of n
 *                     (row stride partial_cols); the RMS still spans all H.
 *   partial_cols      0 < P <= H, P % 8 == 0 (patterns 7, 8; ignored otherwise).
 *   quant_out         patterns 2, 4, 6, 7: FP8 E4M3 codes, uint8 [T, H].
 *                     patterns 3, 5: NVFP4 E2M1 codes, uint8 [T, H/2], two per
 *                     byte, element 2k in the low nibble of byte k.
 *   scale_out         patterns 6, 7: fp32 [T, H/128], s = amax(|n| over 128
 *                     columns) / 448, codes e4m3(n / s) (0 for an all-zero group).
 *                     patterns 3, 5: E4M3 scale factors, one per 16 columns,
 *                     SF = e4m3(g * amax/6), codes e2m1(n * (g / value(SF))),
 *                     laid out per sf_layout:
 *                       TS_SF_LINEAR: uint8 [T, H/16];
 *                       TS_SF_SWIZZLED_128x4: uint8 [ceil(T/128)*128,
 *                       ceil(H/64)*4] in 512-byte tiles of 128 rows x 4
 *                       columns; SF (m, k) at byte
 *                       ((m/128)*(Kp/4) + k/4)*512 + (m%32)*16 + ((m%128)/32)*4 + k%4
 *                       with Kp = ceil(H/64)*4.  Padding bytes are written as 0.
 *                       TS_SF_SWIZZLED_8x4: uint8 [ceil(T/8)*8, Kp] in 32-byte
 *                       tiles of 8 rows x 4 columns, row-major inside a tile:
 *                       SF (m, k) at byte ((m/8)*(Kp/4) + k/4)*32 + (m%8)*4 + k%4.
 *                       Padding bytes are written as 0.  (The pages name both
 *                       swizzled layouts without defining them; these are the
 *                       library's definitions.)
 *   sf_layout         ts_sf_layout_t (patterns 3, 5; ignored otherwise).
 */
typedef struct {
    void *allreduce_out;
    void *residual_out;
    void *norm_out;
    void *partial_norm_out;
    int64_t partial_cols;
    void *quant_out;
    void *scale_out;
    int32_t sf_layout;
    int32_t reserved; /* must be 0 */
} ts_outs_t;

/*
 * ts_fused_reduce_norm: one AllReduceFusionPattern over T rows of width H
 * (tokenspeed trtllm.py `trtllm_allreduce_fusion`; the math of tokenspeed
 * triton.py `amd_allreduce_residual_rmsnorm_kernel` / `amd_all_reduce_kernel`):
 *
 *   a[t,j]  = ((0 + p0[t,j]) + p1[t,j]) + ... + p_{R-1}[t,j]      fp32, r ascending
 *   x[t,j]  = a[t,j] + residual[t,j]                             fp32
 *   s[t]    = rsqrt(sum_j x[t,j]^2 / H + eps)                    fp32
 *   n[t,j]  = bf16((x[t,j] * s[t]) * gamma[j])
 *   then the outputs listed above for the pattern.
 *
 *   pattern       ts_pattern_t.
 *   partials      host array of R device-accessible pointers, each bf16 [T, H].
 *   R             1..16.
 *   residual      bf16 [T, H]; required for patterns 1..8 (ignored for 0).
 *   gamma         bf16 [H] (rms_gamma); required for patterns 1..8.
 *   eps           rms_eps, added inside the rsqrt (e.g. 1e-6).
 *   scale_factor  fp32[1] in device-accessible memory: the per-tensor FP8 scale
 *                 sigma (patterns 2, 4: code = e4m3(n * sigma)) or the NVFP4
 *                 global scale g (patterns 3, 5); required for 2..5, ignored
 *                 otherwise.  A pointer, read by the kernel, so the call can be
 *                 captured in a CUDA graph.
 *   T             rows (tokens), >= 0.  T == 0 validates and returns TS_OK
 *                 without launching; the per-row buffers (partials, residual,
 *                 outputs) may then be NULL, as empty tensors are.
 *   H             hidden size: multiple of 8, <= 16384; multiple of 128 for
 *                 patterns 6, 7; multiple of 16 for patterns 3, 5.
 *   outs          host pointer to the output set (see ts_outs_t).
 *   flags         0, TS_FLAG_PDL, or TS_FLAG_PDL with TS_FLAG_PDL_EARLY_READ or
 *                 TS_FLAG_PDL_INDEPENDENT; other bits: TS_ERR_UNSUPPORTED.
 *   stream        cudaStream_t.
 */
TS_API int ts_fused_reduce_norm(int pattern, const void *const *partials, int R, const void *residual,
                                const void *gamma, float eps, const float *scale_factor, int64_t T,
                                int64_t H, const ts_outs_t *outs, uint32_t flags, void *stream);

/* Codes identical to `ReduceScatterFusionPattern` (tokenspeed trtllm.py). */
typedef enum {
    TS_RS = 0,                              /* kReduceScatter                           */
    TS_RS_RES_RMS = 1,                      /* kRSResidualRMSNorm                       */
    TS_RS_RES_RMS_FP8 = 2,                  /* kRSResidualRMSNormFP8Quant               */
    TS_RS_RES_RMS_FP4 = 3,                  /* kRSResidualRMSNormFP4Quant               */
    TS_RS_RES_RMS_OUT_FP8 = 4,              /* kRSResidualRMSNormOutFP8Quant            */
    TS_RS_RES_RMS_OUT_FP4 = 5,              /* kRSResidualRMSNormOutFP4Quant            */
    TS_RS_RES_RMS_FP8_BLOCKWISE = 6,        /* kRSResidualRMSNormFP8BlockWiseQuant      */
    TS_RS_ADD_RES_RMS_FP8_BLOCKWISE = 7,    /* kRSAddResidualRMSNormFP8BlockWiseQuant   */
    TS_RS_ADD_RES_RMS = 8                   /* kRSAddResidualRMSNorm                    */
} ts_rs_pattern_t;

/*
 * ts_reducescatter_fused_norm: one rank's output of the reduce-scatter fusion
 * (tokenspeed trtllm.py `trtllm_reducescatter_fusion`), with the R ranks'
 * partials resident on this GPU (world size = R).  Rank `rank` owns the token
 * slice [start, start + count) of tokenspeed triton.py `rsag_get_token_dist`:
 * count = T/R, plus one for the first T%R ranks; slices in rank order.  Over
 * that slice the call computes the all-reduce-form epilogue (the table of
 * ts_outs_t, for the codes mapped below), with
 *
 *   x[i,j] = ((sum over r ascending of p_r[start+i, j]) + add_in[i,j]) + residual[i,j]
 *
 * (add_in only for codes 7 and 8), outs->allreduce_out playing the part of
 * `reducescatter_out` = bf16(sum of the partials, before add_in).
 *
 *   rs_pattern    ts_rs_pattern_t.  0..6 behave as AllReduceFusionPattern
 *                 0..6 on the slice; 7 = 6 with add_in; 8 = 1 with add_in.
 *   partials      host array of R device-accessible pointers, each bf16 [T, H] (all T
 *                 tokens; only the slice's rows are read).
 *   rank          0..R-1, or -1 for every rank's slice in one launch (the
 *                 slices in rank order are all T tokens: count = T, start = 0).
 *   add_in        bf16 [count, H]; required for codes 7 and 8, NULL otherwise.
 *   residual      bf16 [count, H] (the slice's rows; codes 1..8).
 *   outs          outputs with count rows (partial_norm_out must be NULL).
 *   gamma, eps, scale_factor, H, flags, stream: as for ts_fused_reduce_norm.
 * A rank whose slice is empty (T < R) validates and returns TS_OK.
 */
TS_API int ts_reducescatter_fused_norm(int rs_pattern, const void *const *partials, int R, int rank,
                                       const void *add_in, const void *residual, const void *gamma,
                                       float eps, const float *scale_factor, int64_t T, int64_t H,
                                       const ts_outs_t *outs, uint32_t flags, void *stream);

/* Codes identical to `AllGatherFusionPattern` (tokenspeed trtllm.py). */
typedef enum {
    TS_AG = 0,                      /* kAllGather                           */
    TS_AG_RMS = 1,                  /* kAllGatherfusedRMS                   */
    TS_AG_RMS_FP8_BLOCKWISE = 2     /* kAllGatherfusedRMSFP8BlockWiseQuant  */
} ts_ag_pattern_t;

/*
 * ts_allgather_fused_norm: the all-gather fusion with the dual RMSNorm of MLA
 * row segments (tokenspeed trtllm.py `trtllm_allgather_fusion`), with the R
 * ranks' token slices resident on this GPU.  The gathered tensor is the
 * slices in rank order (rank r holds T/R tokens, the first T%R ranks one
 * more: tokenspeed triton.py `rsag_get_token_dist`).  Each gathered row is
 * x (q_lora_rank columns) | y (kv_lora_rank) | rope (qk_rope_head_dim):
 *
 *   allgather_out[t, :] = the row                                  (all patterns)
 *   x_norm_out[t, j]    = bf16((x_j * rsqrt(sum(x^2)/q + x_eps)) * x_gamma[j])
 *   y_norm_out[t, j]    = bf16((y_j * rsqrt(sum(y^2)/kv + y_eps)) * y_gamma[j])
 *   pattern 2: the x norm n in FP8 1x128 blocks: scale_out[t, g] = amax/448 (fp32),
 *              quant_out[t, j] = e4m3(n_j / s) (0 for an all-zero block).
 *   The rope columns only appear in allgather_out.
 *
 *   ag_pattern    ts_ag_pattern_t.
 *   inputs        host array of R device-accessible pointers; inputs[r] is bf16
 *                 [count_r, hidden] (may be NULL when count_r == 0).
 *   T             gathered tokens, >= 0 (T == 0 returns TS_OK).
 *   hidden        = q_lora_rank + kv_lora_rank + qk_rope_head_dim <= 2112.
 *   q_lora_rank   positive multiple of 128; kv_lora_rank, qk_rope_head_dim
 *                 multiples of 8 (kv > 0, rope >= 0).
 *   x_gamma, y_gamma  bf16 [q_lora_rank], [kv_lora_rank] (patterns 1, 2).
 *   outputs       allgather_out bf16 [T, hidden] (required); x_norm_out bf16
 *                 [T, q] (required in 1, optional in 2, NULL in 0); y_norm_out
 *                 bf16 [T, kv] (1, 2); quant_out e4m3 [T, q] and scale_out fp32
 *                 [T, q/128] (2 only).  No output may overlap an input or
 *                 another output.
 *   flags, stream as for ts_fused_reduce_norm.
 */
TS_API int ts_allgather_fused_norm(int ag_pattern, const void *const *inputs, int R, int64_t T,
                                   int64_t hidden, int64_t q_lora_rank, int64_t kv_lora_rank,
                                   int64_t qk_rope_head_dim, const void *x_gamma, const void *y_gamma,
                                   float x_eps, float y_eps, void *allgather_out, void *x_norm_out,
                                   void *y_norm_out, void *quant_out, void *scale_out, uint32_t flags,
                                   void *stream);

/*
 * ts_qk_norm_sharded: MiniMax tensor-parallel QK-RMSNorm with the R shards
 * resident on this GPU (vLLM rms_norm_tp `_minimax_qk_norm_tp_eager`, split
 * as `_minimax_qk_var_kernel` + all-reduce of the [T, 2] fp32 variance +
 * `_minimax_rms_apply_kernel`; here one fused kernel):
 *
 *   vq_r[t] = sum_{j<Q} x_r[t,j]^2 / Q,   vk_r[t] = sum_{j<K} x_r[t,Q+j]^2 / K   fp32
 *   Vq[t]   = sum over r ascending of vq_r[t]   (likewise Vk)                fp32
 *   q_out[t, r*Q + j] = bf16((x_r[t,j]   * rsqrt(Vq[t]/R + eps)) * q_weight[r*Q + j])
 *   k_out[t, r*K + j] = bf16((x_r[t,Q+j] * rsqrt(Vk[t]/R + eps)) * k_weight[r*K + j])
 *
 *   qkv_shards    host array of R device-accessible pointers; shard r is bf16 [T, row_stride]
 *                 holding q (Q columns) | k (K columns) | v (not read).
 *   R             1..16.
 *   T             tokens, >= 0 (T == 0 returns TS_OK without launching; the
 *                 shards and outputs may then be NULL).
 *   row_stride    elements between consecutive tokens of a shard; multiple of 8,
 *                 >= Q + K.
 *   q_shard (Q)   8 <= Q <= 4096, multiple of 8.   k_shard (K): 8 <= K <= 1024,
 *                 multiple of 8.
 *   q_weight      bf16 [R*Q]; shard r uses q_weight[r*Q .. r*Q+Q).
 *   k_weight      bf16 [R*K].
 *   eps           added inside the rsqrt after the division by R.
 *   q_out, ldq    bf16 [T, ldq], ldq >= R*Q, multiple of 8: shard r's block at
 *                 columns r*Q .. r*Q+Q (the unsharded, hidden-concatenated layout).
 *   k_out, ldk    bf16 [T, ldk], ldk >= R*K, multiple of 8.
 *   flags         0 or TS_FLAG_PDL.
 *   Outputs must not overlap the shards, the weights or each other.
 */
TS_API int ts_qk_norm_sharded(const void *const *qkv_shards, int R, int64_t T, int64_t row_stride,
                              int64_t q_shard, int64_t k_shard, const void *q_weight,
                              const void *k_weight, float eps, void *q_out, int64_t ldq, void *k_out,
                              int64_t ldk, uint32_t flags, void *stream);

/*
 * ts_rms_norm_sharded: single-matrix RMSNorm over a hidden dim split in R
 * shards resident on this GPU (tokenspeed trtllm.py `minimax_allreduce_rms`:
 * the all-reduce of the per-token variance, then each shard's slice of the
 * norm with its slice of the weight), the one-segment form of the QK norm:
 *
 *   v_r[t] = sum_{j<W} x_r[t,j]^2 / W                                   fp32
 *   V[t]   = sum over r ascending of v_r[t]                             fp32
 *   out[t, r*W + j] = bf16((x_r[t,j] * rsqrt(V[t]/R + eps)) * weight[r*W + j])
 *
 *   shards        host array of R device-accessible pointers, shard r bf16 [T, row_stride]
 *                 (its slice in the first W columns).
 *   R             1..16.     T: tokens, >= 0 (T == 0 returns TS_OK).
 *   row_stride    multiple of 8, >= W.
 *   width (W)     8 <= W <= 4096, multiple of 8.
 *   weight        bf16 [R*W].
 *   out, ldo      bf16 [T, ldo], ldo >= R*W, multiple of 8; shard r's block at
 *                 columns r*W .. r*W+W.  Must not overlap the inputs.
 *   flags         0 or TS_FLAG_PDL.
 */
TS_API int ts_rms_norm_sharded(const void *const *shards, int R, int64_t T, int64_t row_stride,
                               int64_t width, const void *weight, float eps, void *out, int64_t ldo,
                               uint32_t flags, void *stream);

/* Static text for a ts_status_t value ("TS_OK", "TS_ERR_SHAPE", ...). */
TS_API const char *ts_status_string(int status);

/* Reason for the most recent failed call on the calling thread ("" if none).
 * The string stays valid until the next call on the same thread. */
TS_API const char *ts_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* TS_FUSED_NORM_H */

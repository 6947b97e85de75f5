/*
 * Reference oracle for the fused "reduce partials -> add residual -> RMSNorm
 * -> optional FP8 / NVFP4 quantise" epilogue and for the tensor-parallel
 * MiniMax QK-RMSNorm, as plain single-threaded C.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; it is written from the definitions on the source pages:
 *
 *   [P1] tokenspeed `thirdparty/cuda/trtllm.py`: `AllReduceFusionPattern`
 *        (codes 0..8), `QuantizationSFLayout`, `trtllm_allreduce_fusion`
 *        (inputs/outputs, `scale_factor` as an fp32 scalar, `fp32_acc`).
 *   [P2] tokenspeed `ops/communication/triton.py`: `amd_all_reduce_kernel`
 *        (the sum-only all-reduce) and `amd_allreduce_residual_rmsnorm_kernel`
 *        (reduce -> +residual -> mean of squares -> rsqrt(var+eps) ->
 *        x*scale*weight).
 *   [P3] vLLM `minimax_rms_norm/rms_norm_tp`: `_minimax_qk_norm_tp_eager`,
 *        `_minimax_qk_var_kernel`, `_minimax_rms_apply_kernel`.
 *
 * Precision.  The pages fix fp32 for the reduction and for every elementwise
 * step (the partials are widened to float32 and summed in a float32
 * accumulator, peers in ascending order; the residual is added in fp32; the
 * norm is x*scale*weight in fp32).  They leave the order of the row-wide sum
 * of squares open (a `tl.sum`), so the oracle takes the ideal: the sum of
 * squares is accumulated in double and rounded once to fp32, and rsqrt is the
 * correctly rounded fp32 value of 1/sqrt.  Everything else is IEEE fp32,
 * round-to-nearest-even, in the written order; this file must be compiled
 * with -ffp-contract=off and without fast-math.
 *
 * Readings where the pages are silent (numbered as in the design notes):
 *   c1  partial sum order ((0 + p0) + p1) + ... + p_{R-1}, then + residual.
 *   c2  the norm uses the unrounded fp32 x, not the bf16 residual_out.
 *   c6  every quantiser reads the bf16-rounded norm value n.
 *   c7  FP8 per-tensor: code = e4m3(n * scale_factor).
 *   c8  E4M3 (FN variant, max 448): round to nearest even, saturate to +-448.
 *   c9  1x128 blockwise: s = amax/448 (fp32 divide), code = e4m3(n / s);
 *       an all-zero group gives s = 0 and codes 0.
 *   c11 NVFP4: SF = e4m3(g * (amax/6)); d = value(SF);
 *       code = e2m1(n * (g / d)), or 0 when d == 0.
 *   c12 E2M1 grid {0,.5,1,1.5,2,3,4,6}: nearest, ties to even code, saturate 6.
 *   c13 two E2M1 codes per byte, even element in the low nibble.
 *   c14 SWIZZLED_128x4 scale-factor tile map (see orc_sf_offset_swizzled_128x4).
 *   c21 SWIZZLED_8x4 scale-factor tile map (see orc_sf_offset_swizzled_8x4).
 *       The pages only name these two layouts, so both maps are readings.
 *       The 128x4 map is pinned to the layout an NVFP4 block-scaled GEMM
 *       reads its scales in (a GPU test feeds scales placed by this map to
 *       PyTorch's NVFP4 scaled matmul).  The 8x4 map is parity unpinned: the
 *       tests pin only what follows from the reading (a bijection onto the
 *       padded buffer, the tile structure, zero padding).
 *   c15 partial_norm_out holds the first P columns of n; the RMS is over all H.
 *   c18 QK: rsqrt(V / R + eps), V the fp32 shard-ascending sum of shard means.
 *   c25 a sum of squares past fp32's range is +inf (fp32 accumulation), so
 *       rsqrt gives 0 and the norm of such a row is +-0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats, written from their definitions.                           */
/* ------------------------------------------------------------------------ */

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.  Normal numbers
 * (1 + f/128) * 2^(e-127); subnormals f * 2^-133; exponent 255 is inf/NaN. */
float orc_bf16_decode(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0xFF)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -133);
    else
        v = ldexp(1.0 + f / 128.0, e - 127);
    return (float)(sign ? -v : v);
}

/* Round |x| to the bfloat16 grid: the spacing of the grid in the binade of
 * |x| is 2^(E-7) (E = floor(log2|x|), clamped below at -126 for the
 * subnormal range); nearbyint() rounds to nearest, ties to even, which is
 * the even fraction because the fraction is the integer multiple's low bits. */
uint16_t orc_bf16_encode(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return (uint16_t)(sign | 0x7FC0);
    double a = fabs((double)x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;
    if (E < -126)
        E = -126;
    double q = ldexp(1.0, E - 7);
    double n = nearbyint(a / q);
    double r = n * q;
    double max_finite = ldexp(255.0 / 128.0, 127);
    if (r > max_finite)
        return (uint16_t)(sign | 0x7F80);
    if (r < ldexp(1.0, -126)) /* subnormal (or rounded up into the min normal below) */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -133)));
    frexp(r, &e2);
    int Er = e2 - 1;
    int frac = (int)((r / ldexp(1.0, Er) - 1.0) * 128.0);
    return (uint16_t)(sign | ((Er + 127) << 7) | frac);
}

/* FP8 E4M3 ("FN": no infinities, S.1111.111 is NaN): 4 exponent bits with
 * bias 7, 3 fraction bits.  Normal (1 + f/8) * 2^(e-7), subnormal f * 2^-9,
 * largest finite 1.75 * 2^8 = 448. */
float orc_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int f = c & 0x7;
    double v;
    if (e == 0xF && f == 0x7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp(1.0 + f / 8.0, e - 7);
    return (float)(sign ? -v : v);
}

/* Round to nearest on the E4M3 grid, ties to even, and saturate anything
 * beyond 448 (infinities included) to +-448.  Sign is kept (-0 -> 0x80). */
uint8_t orc_e4m3_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)x);
    if (a == 0.0)
        return sign;
    double r;
    if (isinf(a)) {
        r = 448.0;
    } else {
        int e2;
        frexp(a, &e2);
        int E = e2 - 1;
        if (E < -6)
            E = -6;
        double q = ldexp(1.0, E - 3);
        r = nearbyint(a / q) * q;
        if (r > 448.0)
            r = 448.0;
    }
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -6))
        return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    int e2;
    frexp(r, &e2);
    int Er = e2 - 1;
    int frac = (int)((r / ldexp(1.0, Er) - 1.0) * 8.0);
    return (uint8_t)(sign | ((Er + 7) << 3) | frac);
}

/* FP4 E2M1: 2 exponent bits with bias 1, 1 fraction bit, no inf/NaN.
 * Values 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6. */
float orc_e2m1_decode(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 0x3;
    int f = c & 0x1;
    double v = (e == 0) ? 0.5 * f : ldexp(1.0 + f / 2.0, e - 1);
    return (float)(sign ? -v : v);
}

/* Nearest E2M1 value, ties to the even code, saturating to +-6.  The format
 * has no NaN; a NaN input maps to +-6 here (never reached by the path). */
uint8_t orc_e2m1_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x8 : 0;
    double a = fabs((double)x);
    double r;
    if (isnan(x) || isinf(a)) {
        r = 6.0;
    } else if (a == 0.0) {
        return sign;
    } else {
        int e2;
        frexp(a, &e2);
        int E = e2 - 1;
        if (E < 0)
            E = 0;
        double q = ldexp(1.0, E - 1);
        r = nearbyint(a / q) * q;
        if (r > 6.0)
            r = 6.0;
    }
    if (r == 0.0)
        return sign;
    if (r < 1.0)
        return (uint8_t)(sign | 0x1); /* 0.5 */
    int e2;
    frexp(r, &e2);
    int Er = e2 - 1;
    int frac = (int)((r / ldexp(1.0, Er) - 1.0) * 2.0);
    return (uint8_t)(sign | ((Er + 1) << 1) | frac);
}

void orc_bf16_encode_n(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_encode(x[i]);
}

void orc_e4m3_encode_n(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(x[i]);
}

void orc_e2m1_encode_n(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e2m1_encode(x[i]);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 scale-factor layouts ([P1] `QuantizationSFLayout`).                */
/* ------------------------------------------------------------------------ */

/* Columns of the SWIZZLED_128x4 buffer: the number of scale factors per row
 * (n_sf_cols = H/16) padded up to a multiple of 4. */
int64_t orc_sf_swizzled_cols(int64_t n_sf_cols) { return (n_sf_cols + 3) / 4 * 4; }

/* Rows of the SWIZZLED_128x4 buffer: rows padded up to a multiple of 128. */
int64_t orc_sf_swizzled_rows(int64_t rows) { return (rows + 127) / 128 * 128; }

/* Byte offset of scale factor (m, k) in the SWIZZLED_128x4 layout (reading
 * c14).  The buffer is a row-major grid of 128-row x 4-column tiles of 512
 * bytes each.  Inside a tile, row m%128 = 32*i + j (i = 0..3, j = 0..31)
 * and column k%4 sit at byte 16*j + 4*i + k%4: the 32 rows j are the outer
 * 16-byte strides and each 16-byte group holds the 4 columns of rows j,
 * j+32, j+64, j+96. */
int64_t orc_sf_offset_swizzled_128x4(int64_t m, int64_t k, int64_t n_sf_cols)
{
    int64_t tiles_per_row = orc_sf_swizzled_cols(n_sf_cols) / 4;
    int64_t tile = (m / 128) * tiles_per_row + (k / 4);
    int64_t i = (m % 128) / 32;
    int64_t j = m % 32;
    return tile * 512 + j * 16 + i * 4 + (k % 4);
}

/* Rows of the SWIZZLED_8x4 buffer: rows padded up to a multiple of 8. */
int64_t orc_sf_swizzled8_rows(int64_t rows) { return (rows + 7) / 8 * 8; }

/* Byte offset of scale factor (m, k) in the SWIZZLED_8x4 layout (the pages
 * only name it; reading c21): a row-major grid of 8-row x 4-column tiles of 32
 * bytes, row-major inside a tile (row m%8 at byte 4*(m%8), column k%4 next). */
int64_t orc_sf_offset_swizzled_8x4(int64_t m, int64_t k, int64_t n_sf_cols)
{
    int64_t tiles_per_row = orc_sf_swizzled_cols(n_sf_cols) / 4;
    int64_t tile = (m / 8) * tiles_per_row + (k / 4);
    return tile * 32 + (m % 8) * 4 + (k % 4);
}

/* Scatter a LINEAR [rows, n_sf_cols] matrix into the padded SWIZZLED_8x4
 * buffer; padding bytes are 0. */
void orc_sf_swizzle_8x4(const uint8_t *linear, int64_t rows, int64_t n_sf_cols, uint8_t *out)
{
    int64_t size = orc_sf_swizzled8_rows(rows) * orc_sf_swizzled_cols(n_sf_cols);
    memset(out, 0, (size_t)size);
    for (int64_t m = 0; m < rows; ++m)
        for (int64_t k = 0; k < n_sf_cols; ++k)
            out[orc_sf_offset_swizzled_8x4(m, k, n_sf_cols)] = linear[m * n_sf_cols + k];
}

/* Scatter a LINEAR [rows, n_sf_cols] scale-factor matrix into the padded
 * SWIZZLED_128x4 buffer; padding bytes are 0. */
void orc_sf_swizzle_128x4(const uint8_t *linear, int64_t rows, int64_t n_sf_cols, uint8_t *out)
{
    int64_t size = orc_sf_swizzled_rows(rows) * orc_sf_swizzled_cols(n_sf_cols);
    memset(out, 0, (size_t)size);
    for (int64_t m = 0; m < rows; ++m)
        for (int64_t k = 0; k < n_sf_cols; ++k)
            out[orc_sf_offset_swizzled_128x4(m, k, n_sf_cols)] = linear[m * n_sf_cols + k];
}

/* ------------------------------------------------------------------------ */
/* Fused reduce -> residual -> RMSNorm (-> quantise), one row at a time.     */
/* ------------------------------------------------------------------------ */

enum {
    ORC_AR = 0,                        /* kAllReduce */
    ORC_AR_RES_RMS = 1,                /* kARResidualRMSNorm */
    ORC_AR_RES_RMS_FP8 = 2,            /* kARResidualRMSNormFP8Quant */
    ORC_AR_RES_RMS_FP4 = 3,            /* kARResidualRMSNormFP4Quant */
    ORC_AR_RES_RMS_OUT_FP8 = 4,        /* kARResidualRMSNormOutFP8Quant */
    ORC_AR_RES_RMS_OUT_FP4 = 5,        /* kARResidualRMSNormOutFP4Quant */
    ORC_AR_RES_RMS_FP8_BLOCK = 6,      /* kARResidualRMSNormFP8BlockWiseQuant */
    ORC_AR_RES_RMS_PART_FP8_BLOCK = 7, /* kARResidualRMSNormPartialOutFP8BlockWiseQuant */
    ORC_AR_RES_RMS_PART = 8            /* kARResidualRMSNormPartialOut */
};

#define ORC_FP8_BLOCK 128
#define ORC_FP4_BLOCK 16

/* Mean of squares of n values whose sum of squares ss was accumulated in
 * double.  The pages accumulate the squares in fp32 (the AMD kernel's
 * `tl.sum(residual_out * residual_out)`, the var kernel's `tl.sum(x * x)`), so
 * a sum past the fp32 overflow threshold (2^128 - 2^103, where round-to-
 * nearest reaches infinity) is +inf; otherwise it is ss / n rounded once. */
static float mean_of_squares(double ss, double n)
{
    if (ss >= ldexp(2.0 - ldexp(1.0, -24), 127))
        return INFINITY;
    return (float)(ss / n);
}

/* Row-wise evaluation of one AllReduceFusionPattern on the rows listed in
 * rows[0..nrows).  Inputs: R partial tensors and the residual, bf16 [*, H]
 * row-major (stride H); gamma bf16 [H].  Outputs are compact, one row per
 * listed row: allreduce_out / residual_out / norm_out bf16 [nrows, H],
 * partial_norm_out bf16 [nrows, partial_cols], quant_out e4m3 [nrows, H]
 * (patterns 2,4,6,7) or packed e2m1 [nrows, H/2] (3,5), block_scale_out fp32
 * [nrows, H/128] (6,7), sf_out LINEAR e4m3 [nrows, H/16] (3,5).  A NULL
 * output is skipped.  Returns 0, or -1 on an unknown pattern / bad sizes.
 *
 * Steps follow [P2] `amd_allreduce_residual_rmsnorm_kernel`:
 *   reduced  = sum over peers of float32(partial), peers ascending, from 0
 *   x        = reduced + float32(residual)          (stored as residual_out)
 *   variance = sum(x*x) / H
 *   scale    = rsqrt(variance + eps)
 *   norm     = x * scale * weight
 * and [P2] `amd_all_reduce_kernel` for kAllReduce (the sum alone). */
/* The row pipeline shared by the all-reduce and reduce-scatter forms.  The
 * partials are indexed by the listed row; residual and add_in (NULL = none)
 * by the listed row minus local_row0 (0 for the all-reduce form; the first
 * row of the rank's token slice for the reduce-scatter form). */
static int fused_rows_core(int pattern, int R, const uint16_t *const *partials,
                           const uint16_t *add_in, const uint16_t *residual, int64_t local_row0,
                           const uint16_t *gamma, float eps, float scale_factor, int64_t H,
                           int64_t partial_cols, const int64_t *rows, int64_t nrows,
                           uint16_t *allreduce_out, uint16_t *residual_out, uint16_t *norm_out,
                           uint16_t *partial_norm_out, uint8_t *quant_out, float *block_scale_out,
                           uint8_t *sf_out)
{
    if (pattern < 0 || pattern > 8 || R < 1 || H < 1)
        return -1;
    int fp8_tensor = (pattern == ORC_AR_RES_RMS_FP8 || pattern == ORC_AR_RES_RMS_OUT_FP8);
    int fp8_block = (pattern == ORC_AR_RES_RMS_FP8_BLOCK || pattern == ORC_AR_RES_RMS_PART_FP8_BLOCK);
    int fp4 = (pattern == ORC_AR_RES_RMS_FP4 || pattern == ORC_AR_RES_RMS_OUT_FP4);
    int partial = (pattern == ORC_AR_RES_RMS_PART || pattern == ORC_AR_RES_RMS_PART_FP8_BLOCK);
    if (fp8_block && H % ORC_FP8_BLOCK)
        return -1;
    if (fp4 && H % ORC_FP4_BLOCK)
        return -1;
    if (partial && (partial_cols < 1 || partial_cols > H))
        return -1;

    float *x = (float *)malloc(sizeof(float) * (size_t)H);
    float *n = (float *)malloc(sizeof(float) * (size_t)H);
    if (!x || !n) {
        free(x);
        free(n);
        return -1;
    }

    for (int64_t ri = 0; ri < nrows; ++ri) {
        const int64_t row = rows[ri];
        const int64_t in_off = row * H;
        const int64_t loc_off = (row - local_row0) * H;

        /* reduce: fp32 accumulator starting at +0, peers in ascending order */
        for (int64_t j = 0; j < H; ++j) {
            float acc = 0.0f;
            for (int r = 0; r < R; ++r)
                acc = acc + orc_bf16_decode(partials[r][in_off + j]);
            x[j] = acc;
        }
        if (allreduce_out)
            for (int64_t j = 0; j < H; ++j)
                allreduce_out[ri * H + j] = orc_bf16_encode(x[j]);
        if (pattern == ORC_AR)
            continue;

        /* the reduce-scatter "Add" operand, in fp32, before the residual */
        if (add_in)
            for (int64_t j = 0; j < H; ++j)
                x[j] = x[j] + orc_bf16_decode(add_in[loc_off + j]);

        /* residual add, in fp32; residual_out is its bf16 rounding */
        for (int64_t j = 0; j < H; ++j)
            x[j] = x[j] + orc_bf16_decode(residual[loc_off + j]);
        if (residual_out)
            for (int64_t j = 0; j < H; ++j)
                residual_out[ri * H + j] = orc_bf16_encode(x[j]);

        /* mean of squares of the unrounded fp32 x (double accumulation) */
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j)
            ss += (double)x[j] * (double)x[j];
        float variance = mean_of_squares(ss, (double)H);
        float t = variance + eps;
        float scale = (float)(1.0 / sqrt((double)t));

        /* norm = (x * scale) * weight, rounded to bf16; n keeps that value */
        for (int64_t j = 0; j < H; ++j) {
            float y = (x[j] * scale) * orc_bf16_decode(gamma[j]);
            uint16_t b = orc_bf16_encode(y);
            n[j] = orc_bf16_decode(b);
            if (norm_out)
                norm_out[ri * H + j] = b;
            if (partial && partial_norm_out && j < partial_cols)
                partial_norm_out[ri * partial_cols + j] = b;
        }

        if (fp8_tensor && quant_out) {
            for (int64_t j = 0; j < H; ++j)
                quant_out[ri * H + j] = orc_e4m3_encode(n[j] * scale_factor);
        }

        if (fp8_block) {
            const int64_t G = H / ORC_FP8_BLOCK;
            for (int64_t g = 0; g < G; ++g) {
                float amax = 0.0f;
                for (int64_t j = g * ORC_FP8_BLOCK; j < (g + 1) * ORC_FP8_BLOCK; ++j)
                    if (fabsf(n[j]) > amax)
                        amax = fabsf(n[j]);
                float s = amax / 448.0f;
                if (block_scale_out)
                    block_scale_out[ri * G + g] = s;
                if (quant_out)
                    for (int64_t j = g * ORC_FP8_BLOCK; j < (g + 1) * ORC_FP8_BLOCK; ++j)
                        quant_out[ri * H + j] = (s == 0.0f) ? 0 : orc_e4m3_encode(n[j] / s);
            }
        }

        if (fp4) {
            const int64_t G = H / ORC_FP4_BLOCK;
            const float g_scale = scale_factor;
            for (int64_t g = 0; g < G; ++g) {
                float amax = 0.0f;
                for (int64_t j = g * ORC_FP4_BLOCK; j < (g + 1) * ORC_FP4_BLOCK; ++j)
                    if (fabsf(n[j]) > amax)
                        amax = fabsf(n[j]);
                uint8_t sf = orc_e4m3_encode(g_scale * (amax / 6.0f));
                float d = orc_e4m3_decode(sf);
                if (sf_out)
                    sf_out[ri * G + g] = sf;
                float es = (d == 0.0f) ? 0.0f : g_scale / d;
                if (quant_out) {
                    for (int64_t j = g * ORC_FP4_BLOCK; j < (g + 1) * ORC_FP4_BLOCK; j += 2) {
                        uint8_t lo = (d == 0.0f) ? 0 : orc_e2m1_encode(n[j] * es);
                        uint8_t hi = (d == 0.0f) ? 0 : orc_e2m1_encode(n[j + 1] * es);
                        quant_out[ri * (H / 2) + j / 2] = (uint8_t)(lo | (hi << 4));
                    }
                }
            }
        }
    }
    free(x);
    free(n);
    return 0;
}

/* Row-wise evaluation of one AllReduceFusionPattern on the rows listed in
 * rows[0..nrows).  Inputs: R partial tensors and the residual, bf16 [*, H]
 * row-major (stride H); gamma bf16 [H].  Outputs are compact, one row per
 * listed row (see fused_rows_core and the output list above).  Returns 0, or
 * -1 on an unknown pattern / bad sizes. */
int orc_fused_reduce_norm_rows(int pattern, int R, const uint16_t *const *partials,
                               const uint16_t *residual, const uint16_t *gamma, float eps,
                               float scale_factor, int64_t H, int64_t partial_cols,
                               const int64_t *rows, int64_t nrows, uint16_t *allreduce_out,
                               uint16_t *residual_out, uint16_t *norm_out,
                               uint16_t *partial_norm_out, uint8_t *quant_out,
                               float *block_scale_out, uint8_t *sf_out)
{
    return fused_rows_core(pattern, R, partials, NULL, residual, 0, gamma, eps, scale_factor, H,
                           partial_cols, rows, nrows, allreduce_out, residual_out, norm_out,
                           partial_norm_out, quant_out, block_scale_out, sf_out);
}

/* ------------------------------------------------------------------------ */
/* Reduce-scatter fusion restated for one GPU ([P1] `trtllm_reducescatter_  */
/* fusion`, `ReduceScatterFusionPattern`; token split of [P2]               */
/* `rsag_get_token_dist`).                                                  */
/* ------------------------------------------------------------------------ */

/* Token slice of rank `rank` among `world` ranks: T/world tokens each, the
 * first T%world ranks one more, slices in rank order. */
void orc_rs_token_split(int64_t T, int world, int rank, int64_t *start, int64_t *count)
{
    int64_t base = T / world, extra = T % world;
    *count = base + (rank < extra ? 1 : 0);
    *start = rank * base + (rank < extra ? rank : extra);
}

/* Rank `rank`'s output of the reduce-scatter fusion, all R partials local
 * (world size = R).  partials: R bf16 [T, H] (every rank's contribution for
 * all T tokens); add_in and residual: bf16 [count, H] for the rank's slice
 * (add_in only for codes 7 and 8).  ReduceScatterFusionPattern codes:
 *   0 kReduceScatter                          -> all-reduce form 0
 *   1..6 kRSResidualRMSNorm...FP8BlockWise    -> all-reduce forms 1..6
 *   7 kRSAddResidualRMSNormFP8BlockWiseQuant  -> form 6 with add_in
 *   8 kRSAddResidualRMSNorm                   -> form 1 with add_in
 * with x = ((sum of partials) + add_in) + residual, and reducescatter_out =
 * bf16(sum of partials) (before add_in).  Outputs are compact [count, ...]. */
int orc_reducescatter_fused_norm(int rs_pattern, int R, const uint16_t *const *partials, int64_t T,
                                 int rank, const uint16_t *add_in, const uint16_t *residual,
                                 const uint16_t *gamma, float eps, float scale_factor, int64_t H,
                                 uint16_t *reducescatter_out, uint16_t *residual_out,
                                 uint16_t *norm_out, uint8_t *quant_out, float *block_scale_out,
                                 uint8_t *sf_out)
{
    if (rs_pattern < 0 || rs_pattern > 8 || R < 1 || rank < 0 || rank >= R || T < 0)
        return -1;
    const int with_add = (rs_pattern == 7 || rs_pattern == 8);
    const int form = rs_pattern == 7 ? ORC_AR_RES_RMS_FP8_BLOCK : (rs_pattern == 8 ? ORC_AR_RES_RMS : rs_pattern);
    if (with_add && !add_in)
        return -1;
    int64_t start, count;
    orc_rs_token_split(T, R, rank, &start, &count);
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(count > 0 ? count : 1));
    if (!rows)
        return -1;
    for (int64_t i = 0; i < count; ++i)
        rows[i] = start + i;
    int rc = fused_rows_core(form, R, partials, with_add ? add_in : NULL, residual, start, gamma, eps,
                             scale_factor, H, 0, rows, count, reducescatter_out, residual_out,
                             norm_out, NULL, quant_out, block_scale_out, sf_out);
    free(rows);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* MiniMax tensor-parallel QK-RMSNorm ([P3]).                                */
/* ------------------------------------------------------------------------ */

/* For every listed token t and every shard r (shard r's row holds
 * q (Q values) | k (K values) | v at element stride row_stride):
 *   vq_r = mean over j < Q of float32(q)^2     ([P3] `_minimax_qk_var_kernel`)
 *   vk_r = mean over j < K of float32(k)^2
 *   Vq = sum over r ascending of vq_r, fp32    (the all-reduce of the [T,2]
 *   Vk likewise                                 variance, `_all_reduce_variance`)
 *   q_out[t, r*Q + j] = bf16((q * rsqrt(Vq/R + eps)) * wq[r*Q + j])
 *   k_out[t, r*K + j] = bf16((k * rsqrt(Vk/R + eps)) * wk[r*K + j])
 * ([P3] `_minimax_rms_apply_kernel`, `_minimax_qk_norm_tp_eager`).
 * Outputs are compact [nrows, R*Q] and [nrows, R*K].  The shard means are
 * rounded to fp32 as the var kernel stores them; inside one shard the sum of
 * squares is accumulated in double (ideal order).  Returns 0 or -1. */
int orc_qk_norm_sharded_rows(int R, const uint16_t *const *shards, int64_t row_stride, int64_t Q,
                             int64_t K, const uint16_t *wq, const uint16_t *wk, float eps,
                             const int64_t *rows, int64_t nrows, uint16_t *q_out, uint16_t *k_out)
{
    if (R < 1 || Q < 1 || K < 1 || row_stride < Q + K)
        return -1;
    for (int64_t ri = 0; ri < nrows; ++ri) {
        const int64_t t = rows[ri];
        float Vq = 0.0f, Vk = 0.0f;
        for (int r = 0; r < R; ++r) {
            const uint16_t *base = shards[r] + t * row_stride;
            double sq = 0.0, sk = 0.0;
            for (int64_t j = 0; j < Q; ++j) {
                double v = orc_bf16_decode(base[j]);
                sq += v * v;
            }
            for (int64_t j = 0; j < K; ++j) {
                double v = orc_bf16_decode(base[Q + j]);
                sk += v * v;
            }
            float vq = mean_of_squares(sq, (double)Q);
            float vk = mean_of_squares(sk, (double)K);
            Vq = Vq + vq;
            Vk = Vk + vk;
        }
        float iq = (float)(1.0 / sqrt((double)(Vq / (float)R + eps)));
        float ik = (float)(1.0 / sqrt((double)(Vk / (float)R + eps)));
        for (int r = 0; r < R; ++r) {
            const uint16_t *base = shards[r] + t * row_stride;
            for (int64_t j = 0; j < Q; ++j) {
                float y = (orc_bf16_decode(base[j]) * iq) * orc_bf16_decode(wq[r * Q + j]);
                q_out[ri * R * Q + r * Q + j] = orc_bf16_encode(y);
            }
            for (int64_t j = 0; j < K; ++j) {
                float y = (orc_bf16_decode(base[Q + j]) * ik) * orc_bf16_decode(wk[r * K + j]);
                k_out[ri * R * K + r * K + j] = orc_bf16_encode(y);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Single-matrix sharded RMSNorm ([P1] `minimax_allreduce_rms`: all-reduce  */
/* of the per-token variance of a hidden dim split over R ranks, then       */
/* RMSNorm of each rank's slice with its slice of the weight).              */
/* ------------------------------------------------------------------------ */

/* For every listed token t and every shard r (W values at stride row_stride):
 *   v_r = mean over j < W of float32(x_r[t,j])^2   (double sum, rounded once)
 *   V   = sum over r ascending of v_r, fp32
 *   out[t, r*W + j] = bf16((x_r[t,j] * rsqrt(V/R + eps)) * weight[r*W + j])
 * The same steps as the QK norm above, for one segment.  Outputs are
 * compact [nrows, R*W].  Returns 0 or -1. */
int orc_rms_norm_sharded_rows(int R, const uint16_t *const *shards, int64_t row_stride, int64_t W,
                              const uint16_t *weight, float eps, const int64_t *rows, int64_t nrows,
                              uint16_t *out)
{
    if (R < 1 || W < 1 || row_stride < W)
        return -1;
    for (int64_t ri = 0; ri < nrows; ++ri) {
        const int64_t t = rows[ri];
        float V = 0.0f;
        for (int r = 0; r < R; ++r) {
            const uint16_t *base = shards[r] + t * row_stride;
            double s = 0.0;
            for (int64_t j = 0; j < W; ++j) {
                double v = orc_bf16_decode(base[j]);
                s += v * v;
            }
            V = V + mean_of_squares(s, (double)W);
        }
        float inv = (float)(1.0 / sqrt((double)(V / (float)R + eps)));
        for (int r = 0; r < R; ++r) {
            const uint16_t *base = shards[r] + t * row_stride;
            for (int64_t j = 0; j < W; ++j) {
                float y = (orc_bf16_decode(base[j]) * inv) * orc_bf16_decode(weight[r * W + j]);
                out[ri * R * W + r * W + j] = orc_bf16_encode(y);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* All-gather fusion with the dual RMSNorm of MLA segments, restated for one */
/* GPU ([P1] `trtllm_allgather_fusion`, `AllGatherFusionPattern`).          */
/* ------------------------------------------------------------------------ */

/* RMSNorm of one segment of a row: n_j = bf16((v_j * rsqrt(mean(v^2) + eps)) * w_j),
 * mean in double rounded to fp32, rsqrt correctly rounded; nf receives the
 * bf16-rounded values widened back to fp32. */
static void segment_rmsnorm(const uint16_t *v, int64_t width, const uint16_t *w, float eps,
                            uint16_t *out, float *nf)
{
    double ss = 0.0;
    for (int64_t j = 0; j < width; ++j) {
        double d = orc_bf16_decode(v[j]);
        ss += d * d;
    }
    float var = mean_of_squares(ss, (double)width);
    float s = (float)(1.0 / sqrt((double)(var + eps)));
    for (int64_t j = 0; j < width; ++j) {
        uint16_t b = orc_bf16_encode((orc_bf16_decode(v[j]) * s) * orc_bf16_decode(w[j]));
        if (out)
            out[j] = b;
        nf[j] = orc_bf16_decode(b);
    }
}

/* The gathered token rows [T, hidden] are the R ranks' slices in rank order
 * (rank r holds T/R tokens, the first T%R ranks one more: [P2]
 * `rsag_get_token_dist`); inputs[r] is rank r's [count_r, hidden] slice.
 * Each row is x (q_lora_rank columns) | y (kv_lora_rank) | rope (the rest).
 *   pattern 0 kAllGather                       allgather_out only
 *   pattern 1 kAllGatherfusedRMS               + x_norm_out [T, q], y_norm_out [T, kv]
 *   pattern 2 kAllGatherfusedRMSFP8BlockWiseQuant
 *             + y_norm_out, and the x norm as FP8 1x128 blocks: quant_out
 *             e4m3 [T, q], scale_out fp32 [T, q/128] (s = amax/448, code =
 *             e4m3(n/s), 0 for an all-zero block); x_norm_out optional.
 * Each norm is its own RMSNorm over its segment with its gamma and eps.
 * Outputs are compact, one row per listed gathered row.  Returns 0 or -1. */
int orc_allgather_fused_norm_rows(int pattern, int R, const uint16_t *const *inputs, int64_t T,
                                  int64_t hidden, int64_t q, int64_t kv, const uint16_t *x_gamma,
                                  const uint16_t *y_gamma, float x_eps, float y_eps, const int64_t *rows,
                                  int64_t nrows, uint16_t *allgather_out, uint16_t *x_norm_out,
                                  uint16_t *y_norm_out, uint8_t *quant_out, float *scale_out)
{
    if (pattern < 0 || pattern > 2 || R < 1 || q < 1 || kv < 1 || q + kv > hidden)
        return -1;
    if (pattern == 2 && q % ORC_FP8_BLOCK)
        return -1;
    float *nx = (float *)malloc(sizeof(float) * (size_t)q);
    float *ny = (float *)malloc(sizeof(float) * (size_t)kv);
    if (!nx || !ny) {
        free(nx);
        free(ny);
        return -1;
    }
    for (int64_t ri = 0; ri < nrows; ++ri) {
        const int64_t t = rows[ri];
        /* which rank's slice holds gathered row t */
        int rank = 0;
        int64_t start = 0, count = 0;
        for (int r = 0; r < R; ++r) {
            orc_rs_token_split(T, R, r, &start, &count);
            if (t >= start && t < start + count) {
                rank = r;
                break;
            }
        }
        const uint16_t *row = inputs[rank] + (t - start) * hidden;
        if (allgather_out)
            for (int64_t j = 0; j < hidden; ++j)
                allgather_out[ri * hidden + j] = row[j];
        if (pattern == 0)
            continue;
        segment_rmsnorm(row, q, x_gamma, x_eps, x_norm_out ? x_norm_out + ri * q : NULL, nx);
        segment_rmsnorm(row + q, kv, y_gamma, y_eps, y_norm_out ? y_norm_out + ri * kv : NULL, ny);
        if (pattern == 2) {
            const int64_t G = q / ORC_FP8_BLOCK;
            for (int64_t g = 0; g < G; ++g) {
                float amax = 0.0f;
                for (int64_t j = g * ORC_FP8_BLOCK; j < (g + 1) * ORC_FP8_BLOCK; ++j)
                    if (fabsf(nx[j]) > amax)
                        amax = fabsf(nx[j]);
                float xs = amax / 448.0f;
                if (scale_out)
                    scale_out[ri * G + g] = xs;
                if (quant_out)
                    for (int64_t j = g * ORC_FP8_BLOCK; j < (g + 1) * ORC_FP8_BLOCK; ++j)
                        quant_out[ri * q + j] = (xs == 0.0f) ? 0 : orc_e4m3_encode(nx[j] / xs);
            }
        }
    }
    free(nx);
    free(ny);
    return 0;
}

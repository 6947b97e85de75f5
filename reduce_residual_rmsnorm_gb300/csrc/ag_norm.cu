// All-gather fusion with the dual RMSNorm of MLA segments, restated for one
// GPU (tokenspeed trtllm.py `trtllm_allgather_fusion`, `AllGatherFusionPattern`):
// the R ranks' token slices (tokenspeed triton.py `rsag_get_token_dist`: T/R
// tokens each, the first T%R ranks one more) are gathered in rank order, and
// each gathered row x (q_lora_rank) | y (kv_lora_rank) | rope gets
//   x_norm = bf16((x * rsqrt(mean(x^2) + x_eps)) * x_gamma)
//   y_norm = bf16((y * rsqrt(mean(y^2) + y_eps)) * y_gamma)
// and, for kAllGatherfusedRMSFP8BlockWiseQuant, the x norm in FP8 1x128
// blocks (s = amax/448, code = e4m3(n / s), 0 for an all-zero block).
//
// One warp per gathered row (rows are at most 2112 wide: 264 chunks of 8, at
// most 9 per lane), 8 rows per CTA.  The row stays in registers as packed
// bf16; q_lora_rank % 128 == 0 puts the x/y boundary on a half-warp boundary,
// so the 16-lane shuffles of an FP8 block never mix x with y.  The FP8 form of
// a 2112-wide row fits the 64 registers that four CTAs per SM allow.  On the
// R=8, T=65536, 1536 | 512 | 64 workload this single-warp arrangement beat
// the others measured, even while it still spilled 3 registers: 115.0 us
// against 122.2 us with the x norms parked in shared memory for a second
// pass, 123.8 us at 3 CTAs per SM and 133.3 us with two warps per row (it
// now takes 111.2 us, without spilling).  Calls of at most half a wave of
// rows use a second form with one warp per row segment (ag_seg_kernel).
#include "device_util.cuh"
#include "launch.h"

namespace tsfn {

namespace {

constexpr int kRowsPerCta = 8;

// Where gathered row t lives: rank `rank`'s slice, local row `local`.  The
// ranks' row counts come from the host (T < 2^31), and the two divisions by
// them are multiply-highs (int_div.h).
__device__ __forceinline__ const uint16_t *gathered_row(const AGArgs &a, int64_t t)
{
    const uint32_t tu = (uint32_t)t;
    uint32_t rank, local;
    if (tu < a.split) {
        rank = div_by(tu, a.div_hi);
        local = tu - rank * (a.base + 1);
    } else {
        const uint32_t t2 = tu - a.split;
        const uint32_t k = div_by(t2, a.div_lo);
        rank = a.extra + k;
        local = t2 - k * a.base;
    }
    return a.inputs[rank] + (int64_t)local * a.hidden;
}

// The two norms (and the FP8 x blocks) of gathered row t, whose x and y
// chunks lane + 32 i are in v[i] (the rope chunks are not read).
template <int CPL, int PATTERN>
__device__ __forceinline__ void ag_row_norms(const AGArgs &a, int64_t t, int lane, const uint4 (&v)[CPL])
{
    const int qc = a.q >> 3, kc = a.kv >> 3;
    float sx = 0.0f, sy = 0.0f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < qc + kc) {
            const float s = sumsq_bf16x8(v[i], 0.0f);
            if (c < qc)
                sx += s;
            else
                sy += s;
        }
    }
    sx = warp_sum(sx);
    sy = warp_sum(sy);
    const float scx = rsqrtf(__fadd_rn(__fdiv_rn(sx, (float)a.q), a.x_eps));
    const float scy = rsqrtf(__fadd_rn(__fdiv_rn(sy, (float)a.kv), a.y_eps));

#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        const bool is_x = c < qc;
        const bool is_y = !is_x && c < qc + kc;
        float nf[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            nf[e] = 0.0f;
        if (is_x || is_y) {
            float f[8], g[8];
            unpack8(v[i], f);
            const uint16_t *gam = is_x ? a.x_gamma + (int64_t)c * 8 : a.y_gamma + (int64_t)(c - qc) * 8;
            unpack8(ld_keep(gam), g);
            const float sc = is_x ? scx : scy;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                nf[e] = __fmul_rn(__fmul_rn(f[e], sc), g[e]);
            const uint4 nb = pack8(nf);
            unpack8(nb, nf);  // the quantiser reads the bf16-rounded norm
            if (is_x) {
                if (a.x_norm_out != nullptr)
                    st_v4(a.x_norm_out + t * a.q + (int64_t)c * 8, nb);
            } else {
                st_v4(a.y_norm_out + t * a.kv + (int64_t)(c - qc) * 8, nb);
            }
        }
        if (PATTERN == 2 && 32 * i < qc) {
            // 16 lanes = one 128-column block of x; every lane of the warp
            // takes part (x may end half-way through the warp)
            float amax = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                amax = fmaxf(amax, fabsf(nf[e]));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            if (is_x) {
                const float sg = div_const_rn(amax, 448.0f, kRcp448);
                if ((c & 15) == 0)
                    st_f32_wb(a.scale_out + t * (a.q >> 7) + (c >> 4), sg);
                st_v2(a.quant_out + t * a.q + (int64_t)c * 8,
                      sg != 0.0f ? e4m3_block_codes(nf, sg) : make_uint2(0, 0));
            }
        }
    }
}

// At least four 256-thread CTAs (32 warps) per SM: at most 64 registers.
template <int CPL, int PATTERN>
__global__ void __launch_bounds__(kRowsPerCta * 32, 4) ag_norm_kernel(const __grid_constant__ AGArgs a)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kRowsPerCta + warp;
    pdl_wait();
    if (t >= a.T)
        return;

    const int hidden = a.hidden;
    const uint16_t *row = gathered_row(a, t);
    const int nch = hidden >> 3;

    uint4 v[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < nch)
            v[i] = ld_stream(row + (int64_t)c * 8);
    }
    pdl_launch_dependents();
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = lane + 32 * i;
        if (c < nch)
            st_v4(a.allgather_out + t * hidden + (int64_t)c * 8, v[i]);
    }
    if constexpr (PATTERN != 0)
        ag_row_norms<CPL, PATTERN>(a, t, lane, v);
}

// ---------------------------------------------------------------------------
// Segment form, for calls of at most half a wave of the row kernel (16 rows
// per SM): one warp per (gathered row, segment), segment 0 the x columns and segment 1 the
// y and rope columns.  The two norms do not depend on each other, so the two
// warps of a row never wait for one another, and a short call spreads its work
// over twice the warps (R=8, 1536 | 512 | 64: T=1024 3.7 us against 4.5 for
// the bf16 norms, 5.0 against 5.9 with FP8 1x128; T=16 3.1 against 4.3 and
// 4.4 against 5.7).  With more rows than warp slots the row kernel is faster
// (T=4096 bf16 8.6 us against 9.2; T=65536 FP8 109.5 against 125.5: the x
// warps' FP8 epilogue is then covered by half the warps).
// ---------------------------------------------------------------------------

// AHEAD: each chunk's gamma requested one chunk ahead (below).  The FP8 x
// segment of more than 4 chunks per lane then needs the registers of 3 CTAs
// per SM; its plain instance, at 4 CTAs per SM, serves the larger calls.
template <int CPL, int PATTERN, bool AHEAD>
__global__ void __launch_bounds__(kRowsPerCta * 32, (AHEAD && PATTERN == 2 && CPL > 4) ? 3 : 4)
    ag_seg_kernel(const __grid_constant__ AGArgs a)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (kRowsPerCta / 2) + (warp >> 1);
    const int seg = warp & 1;
    pdl_wait();
    if (t >= a.T)
        return;

    const int hidden = a.hidden;
    const uint16_t *row = gathered_row(a, t);
    const int qc = a.q >> 3, kc = a.kv >> 3, nch = hidden >> 3;
    const int c0 = seg ? qc : 0;        // the segment's first chunk
    const int c1 = seg ? nch : qc;      // one past its last chunk
    const int cn = seg ? qc + kc : qc;  // one past its last normalised chunk
    // chunk c sits on lane c % 32, as in the row kernel, so that the per-lane
    // sums and the warp reduction round the same way: a row's bits do not
    // depend on which form computed it
    const int cb = c0 & ~31;

    uint4 v[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = cb + lane + 32 * i;
        if (c >= c0 && c < c1)
            v[i] = ld_stream(row + (int64_t)c * 8);
    }
    pdl_launch_dependents();
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = cb + lane + 32 * i;
        if (c >= c0 && c < c1)
            st_v4(a.allgather_out + t * hidden + (int64_t)c * 8, v[i]);
    }
    if constexpr (PATTERN == 0)
        return;

    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = cb + lane + 32 * i;
        if (c >= c0 && c < cn)
            ss += sumsq_bf16x8(v[i], 0.0f);
    }
    ss = warp_sum(ss);
    const float sc = seg ? rsqrtf(__fadd_rn(__fdiv_rn(ss, (float)a.kv), a.y_eps))
                         : rsqrtf(__fadd_rn(__fdiv_rn(ss, (float)a.q), a.x_eps));
    const uint16_t *gamma = seg ? a.y_gamma : a.x_gamma;  // indexed by chunk c - c0
    uint16_t *norm_out = seg ? a.y_norm_out : a.x_norm_out;
    const int64_t norm_ld = seg ? a.kv : a.q;

    // With AHEAD a chunk's gamma is requested one chunk ahead, before the
    // previous chunk's stores: loads and stores are issued in order, so a
    // load issued in its own iteration starts a full round trip (from DRAM on
    // a cold call) only after the previous chunk is done.
    uint4 gnext = make_uint4(0, 0, 0, 0);
    if (AHEAD && cb + lane >= c0 && cb + lane < cn)
        gnext = ld_keep(gamma + (int64_t)(cb + lane - c0) * 8);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const int c = cb + lane + 32 * i;
        const bool live = c >= c0 && c < cn;
        const uint4 gcur = gnext;
        if (AHEAD && i + 1 < CPL && c + 32 >= c0 && c + 32 < cn)
            gnext = ld_keep(gamma + (int64_t)(c + 32 - c0) * 8);
        float nf[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            nf[e] = 0.0f;
        if (live) {
            float f[8], g[8];
            unpack8(v[i], f);
            unpack8(AHEAD ? gcur : ld_keep(gamma + (int64_t)(c - c0) * 8), g);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                nf[e] = __fmul_rn(__fmul_rn(f[e], sc), g[e]);
            const uint4 nb = pack8(nf);
            if (norm_out != nullptr)
                st_v4(norm_out + t * norm_ld + (int64_t)(c - c0) * 8, nb);
            if (PATTERN == 2 && seg == 0)
                unpack8(nb, nf);  // the quantiser reads the bf16-rounded norm
        }
        if (PATTERN == 2 && seg == 0 && 32 * i < qc) {
            // 16 lanes = one 128-column block of x; every lane of the warp
            // takes part (x may end half-way through the warp)
            float amax = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                amax = fmaxf(amax, fabsf(nf[e]));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            if (live) {
                const float sg = div_const_rn(amax, 448.0f, kRcp448);
                if ((c & 15) == 0)
                    st_f32_wb(a.scale_out + t * (a.q >> 7) + (c >> 4), sg);
                st_v2(a.quant_out + t * a.q + (int64_t)c * 8,
                      sg != 0.0f ? e4m3_block_codes(nf, sg) : make_uint2(0, 0));
            }
        }
    }
}

template <int CPL>
cudaError_t launch_cpl(const AGArgs &a, bool pdl, cudaStream_t s)
{
    const dim3 g((unsigned)((a.T + kRowsPerCta - 1) / kRowsPerCta)), b(kRowsPerCta * 32);
    switch (a.pattern) {
    case 0: return launch_kernel(ag_norm_kernel<CPL, 0>, g, b, 0, s, pdl, a);
    case 1: return launch_kernel(ag_norm_kernel<CPL, 1>, g, b, 0, s, pdl, a);
    default: return launch_kernel(ag_norm_kernel<CPL, 2>, g, b, 0, s, pdl, a);
    }
}

template <int CPL>
cudaError_t launch_seg(const AGArgs &a, bool pdl, cudaStream_t s, int sms)
{
    constexpr int rows = kRowsPerCta / 2;
    const dim3 g((unsigned)((a.T + rows - 1) / rows)), b(kRowsPerCta * 32);
    switch (a.pattern) {
    case 0: return launch_kernel(ag_seg_kernel<CPL, 0, true>, g, b, 0, s, pdl, a);
    case 1: return launch_kernel(ag_seg_kernel<CPL, 1, true>, g, b, 0, s, pdl, a);
    default:
        // an FP8 x segment of more than 6 chunks per lane does not fit the
        // register budget without spilling: one warp per row there
        if constexpr (CPL > 6) {
            return launch_cpl<CPL>(a, pdl, s);
        } else if constexpr (CPL > 4) {
            // The gammas requested ahead need 3 CTAs per SM.  Measured on R=8
            // 1536 | 512 | 64, back-to-back launches: up to 6 rows per SM that
            // instance is faster (T=16 3.60 us against 4.24, T=896 4.07 against
            // 4.70); from 1024 rows on it lost at some T (5.21 against 4.68 at
            // T=1024), so larger calls keep the plain instance.
            if (a.T > 6 * (int64_t)sms)
                return launch_kernel(ag_seg_kernel<CPL, 2, false>, g, b, 0, s, pdl, a);
            return launch_kernel(ag_seg_kernel<CPL, 2, true>, g, b, 0, s, pdl, a);
        } else {
            return launch_kernel(ag_seg_kernel<CPL, 2, true>, g, b, 0, s, pdl, a);
        }
    }
}

}  // namespace

cudaError_t launch_ag(const AGArgs &a, bool pdl, cudaStream_t stream)
{
    const int per_lane = (a.hidden / 8 + 31) / 32;  // 1..9
    const int sms = current_device_sms();
    if (sms > 0 && a.T <= 16 * (int64_t)sms) {
        // at most half a wave of the row kernel (a warp per row, 32 warps per
        // SM): two warps per row, one per segment, still fit one wave
        const int qc = a.q / 8, nch = a.hidden / 8;
        const int qpl = (qc + 31) / 32, ypl = (nch + 31) / 32 - qc / 32;
        const int seg_lane = qpl > ypl ? qpl : ypl;  // chunk slots per lane of the wider segment
        if (seg_lane <= 1) return launch_seg<1>(a, pdl, stream, sms);
        if (seg_lane <= 2) return launch_seg<2>(a, pdl, stream, sms);
        if (seg_lane <= 4) return launch_seg<4>(a, pdl, stream, sms);
        if (seg_lane <= 6) return launch_seg<6>(a, pdl, stream, sms);
        return launch_seg<9>(a, pdl, stream, sms);
    }
    if (per_lane <= 1) return launch_cpl<1>(a, pdl, stream);
    if (per_lane <= 2) return launch_cpl<2>(a, pdl, stream);
    if (per_lane <= 4) return launch_cpl<4>(a, pdl, stream);
    return launch_cpl<9>(a, pdl, stream);
}

}  // namespace tsfn

// Device helpers shared by the kernels: 128-bit global access, bf16 <-> fp32,
// and the FP8 E4M3 / FP4 E2M1 conversions (hardware cvt with round-to-nearest-
// even and saturation to the largest finite value).
#pragma once

#include <cstdint>

namespace tsfn {

// ---------------------------------------------------------------------------
// 128-bit loads / stores
// ---------------------------------------------------------------------------

// Streaming load: data read exactly once (partials, residual, shard rows).
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Read-only, reused across rows (gamma, q/k weights): keep in L1/L2.
__device__ __forceinline__ uint4 ld_keep(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Outputs are stored with the streaming (evict-first) hint: each is written
// once and read by a later kernel, and keeping a step's ~100 MB of dirty
// output lines from crowding L2 measured 3 % faster on the R=8 T=4096 H=7168
// step (92.8 us vs 96.0 us).
__device__ __forceinline__ void st_v4(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void *p, uint2 v)
{
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_u32(void *p, uint32_t v)
{
    asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_u8(void *p, uint32_t v)
{
    asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_f32(void *p, float v)
{
    asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Write-back store, for outputs so narrow per row that neighbouring rows share
// a 32-byte sector (the all-gather's 1x128 block scales, 48 bytes per
// 1536-wide x): the lines stay in L2 until the sector is complete.
__device__ __forceinline__ void st_f32_wb(void *p, float v)
{
    asm volatile("st.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Prefetch `bytes` (a multiple of 16, from a 16-byte aligned address) into L2
// with one bulk request; nothing waits for it.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// bf16 <-> fp32
// ---------------------------------------------------------------------------

// Widen the two bf16 halves of a 32-bit word (exact: bf16 is the high half of
// an fp32 bit pattern).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// acc[i] = RN(acc[i] + element i of the 8 bf16 in v): Blackwell's mixed
// bf16 + fp32 add widens the bf16 operand exactly inside the instruction, so
// this is bit for bit __fadd_rn(acc[i], widened element i) without unpacking.
__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 &v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .b16 lo, hi;\n\t"
            "mov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %0;\n\t"
            "add.rn.f32.bf16 %1, hi, %1;\n\t}"
            : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
            : "r"(w[i]));
}

// s = RN(e * e + s) over the 8 bf16 elements of v in order, each product of
// the exactly widened element with itself (the mixed bf16 fma).
__device__ __forceinline__ float sumsq_bf16x8(const uint4 &v, float s)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .b16 lo, hi;\n\t"
            "mov.b32 {lo, hi}, %1;\n\t"
            "fma.rn.f32.bf16 %0, lo, lo, %0;\n\t"
            "fma.rn.f32.bf16 %0, hi, hi, %0;\n\t}"
            : "+f"(s)
            : "r"(w[i]));
    return s;
}

// Round two fp32 values to bf16 (nearest, ties to even); lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8])
{
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// ---------------------------------------------------------------------------
// FP8 E4M3 and FP4 E2M1
// ---------------------------------------------------------------------------

// Two fp32 -> two E4M3 codes (nearest-even, saturating to +-448); lo in bits 0..7.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four fp32 -> four E4M3 codes in one word, element i in byte i (the two
// 16-bit pairs packed by one move).
__device__ __forceinline__ uint32_t cvt_e4m3x4(float f0, float f1, float f2, float f3)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(f0), "f"(f1), "f"(f2), "f"(f3));
    return r;
}

// Eight fp32 -> eight E4M3 codes, element i in byte i.
__device__ __forceinline__ uint2 cvt_e4m3x8(const float (&f)[8])
{
    return make_uint2(cvt_e4m3x4(f[0], f[1], f[2], f[3]), cvt_e4m3x4(f[4], f[5], f[6], f[7]));
}

// Two fp32 -> two E2M1 codes (nearest-even, saturating to +-6); lo in bits 0..3.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// Eight fp32 -> eight E2M1 codes packed in 32 bits, element i in nibble i
// (four byte-sized pairs packed by one move).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&f)[8])
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
    return r;
}

// One fp32 -> one E4M3 code.
__device__ __forceinline__ uint32_t cvt_e4m3(float v) { return cvt_e4m3x2(v, 0.0f) & 0xFFu; }

// Value of an E4M3 code (FN variant: bias 7; exponent field 0 is subnormal,
// f * 2^-9; 0x7F / 0xFF are NaN), by the hardware conversion to f16 (which
// holds every E4M3 value exactly) and from f16 to fp32.
__device__ __forceinline__ float e4m3_value(uint32_t c)
{
    float v;
    asm("{\n\t.reg .b16 h, lo, hi;\n\t.reg .b32 d;\n\t"
        "cvt.u16.u32 h, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 d, h;\n\t"
        "mov.b32 {lo, hi}, d;\n\t"
        "cvt.f32.f16 %0, lo;\n\t}"
        : "=f"(v)
        : "r"(c & 0xFFu));
    return v;
}

// RN(a / d) for a bf16-valued a >= 0 (a block's amax) and a constant divisor
// d passed with its correctly rounded reciprocal r = RN(1/d), without a
// divide: q0 = RN(a r), corrected once by the fused multiply-add remainder
// RN(q0 d - a) (Markstein's correction, as below).  For d = 448 and d = 6 a
// sweep of every non-negative bf16 value on the GPU checks it against the
// IEEE divide bit for bit; an infinite or NaN a keeps q0 (inf or NaN, as the
// divide).
__device__ __forceinline__ float div_const_rn(float a, float d, float r)
{
    const float q0 = __fmul_rn(a, r);
    const float q = __fmaf_rn(-__fmaf_rn(q0, d, -a), r, q0);
    return a <= 0x1.fffffep127f ? q : q0;
}
constexpr float kRcp448 = 0x1.24924ap-9f;  // RN(1/448)
constexpr float kRcp6 = 0x1.555556p-3f;    // RN(1/6)

// E4M3 codes of the quotients n[i] / s of one FP8 1x128 block, s = amax/448
// (amax the block's largest |n|, s > 0), for bf16-valued n, without a divide
// per element.
//
// Each quotient is q0 = RN(n r) from the correctly rounded reciprocal
// r = RN(1/s), with one remainder correction q = RN(q0 - RN(q0 s - n) r), the
// remainder taken by a fused multiply-add (Markstein's correction, IBM J. Res.
// Develop. 34(1), 1990).  A scale s below 2^-112 is first multiplied, with n,
// by 2^64 (exact: both are powers-of-two shifts), so that 1/s stays finite;
// for s = +inf the remainder term is dropped, leaving q = RN(n * 0) (a signed
// zero, or NaN for an infinite n, as the IEEE quotient).  Over every pair of
// bf16 values n, amax with |n| <= amax this gives the E4M3 code of the
// correctly rounded quotient n / s; the quotient itself can differ from it in
// the last fp32 bit only where n is so small that the code is 0 either way.
// A sweep of the whole domain on the GPU checks the codes against the IEEE
// divide.
__device__ __forceinline__ uint2 e4m3_block_codes(const float (&n)[8], float s)
{
    const float k = s < 0x1p-112f ? 0x1p64f : 1.0f;
    const float sk = __fmul_rn(s, k);
    const float r = __frcp_rn(sk);
    const float sr = sk <= 0x1.fffffep127f ? sk : 0.0f;
    float q[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float nk = __fmul_rn(n[e], k);
        const float q0 = __fmul_rn(nk, r);
        q[e] = __fmaf_rn(-__fmaf_rn(q0, sr, -nk), r, q0);
    }
    return cvt_e4m3x8(q);
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------

// Wait until the grid this launch depends on (the previous kernel in the
// stream, when launched with programmatic stream serialisation) has completed
// and its memory is visible.  A no-op for a normal launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next kernel in the stream start launching (it still waits in
// pdl_wait() for this grid to complete).  A no-op for a normal launch.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace tsfn

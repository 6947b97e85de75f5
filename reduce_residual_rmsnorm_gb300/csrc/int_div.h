// Division of 31-bit numerators by a divisor fixed for a whole launch, as a
// multiply-high and a shift (T. Granlund and P. L. Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, Theorem 4.2 with
// N = 31 numerator bits).
//
// For a divisor 1 <= d <= 2^31 let l = ceil(log2 d) and m = ceil(2^(31+l) / d).
// Then 2^(31+l) <= m*d < 2^(31+l) + d <= 2^(31+l) + 2^l, which the theorem needs
// for floor(n / d) = floor(m*n / 2^(31+l)) to hold for every 0 <= n < 2^31.
// m < 2^32: d > 2^(l-1) gives m <= 2^32 - 1 for l >= 1, and m = 2^31 for
// d = 1.  Since 2n < 2^32, floor(m*n / 2^(31+l)) = umulhi(2n, m) >> l.
//
// The header compiles as plain C++ too, so that a host program checks the
// same functions the kernels call.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define TSFN_HOST_DEVICE __host__ __device__
#else
#define TSFN_HOST_DEVICE
#endif

namespace tsfn {

struct DivMagic {
    uint32_t m;  // ceil(2^(31+l) / d)
    uint32_t l;  // ceil(log2 d)
};

// The multiplier and shift for divisor d, 1 <= d <= 2^31 (d = 0 is taken as 1).
inline DivMagic div_magic(uint32_t d)
{
    if (d <= 1)
        return DivMagic{0x80000000u, 0u};
    const uint32_t l = 32u - (uint32_t)__builtin_clz(d - 1u);
    const uint64_t m = ((uint64_t)1 << (31u + l)) / d + (((uint64_t)1 << (31u + l)) % d != 0 ? 1u : 0u);
    return DivMagic{(uint32_t)m, l};
}

// floor(n / d) for 0 <= n < 2^31.
TSFN_HOST_DEVICE inline uint32_t div_by(uint32_t n, DivMagic d)
{
#if defined(__CUDA_ARCH__)
    return __umulhi(n << 1, d.m) >> d.l;
#else
    return (uint32_t)(((uint64_t)(n << 1) * d.m) >> 32) >> d.l;
#endif
}

}  // namespace tsfn

// Checks tsfn::div_magic / tsfn::div_by (csrc/int_div.h, the row-to-rank
// division of the all-gather kernels) against the hardware division: every
// numerator below 2^16 and around every multiple of the divisor near 2^31, for
// all divisors up to 4096, powers of two and their neighbours, and pseudo-random
// divisors and numerators across the whole 31-bit range.  Prints "ok".
#include <cstdint>
#include <cstdio>

#include "int_div.h"

static int failures = 0;

static void check(uint32_t n, uint32_t d)
{
    const uint32_t q = tsfn::div_by(n, tsfn::div_magic(d));
    if (q != n / d && failures++ < 10)
        std::printf("n=%u d=%u: %u, expected %u\n", n, d, q, n / d);
}

static void around_multiples(uint32_t d)
{
    const uint32_t top = 0x7FFFFFFFu;
    for (uint32_t n = 0; n < 65536u; ++n)
        check(n, d);
    // the last few multiples below 2^31, and the numerators either side
    uint32_t k = top / d;
    for (int i = 0; i < 64 && k > 0; ++i, --k) {
        const uint64_t base = (uint64_t)k * d;
        for (int o = -2; o <= 2; ++o) {
            const int64_t n = (int64_t)base + o;
            if (n >= 0 && n <= top)
                check((uint32_t)n, d);
        }
    }
    check(top, d);
}

int main()
{
    for (uint32_t d = 1; d <= 4096u; ++d)
        around_multiples(d);
    for (int b = 12; b <= 31; ++b) {
        const uint32_t p = 1u << b;
        around_multiples(p - 1u);
        around_multiples(p);
        if (b < 31)
            around_multiples(p + 1u);
    }
    // xorshift32 pseudo-random divisors and numerators
    uint32_t s = 2463534242u;
    auto next = [&s]() { s ^= s << 13; s ^= s >> 17; s ^= s << 5; return s; };
    for (int i = 0; i < 2000; ++i) {
        const uint32_t d = (next() & 0x7FFFFFFFu) >> (next() % 31u);
        if (d == 0)
            continue;
        for (int j = 0; j < 2000; ++j)
            check(next() & 0x7FFFFFFFu, d);
    }
    if (failures) {
        std::printf("%d failures\n", failures);
        return 1;
    }
    std::printf("ok\n");
    return 0;
}

"""Reading the hand-derived fixtures under tests/golden/, and exact rational
arithmetic with explicit nearest-even rounding to check their derivations
(independent of the oracle and of the GPU path)."""
import math
import os
from fractions import Fraction

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_fixture(name: str) -> dict:
    """Sections of ``tests/golden/<name>``: {section: {key: [ints] or int}};
    hex bf16 lists are parsed as ints, single decimal values as ints."""
    out, cur = {}, None
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = out.setdefault(line[1:-1], {})
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            words = val.split()
            if key in ("pattern", "R", "H", "eps"):
                cur[key] = int(words[0])
            else:
                cur[key] = [int(w, 16) for w in words]
    return out


def bf16_value(bits: int) -> Fraction:
    """Exact value of a finite bf16 bit pattern."""
    bits = int(bits)
    sign = -1 if bits & 0x8000 else 1
    e, m = (bits >> 7) & 0xFF, bits & 0x7F
    assert e != 0xFF, "not finite"
    if e == 0:
        return sign * Fraction(m, 128) * Fraction(2) ** -126
    return sign * (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)


def round_bits(x: Fraction, bits: int) -> Fraction:
    """``x`` rounded to ``bits`` significant bits, ties to even (normal range
    only, which every value of the fixtures is in)."""
    if x == 0:
        return x
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    unit = Fraction(2) ** (e - bits + 1)
    q = a / unit
    n = q.numerator // q.denominator
    rest = q - n
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * unit


def f32(x: Fraction) -> Fraction:
    return round_bits(x, 24)


def bf16_bits(x: Fraction) -> int:
    """Bit pattern of ``x`` rounded to bf16 (positive normal values)."""
    r = round_bits(x, 8)
    assert r > 0
    e = 0
    while Fraction(2) ** e > r:
        e -= 1
    while Fraction(2) ** (e + 1) <= r:
        e += 1
    m = (r / Fraction(2) ** e - 1) * 128
    assert m.denominator == 1
    return ((e + 127) << 7) | int(m)


def f32_rsqrt(t: Fraction) -> Fraction:
    """1/sqrt(t) rounded to fp32, from integer square roots bracketing it
    closely enough that both bounds round the same way."""
    num, den = t.numerator, t.denominator
    k = 120
    r = math.isqrt(den * num * 4 ** k)
    lo, hi = Fraction(r, num * 2 ** k), Fraction(r + 1, num * 2 ** k)
    a, b = f32(lo), f32(hi)
    assert a == b, "bracket too wide"
    return a


def e4m3_code(x: Fraction) -> int:
    """E4M3 code of ``x`` rounded to nearest, ties to even (positive normal
    values up to 448)."""
    r = round_bits(x, 4)
    assert Fraction(2) ** -6 <= r <= 448
    e = 0
    while Fraction(2) ** e > r:
        e -= 1
    while Fraction(2) ** (e + 1) <= r:
        e += 1
    m = (r / Fraction(2) ** e - 1) * 8
    assert m.denominator == 1
    return ((e + 7) << 3) | int(m)


def e4m3_code_value(code: int) -> Fraction:
    """Value of a positive normal E4M3 code."""
    e, m = (code >> 3) & 0xF, code & 7
    assert 0 < e and code < 0x7F
    return (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


E2M1_GRID = [Fraction(v) for v in ("0", "0.5", "1", "1.5", "2", "3", "4", "6")]


def e2m1_nibble(x: Fraction) -> int:
    """E2M1 code (0..7) of a non-negative ``x``: the nearest grid value, ties to
    the even code, saturating at 6."""
    best = 0
    for i, v in enumerate(E2M1_GRID):
        d, db = abs(x - v), abs(x - E2M1_GRID[best])
        if d < db or (d == db and i % 2 == 0):
            best = i
    return best

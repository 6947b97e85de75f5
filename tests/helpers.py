"""Small numpy helpers shared by the tests: bf16 bit handling and ulp distances.

These are comparison utilities, not a second implementation of the method.
"""
import numpy as np
import torch


def f32_of_bf16(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 by bit placement (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_of_f64(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 (ties to even) of float64 values, without a float32 detour."""
    x = np.asarray(x, np.float64)
    codes = np.arange(0x7F80, dtype=np.uint32)  # non-negative finite bf16
    vals = f32_of_bf16(codes.astype(np.uint16)).astype(np.float64)
    a = np.abs(x)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    dlo, dhi = np.abs(a - vals[lo]), np.abs(vals[hi] - a)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[hi] % 2 == 0))
    mag = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint16)
    return mag | np.where(np.signbit(x), 0x8000, 0).astype(np.uint16)


def bf16_bits_of_f32(x: np.ndarray) -> np.ndarray:
    """bf16 bits of float32 values via PyTorch's conversion (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def ordered(bits: np.ndarray, width: int = 16) -> np.ndarray:
    """Map sign-magnitude float bit patterns to integers whose difference is
    the distance in ulps (+0 and -0 both map to 0)."""
    b = np.asarray(bits).astype(np.int64)
    sign = 1 << (width - 1)
    return np.where(b & sign, -(b & (sign - 1)), b)


def ulp_diff(a: np.ndarray, b: np.ndarray, width: int = 16) -> np.ndarray:
    return np.abs(ordered(a, width) - ordered(b, width))


def assert_bf16_close(got, want, max_ulp=1, min_exact=0.99, what=""):
    """bf16 outputs: every element within ``max_ulp`` ulps, and at least
    ``min_exact`` of them bit-identical."""
    got = np.asarray(got, np.uint16)
    want = np.asarray(want, np.uint16)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    d = ulp_diff(got, want)
    worst = int(d.max()) if d.size else 0
    exact = float((d == 0).mean()) if d.size else 1.0
    assert worst <= max_ulp, f"{what}: max ulp distance {worst} > {max_ulp}"
    assert exact >= min_exact, f"{what}: only {exact:.6f} bit-identical (< {min_exact})"
    return worst, exact


def codes_close(got, want, step_of, max_step=1, max_frac=1e-4, what=""):
    """Quantised codes: bit-exact except a fraction <= ``max_frac`` that may be
    ``max_step`` code steps away (an fp32 tie flipping a rounding decision).
    ``step_of`` maps codes to ordered integers."""
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    d = np.abs(step_of(got) - step_of(want))
    frac = float((d != 0).mean()) if d.size else 0.0
    assert int(d.max(initial=0)) <= max_step, f"{what}: a code is {int(d.max())} steps off"
    assert frac <= max_frac, f"{what}: {frac:.2e} of codes differ (> {max_frac})"
    return frac


def e4m3_order(c):
    c = np.asarray(c).astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c)


def e2m1_nibbles(packed):
    p = np.asarray(packed, np.uint8)
    return np.stack([p & 0xF, p >> 4], axis=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)


def e2m1_order(c):
    c = np.asarray(c).astype(np.int64)
    return np.where(c & 0x8, -(c & 0x7), c)

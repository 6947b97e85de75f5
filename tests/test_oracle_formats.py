"""Pins for the oracle's number formats and the NVFP4 scale-factor layout.

The oracle's encoders round with a quantum computed per binade.  Each is
checked here against a different construction: PyTorch's own conversions
(bf16, float8_e4m3fn) and a brute-force nearest-value search over every code
of the format, ties going to the even code.
"""
import numpy as np
import pytest
import torch


def _finite_bf16_table():
    codes = np.arange(1 << 16, dtype=np.uint32)
    vals = (codes << 16).view(np.float32)  # a bf16 is the high half of an fp32
    keep = np.isfinite(vals)
    return codes[keep].astype(np.uint16), vals[keep]


def _nearest_ties_even(x, codes, vals):
    """Brute force: nearest representable magnitude, ties to the even code.
    ``codes``/``vals`` list the non-negative codes of a format."""
    order = np.argsort(vals, kind="stable")
    v, c = vals[order].astype(np.float64), codes[order]
    # drop duplicate magnitudes (e.g. none here, but keep it general)
    uniq, first = np.unique(v, return_index=True)
    v, c = uniq, c[first]
    a = np.abs(x.astype(np.float64))
    hi = np.clip(np.searchsorted(v, a, side="left"), 0, len(v) - 1)
    lo = np.clip(hi - 1, 0, len(v) - 1)
    dlo, dhi = np.abs(a - v[lo]), np.abs(v[hi] - a)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (c[hi] % 2 == 0) & (c[lo] % 2 == 1))
    out = np.where(pick_hi, c[hi], c[lo])
    return out


# --------------------------------------------------------------------------
# bf16
# --------------------------------------------------------------------------

def test_bf16_decode_all_codes(orc):
    codes, vals = _finite_bf16_table()
    got = orc.bf16_decode(codes)
    assert np.array_equal(got.view(np.uint32), vals.view(np.uint32))


def _bf16_probe_inputs(rng):
    codes, vals = _finite_bf16_table()
    pos = np.sort(vals[vals > 0])
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)  # exact ties
    rnd = rng.integers(0, 0x7F800000, size=200_000, dtype=np.uint32).view(np.float32)
    edge = np.array([0.0, 1e-45, 1.17549435e-38, 3.3895314e38, 3.3961776e38, 3.4028235e38],
                    np.float32)
    x = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(np.inf)),
                        rnd, edge, vals])
    return np.concatenate([x, -x]).astype(np.float32)


def test_bf16_encode_matches_torch(orc):
    x = _bf16_probe_inputs(np.random.default_rng(1))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.bf16_encode(x)
    assert np.array_equal(got, ref)


def test_bf16_encode_brute_force(orc):
    codes, vals = _finite_bf16_table()
    nonneg = vals >= 0
    x = _bf16_probe_inputs(np.random.default_rng(2))
    x = x[np.abs(x) <= np.float32(3.3895314e38)]  # below the overflow boundary
    want_mag = _nearest_ties_even(x, codes[nonneg], vals[nonneg])
    want = want_mag | np.where(np.signbit(x), 0x8000, 0).astype(np.uint16)
    assert np.array_equal(orc.bf16_encode(x), want.astype(np.uint16))


def test_bf16_overflow_and_signed_zero(orc):
    x = np.array([3.3961776e38, 3.4028235e38, np.inf, -np.inf, -0.0, 0.0], np.float32)
    got = orc.bf16_encode(x)
    assert list(got) == [0x7F80, 0x7F80, 0x7F80, 0xFF80, 0x8000, 0x0000]


# --------------------------------------------------------------------------
# FP8 E4M3 (FN variant)
# --------------------------------------------------------------------------

def _e4m3_table():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    return codes, vals


def test_e4m3_decode_matches_torch(orc):
    codes, vals = _e4m3_table()
    got = orc.e4m3_decode(codes)
    fin = np.isfinite(vals)
    assert np.array_equal(got[fin], vals[fin])
    assert np.isnan(got[~fin]).all() and set(codes[~fin]) == {0x7F, 0xFF}


def test_e4m3_format_facts(orc):
    # max finite 1.75 * 2^8 = 448 at S.1111.110; min subnormal 2^-9; 1.0 = 0.0111.000
    assert orc.e4m3_decode(np.array([0x7E]))[0] == 448.0
    assert orc.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9
    assert orc.e4m3_decode(np.array([0x38]))[0] == 1.0
    assert orc.e4m3_decode(np.array([0x08]))[0] == 2.0 ** -6


def _e4m3_probe(rng):
    codes, vals = _e4m3_table()
    pos = np.sort(vals[np.isfinite(vals) & (vals > 0)])
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)
    _, bvals = _finite_bf16_table()
    b = bvals[np.abs(bvals) < 1e6]
    x = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                        pos, b, b * np.float32(3.0), rng.standard_normal(100_000).astype(np.float32) * 100,
                        np.array([0.0, 2.0 ** -10, 2.0 ** -10 + 2.0 ** -30, 447.9, 448.0, 455.9, 464.0,
                                  1e4, 3e38], np.float32)])
    return np.concatenate([x, -x]).astype(np.float32)


def test_e4m3_encode_brute_force(orc):
    codes, vals = _e4m3_table()
    keep = np.isfinite(vals) & (vals >= 0)
    x = _e4m3_probe(np.random.default_rng(3))
    sat = np.abs(x) >= 448.0
    want_mag = np.where(sat, 0x7E, _nearest_ties_even(np.minimum(np.abs(x), 448.0), codes[keep], vals[keep]))
    want = (want_mag | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)
    assert np.array_equal(orc.e4m3_encode(x), want)


def test_e4m3_encode_matches_torch_in_range(orc):
    x = _e4m3_probe(np.random.default_rng(4))
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(x), ref)


def test_e4m3_saturates(orc):
    x = np.array([448.0, 449.0, 464.0, 1e10, np.inf, -np.inf, -500.0], np.float32)
    assert list(orc.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


# --------------------------------------------------------------------------
# FP4 E2M1
# --------------------------------------------------------------------------

# E2M1 magnitudes by code 0..7 (2 exponent bits, bias 1, 1 fraction bit;
# code 1 is the subnormal 0.5): the OCP Microscaling formats definition.
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float32)


def test_e2m1_decode(orc):
    got = orc.e2m1_decode(np.arange(16))
    assert np.array_equal(got[:8], E2M1)
    assert np.array_equal(got[8:], -E2M1)


def test_e2m1_encode_ties_and_saturation(orc):
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 1e30, np.inf, -0.0, 0.2, 0.26,
                  -0.75, -5.0001], np.float32)
    want = [0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6, 0x7, 0x7, 0x7, 0x7, 0x8, 0x0, 0x1, 0xA, 0xF]
    assert list(orc.e2m1_encode(x)) == want


def test_e2m1_encode_brute_force(orc):
    rng = np.random.default_rng(5)
    mids = ((E2M1[:-1] + E2M1[1:]) / 2).astype(np.float32)
    _, bvals = _finite_bf16_table()
    b = bvals[np.abs(bvals) <= 6.0]
    x = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(9)),
                        E2M1, b, rng.uniform(-6, 6, 100_000).astype(np.float32)])
    x = np.concatenate([x, -x]).astype(np.float32)
    want_mag = _nearest_ties_even(x, np.arange(8, dtype=np.uint8), E2M1)
    want = (want_mag | np.where(np.signbit(x), 0x8, 0)).astype(np.uint8)
    assert np.array_equal(orc.e2m1_encode(x), want)


# --------------------------------------------------------------------------
# SWIZZLED_128x4 scale-factor layout (the pages only name it; these check the
# structure of the 128x4-tile reading, which stays unpinned by the pages)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (128, 4), (130, 9), (257, 320 // 40), (300, 13)])
def test_swizzle_is_injective_into_padded_buffer(orc, rows, cols):
    pr, pc = orc.sf_swizzled_shape(rows, cols)
    assert pr % 128 == 0 and pc % 4 == 0 and pr >= rows and pc >= cols and pr - rows < 128
    offs = np.array([orc.sf_offset_swizzled_128x4(m, k, cols) for m in range(pr) for k in range(pc)])
    assert offs.min() == 0 and offs.max() == pr * pc - 1
    assert len(np.unique(offs)) == pr * pc  # a bijection on the padded grid


def test_swizzle_tile_structure(orc):
    cols = 20  # 5 tiles of 4 columns per 128-row band
    off = lambda m, k: orc.sf_offset_swizzled_128x4(m, k, cols)  # noqa: E731
    assert off(0, 0) == 0
    assert off(0, 3) == 3  # 4 columns of a row are 4 consecutive bytes
    assert off(32, 0) == 4 and off(64, 0) == 8 and off(96, 0) == 12
    assert off(1, 0) == 16 and off(31, 0) == 31 * 16
    assert off(0, 4) == 512  # next tile along the columns
    assert off(128, 0) == 5 * 512  # next 128-row band
    for m in range(128):
        for k in range(4):
            assert off(m, k) // 512 == 0


def test_swizzle_pads_with_zero(orc):
    rng = np.random.default_rng(6)
    lin = rng.integers(1, 256, size=(130, 9), dtype=np.uint8)
    out = orc.sf_swizzle_128x4(lin)
    pr, pc = orc.sf_swizzled_shape(130, 9)
    assert out.size == pr * pc
    seen = np.zeros(out.size, bool)
    for m in range(130):
        for k in range(9):
            o = orc.sf_offset_swizzled_128x4(m, k, 9)
            assert out[o] == lin[m, k]
            seen[o] = True
    assert (out[~seen] == 0).all()


# --------------------------------------------------------------------------
# SWIZZLED_8x4 (named on the pages, never defined: the 8-row x 4-column tile
# reading; its definition stays unpinned by the pages)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (8, 4), (9, 9), (37, 320 // 8), (130, 13)])
def test_swizzle8_is_injective_into_padded_buffer(orc, rows, cols):
    pr, pc = orc.sf_swizzled8_shape(rows, cols)
    assert pr % 8 == 0 and pc % 4 == 0 and pr >= rows and pc >= cols and pr - rows < 8
    offs = np.array([orc.sf_offset_swizzled_8x4(m, k, cols) for m in range(pr) for k in range(pc)])
    assert offs.min() == 0 and offs.max() == pr * pc - 1
    assert len(np.unique(offs)) == pr * pc


def test_swizzle8_tile_structure(orc):
    cols = 12  # 3 tiles of 4 columns per 8-row band
    off = lambda m, k: orc.sf_offset_swizzled_8x4(m, k, cols)  # noqa: E731
    assert [off(0, k) for k in range(4)] == [0, 1, 2, 3]
    assert off(1, 0) == 4 and off(7, 3) == 31
    assert off(0, 4) == 32 and off(0, 8) == 64
    assert off(8, 0) == 3 * 32


def test_swizzle8_pads_with_zero(orc):
    rng = np.random.default_rng(7)
    lin = rng.integers(1, 256, size=(11, 6), dtype=np.uint8)
    out = orc.sf_swizzle_8x4(lin)
    pr, pc = orc.sf_swizzled8_shape(11, 6)
    assert out.size == pr * pc == 16 * 8
    seen = np.zeros(out.size, bool)
    for m in range(11):
        for k in range(6):
            o = orc.sf_offset_swizzled_8x4(m, k, 6)
            assert out[o] == lin[m, k]
            seen[o] = True
    assert (out[~seen] == 0).all()

"""Pins for the oracle of the fused reduce -> residual -> RMSNorm (-> quant) path.

Each check ties the oracle to something other than itself: exact sums,
closed forms (constant rows), a textbook RMSNorm special case, exact-real
brute force on 4x8 inputs, symmetries (negation, power-of-two scaling,
column permutation), and the error bounds of the FP8/FP4 formats.
"""
from fractions import Fraction
from decimal import Decimal, getcontext

import numpy as np
import pytest

from tests.helpers import (assert_bf16_close, bf16_bits_of_f32, bf16_of_f64, e2m1_nibbles,
                           f32_of_bf16)

EPS = float(np.float32(1e-6))


def _rand_inputs(rng, R, T, H, std=1.0):
    parts = [bf16_bits_of_f32(rng.standard_normal((T, H)).astype(np.float32) * std) for _ in range(R)]
    res = bf16_bits_of_f32(rng.standard_normal((T, H)).astype(np.float32))
    gamma = bf16_bits_of_f32(rng.uniform(0.5, 1.5, H).astype(np.float32))
    return parts, res, gamma


# --------------------------------------------------------------------------
# a1-a3: the reduction and the residual add
# --------------------------------------------------------------------------

def test_exact_sums_on_a_dyadic_grid(orc):
    """Values k/16 with |k| <= 16: every partial sum is exact in fp32 and the
    totals stay on the bf16 grid, so allreduce_out/residual_out must equal the
    exact sums.  A dropped, doubled or sign-flipped term fails."""
    rng = np.random.default_rng(10)
    R, T, H = 8, 5, 64
    ints = rng.integers(-16, 17, size=(R + 1, T, H))
    vals = (ints / 16.0).astype(np.float32)
    parts = [bf16_bits_of_f32(v) for v in vals[:R]]
    res = bf16_bits_of_f32(vals[R])
    gamma = bf16_bits_of_f32(np.ones(H, np.float32))
    out = orc.fused_reduce_norm(1, parts, res, gamma)
    want_ar = bf16_bits_of_f32(ints[:R].sum(0) / 16.0)
    want_res = bf16_bits_of_f32(ints.sum(0) / 16.0)
    assert np.array_equal(out["allreduce_out"], want_ar)
    assert np.array_equal(out["residual_out"], want_res)
    out0 = orc.fused_reduce_norm(0, parts)
    assert np.array_equal(out0["allreduce_out"], want_ar)


def test_sum_matches_exact_real_sum(orc):
    """Random N(0,1) inputs: the fp32 running sum rounded to bf16 equals the
    exact sum rounded to bf16 except near a rounding boundary."""
    rng = np.random.default_rng(11)
    parts, res, gamma = _rand_inputs(rng, 8, 64, 256)
    out = orc.fused_reduce_norm(1, parts, res, gamma)
    exact_ar = sum(f32_of_bf16(p).astype(np.float64) for p in parts)  # exact in float64
    exact_res = exact_ar + f32_of_bf16(res)
    assert_bf16_close(out["allreduce_out"], bf16_of_f64(exact_ar), 1, 0.995, "allreduce_out")
    assert_bf16_close(out["residual_out"], bf16_of_f64(exact_res), 1, 0.995, "residual_out")


def test_single_partial_allreduce_is_identity(orc):
    rng = np.random.default_rng(12)
    parts, _, _ = _rand_inputs(rng, 1, 7, 40)
    out = orc.fused_reduce_norm(0, parts)
    assert np.array_equal(out["allreduce_out"], parts[0])


def test_zero_sum_is_positive_zero(orc):
    """The accumulator starts at +0 ([P2] zeros then +=), so a row of -0
    partials reduces to +0."""
    neg0 = np.full((2, 8), 0x8000, np.uint16)
    out = orc.fused_reduce_norm(0, [neg0, neg0])
    assert (out["allreduce_out"] == 0).all()


# --------------------------------------------------------------------------
# a4-a6: the RMSNorm
# --------------------------------------------------------------------------

@pytest.mark.parametrize("c_parts", [(0.5, 0.25, -0.125), (2.0 ** -10, 0.0, 0.0), (-3.0, 1.0, 0.5),
                                     (2.0 ** -12, 2.0 ** -12, 0.0)])
def test_constant_rows_closed_form(orc, c_parts):
    """x == c on a whole row: norm_j = gamma_j * c / sqrt(c^2 + eps).  The small
    values make eps matter (c^2 near eps)."""
    H, T = 512, 3
    rng = np.random.default_rng(13)
    c_res = 0.0625
    parts = [bf16_bits_of_f32(np.full((T, H), c, np.float32)) for c in c_parts]
    res = bf16_bits_of_f32(np.full((T, H), c_res, np.float32))
    gamma = bf16_bits_of_f32(rng.uniform(0.5, 1.5, H).astype(np.float32))
    out = orc.fused_reduce_norm(1, parts, res, gamma)
    c = sum(c_parts) + c_res
    want = bf16_of_f64(f32_of_bf16(gamma).astype(np.float64) * c / np.sqrt(c * c + EPS))
    assert_bf16_close(out["norm_out"], np.broadcast_to(want, (T, H)), 1, 0.99, "constant rows")


def test_single_partial_zero_residual_is_plain_rmsnorm(orc):
    rng = np.random.default_rng(14)
    parts, _, gamma = _rand_inputs(rng, 1, 32, 1024)
    zero = np.zeros((32, 1024), np.uint16)
    out = orc.fused_reduce_norm(1, parts, zero, gamma)
    x = f32_of_bf16(parts[0]).astype(np.float64)
    want = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + EPS) * f32_of_bf16(gamma)
    assert_bf16_close(out["norm_out"], bf16_of_f64(want), 1, 0.99, "plain RMSNorm")
    assert np.array_equal(out["residual_out"], parts[0])


def test_brute_force_exact_reals_4x8(orc):
    """4x8 inputs on a dyadic grid (so x is exact): the norm is compared with
    the exact real value gamma*x/sqrt(mean(x^2)+eps) at 50 digits."""
    getcontext().prec = 50
    rng = np.random.default_rng(15)
    R, T, H = 3, 4, 8
    ints = rng.integers(-64, 65, size=(R + 1, T, H))
    vals = (ints / 32.0).astype(np.float32)
    parts = [bf16_bits_of_f32(v) for v in vals[:R]]
    res = bf16_bits_of_f32(vals[R])
    gamma = bf16_bits_of_f32(rng.uniform(0.5, 1.5, H).astype(np.float32))
    out = orc.fused_reduce_norm(1, parts, res, gamma)
    g = f32_of_bf16(gamma)
    want = np.empty((T, H))
    for t in range(T):
        x = [Fraction(int(ints[:, t, j].sum()), 32) for j in range(H)]
        ms = sum(v * v for v in x) / H + Fraction(EPS)
        inv = Decimal(1) / (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
        for j in range(H):
            want[t, j] = float(Decimal(x[j].numerator) / Decimal(x[j].denominator) * inv
                               * Decimal(float(g[j])))
    assert_bf16_close(out["norm_out"], bf16_of_f64(want), 1, 0.95, "4x8 brute force")


def test_norm_uses_unrounded_x(orc):
    """Reading c2: the RMSNorm reads the fp32 sum x, not the bf16 residual_out.
    With 8 random partials x is rarely a bf16 value; the norm must match the
    exact-real evaluation on the exact sum (rounding x to bf16 first moves
    about a quarter of the outputs by one ulp)."""
    rng = np.random.default_rng(25)
    parts, res, gamma = _rand_inputs(rng, 8, 16, 1024)
    out = orc.fused_reduce_norm(1, parts, res, gamma)
    x = sum(f32_of_bf16(p).astype(np.float64) for p in parts) + f32_of_bf16(res)
    want = x / np.sqrt((x * x).mean(1, keepdims=True) + EPS) * f32_of_bf16(gamma)
    assert_bf16_close(out["norm_out"], bf16_of_f64(want), 1, 0.995, "norm of fp32 x")


def test_power_of_two_scaling_invariance(orc):
    """With eps = 0 the norm is scale-free; scaling every input by 2^k scales
    every fp32 step exactly, so norm and all codes are bit-identical."""
    rng = np.random.default_rng(16)
    parts, res, gamma = _rand_inputs(rng, 4, 8, 256)
    scaled = [bf16_bits_of_f32(f32_of_bf16(p) * np.float32(8.0)) for p in parts]
    res8 = bf16_bits_of_f32(f32_of_bf16(res) * np.float32(8.0))
    for pat, sf in ((1, 0.0), (2, 37.5), (3, 2688.0 / 9.0), (6, 0.0)):
        a = orc.fused_reduce_norm(pat, parts, res, gamma, eps=0.0, scale_factor=sf)
        b = orc.fused_reduce_norm(pat, scaled, res8, gamma, eps=0.0, scale_factor=sf)
        for k in a:
            if k in ("allreduce_out", "residual_out"):
                continue
            assert np.array_equal(a[k], b[k]), (pat, k)


def test_column_permutation_equivariance(orc):
    rng = np.random.default_rng(17)
    parts, res, gamma = _rand_inputs(rng, 3, 6, 384)
    perm = rng.permutation(384)
    a = orc.fused_reduce_norm(1, parts, res, gamma)
    b = orc.fused_reduce_norm(1, [p[:, perm] for p in parts], res[:, perm], gamma[perm])
    assert np.array_equal(a["residual_out"][:, perm], b["residual_out"])
    assert_bf16_close(b["norm_out"], a["norm_out"][:, perm], 1, 0.999, "permuted")


def test_row_selection_matches_full_evaluation(orc):
    rng = np.random.default_rng(18)
    parts, res, gamma = _rand_inputs(rng, 2, 20, 128)
    full = orc.fused_reduce_norm(1, parts, res, gamma)
    rows = np.array([19, 0, 7, 7])
    sub = orc.fused_reduce_norm(1, parts, res, gamma, rows=rows)
    for k in sub:
        assert np.array_equal(sub[k], full[k][rows])


# --------------------------------------------------------------------------
# a7-a10: partial out and the quantisers
# --------------------------------------------------------------------------

def _negated(b):
    return b ^ np.uint16(0x8000)


@pytest.mark.parametrize("pattern,sf", [(1, 0.0), (2, 40.0), (3, 300.0), (4, 40.0), (5, 300.0),
                                        (6, 0.0), (7, 0.0), (8, 0.0)])
def test_negation_symmetry(orc, pattern, sf):
    """Negating every input negates every nonzero output bit for bit (FP8/FP4
    codes flip their sign bit); scales and SFs are unchanged."""
    rng = np.random.default_rng(19)
    parts, res, gamma = _rand_inputs(rng, 4, 6, 256)
    kw = dict(scale_factor=sf, partial_cols=64)
    a = orc.fused_reduce_norm(pattern, parts, res, gamma, **kw)
    b = orc.fused_reduce_norm(pattern, [_negated(p) for p in parts], _negated(res), gamma, **kw)
    zero_n = (a["norm_out"] & 0x7FFF) == 0  # exact zeros stay +0 under negation
    for k in a:
        if k in ("block_scale_out", "sf_out"):
            assert np.array_equal(a[k], b[k]), k
        elif k == "quant_out" and pattern in (3, 5):
            na, nb = e2m1_nibbles(a[k]), e2m1_nibbles(b[k])
            assert np.array_equal((na ^ 0x8)[~zero_n], nb[~zero_n]), k
        elif k == "quant_out":
            assert np.array_equal((a[k] ^ 0x80)[~zero_n], b[k][~zero_n]), k
        else:
            nz = (a[k] & 0x7FFF) != 0
            assert np.array_equal(_negated(a[k][nz]), b[k][nz]), k
            assert np.array_equal(a[k][~nz], b[k][~nz]), k


def test_out_variants_and_partial_out_agree_with_norm(orc):
    rng = np.random.default_rng(20)
    parts, res, gamma = _rand_inputs(rng, 2, 5, 1024)
    base = orc.fused_reduce_norm(1, parts, res, gamma)
    for pat in (2, 3, 4, 5, 6, 7, 8):
        o = orc.fused_reduce_norm(pat, parts, res, gamma, scale_factor=7.0, partial_cols=256)
        assert np.array_equal(o["residual_out"], base["residual_out"])
        assert np.array_equal(o["norm_out"], base["norm_out"])
        if pat in (7, 8):
            assert np.array_equal(o["partial_norm_out"], base["norm_out"][:, :256])
    a = orc.fused_reduce_norm(2, parts, res, gamma, scale_factor=7.0)
    b = orc.fused_reduce_norm(4, parts, res, gamma, scale_factor=7.0)
    assert np.array_equal(a["quant_out"], b["quant_out"])


def _e4m3_values(codes):
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).float().numpy()


def test_fp8_per_tensor_error_bound(orc):
    """code * (1/sigma) reproduces n within E4M3's half-ulp (2^-4 relative in
    the normal range, 2^-10 absolute in the subnormal range); the largest |n|
    maps to +-448 when sigma = 448/amax."""
    rng = np.random.default_rng(21)
    parts, res, gamma = _rand_inputs(rng, 4, 16, 512)
    n = f32_of_bf16(orc.fused_reduce_norm(1, parts, res, gamma)["norm_out"])
    sigma = np.float32(448.0) / np.float32(np.abs(n).max())
    q = orc.fused_reduce_norm(2, parts, res, gamma, scale_factor=float(sigma))["quant_out"]
    v = n.astype(np.float64) * float(sigma)
    dec = _e4m3_values(q).astype(np.float64)
    bound = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
    assert (np.abs(dec - v) <= bound).all()
    imax = np.unravel_index(np.abs(n).argmax(), n.shape)
    assert q[imax] & 0x7F == 0x7E


def test_fp8_per_tensor_saturates(orc):
    rng = np.random.default_rng(22)
    parts, res, gamma = _rand_inputs(rng, 2, 4, 256)
    q = orc.fused_reduce_norm(2, parts, res, gamma, scale_factor=1e6)["quant_out"]
    n = f32_of_bf16(orc.fused_reduce_norm(1, parts, res, gamma)["norm_out"])
    big = np.abs(n) * 1e6 > 448
    assert ((q[big] & 0x7F) == 0x7E).all()


def test_fp8_blockwise_scale_and_bound(orc):
    rng = np.random.default_rng(23)
    parts, res, gamma = _rand_inputs(rng, 4, 8, 1024)
    n = f32_of_bf16(orc.fused_reduce_norm(1, parts, res, gamma)["norm_out"])
    o = orc.fused_reduce_norm(6, parts, res, gamma)
    s, q = o["block_scale_out"], o["quant_out"]
    assert s.shape == (8, 8) and s.dtype == np.float32
    amax = np.abs(n).reshape(8, 8, 128).max(-1)
    assert np.array_equal(s, amax.astype(np.float32) / np.float32(448.0))  # IEEE fp32 divide
    dec = _e4m3_values(q).reshape(8, 8, 128).astype(np.float64) * s[..., None]
    nn = n.reshape(8, 8, 128).astype(np.float64)
    bound = np.maximum(np.abs(nn) * 2.0 ** -4, 2.0 ** -10 * s[..., None]) * (1 + 1e-5)
    assert (np.abs(dec - nn) <= bound).all()
    # the largest |n| of every group encodes to +-448
    qq = q.reshape(8, 8, 128)
    idx = np.abs(nn).argmax(-1)
    assert ((np.take_along_axis(qq, idx[..., None], -1) & 0x7F) == 0x7E).all()


def test_fp8_blockwise_zero_group(orc):
    H = 256
    zero = np.zeros((2, H), np.uint16)
    gamma = bf16_bits_of_f32(np.ones(H, np.float32))
    o = orc.fused_reduce_norm(6, [zero, zero], zero, gamma)
    assert (o["block_scale_out"] == 0).all() and (o["quant_out"] == 0).all()
    assert (o["norm_out"] == 0).all()


def test_fp4_sf_and_bound(orc):
    """NVFP4: SF ~ g*amax/6 within E4M3's half-ulp; decoded codes reproduce n
    within E2M1's half-ulp (0.25 in units of the block scale d/g, relative
    0.25 above 1); the largest |n| of every block encodes to +-6."""
    rng = np.random.default_rng(24)
    T, H = 8, 512
    parts, res, gamma = _rand_inputs(rng, 4, T, H)
    n = f32_of_bf16(orc.fused_reduce_norm(1, parts, res, gamma)["norm_out"])
    g = np.float32(448.0 * 6.0) / np.float32(np.abs(n).max())
    o = orc.fused_reduce_norm(3, parts, res, gamma, scale_factor=float(g))
    sf, q = o["sf_out"], o["quant_out"]
    assert sf.shape == (T, H // 16) and q.shape == (T, H // 2)
    nb = n.reshape(T, H // 16, 16).astype(np.float64)
    amax = np.abs(nb).max(-1)
    d = _e4m3_values(sf).astype(np.float64)
    target = float(g) * amax / 6.0
    assert (np.abs(d - target) <= np.maximum(target * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-5)).all()
    codes = e2m1_nibbles(q).reshape(T, H // 16, 16)
    mag = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])[codes & 7] * np.where(codes & 8, -1, 1)
    unit = d / float(g)  # value of one E2M1 unit in n's scale
    v = nb / unit[..., None]
    err = np.abs(mag - v)
    assert (err <= np.maximum(0.25, np.abs(v) * 0.25) + 1e-6).all()
    idx = np.abs(nb).argmax(-1)
    assert ((np.take_along_axis(codes, idx[..., None], -1) & 7) == 7).all()


def test_fp4_nibble_order(orc):
    """Reading c13: element 2k in the low nibble of byte k."""
    H = 16
    vals = np.zeros((1, H), np.float32)
    vals[0, 0], vals[0, 1] = 6.0, 1.0  # after the norm: amax element first
    parts = [bf16_bits_of_f32(vals)]
    zero = np.zeros((1, H), np.uint16)
    gamma = bf16_bits_of_f32(np.ones(H, np.float32))
    n = f32_of_bf16(orc.fused_reduce_norm(1, parts, zero, gamma)["norm_out"])
    g = np.float32(448.0 * 6.0) / np.float32(np.abs(n).max())
    q = orc.fused_reduce_norm(3, parts, zero, gamma, scale_factor=float(g))["quant_out"]
    assert q[0, 0] & 0xF == 0x7  # element 0 -> 6 in the low nibble
    assert q[0, 0] >> 4 == 0x2   # element 1 -> 1.0 (6 * 1/6) in the high nibble


def test_fp4_zero_block(orc):
    H = 32
    zero = np.zeros((1, H), np.uint16)
    gamma = bf16_bits_of_f32(np.ones(H, np.float32))
    o = orc.fused_reduce_norm(3, [zero], zero, gamma, scale_factor=100.0)
    assert (o["sf_out"] == 0).all() and (o["quant_out"] == 0).all()


def test_rejects_bad_shapes(orc):
    parts = [np.zeros((2, 100), np.uint16)]
    res = np.zeros((2, 100), np.uint16)
    gamma = np.zeros(100, np.uint16)
    with pytest.raises(ValueError):
        orc.fused_reduce_norm(6, parts, res, gamma)  # H % 128 != 0


def test_sum_of_squares_overflow_follows_fp32(orc):
    """Reading c25: the squares are summed in fp32 on the pages, so a row whose
    sum of squares passes fp32's range normalises to +-0; just below the
    range the closed form holds."""
    H = 256
    gamma = bf16_bits_of_f32(np.full(H, 1.25, np.float32))
    zero = np.zeros((1, H), np.uint16)
    # c = 1.5e19: c^2 = 2.25e38 fits in fp32 but the sum of 256 squares does not
    big = bf16_bits_of_f32(np.full((1, H), 1.5e19, np.float32))
    neg = bf16_bits_of_f32(np.full((1, H), -1.5e19, np.float32))
    ok = bf16_bits_of_f32(np.full((1, H), 1e17, np.float32))       # 256e34 < 3.4e38
    assert (orc.fused_reduce_norm(1, [big], zero, gamma)["norm_out"] == 0x0000).all()
    assert (orc.fused_reduce_norm(1, [neg], zero, gamma)["norm_out"] == 0x8000).all()
    c = float(f32_of_bf16(ok)[0, 0])
    want = bf16_of_f64(np.full((1, H), 1.25 * c / np.sqrt(c * c + EPS)))
    assert np.array_equal(orc.fused_reduce_norm(1, [ok], zero, gamma)["norm_out"], want)

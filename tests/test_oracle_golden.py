"""Hand-derived worked examples (tests/golden/rounding_order.txt) in which the
order of the fp32 operations decides an output bit: the peers' partials added
in ascending order from a zero accumulator, and the norm evaluated as
(x * scale) * weight (tokenspeed ops/communication/triton.py,
`amd_allreduce_residual_rmsnorm_kernel`).  Each derivation is re-checked in
exact rational arithmetic, and the other order is checked to give the other
bit, so that the oracle's agreement pins the order itself."""
from fractions import Fraction

import numpy as np

import oracle
from tests.golden_util import (bf16_bits, bf16_value, e2m1_nibble, e4m3_code, e4m3_code_value, f32, f32_rsqrt,
                               read_fixture)

FIX = read_fixture("rounding_order.txt")


def test_sum_order_derivation():
    c = FIX["sum_order"]
    vals = [bf16_value(b) for b in c["partials"]]
    acc = Fraction(0)
    for v in vals:
        acc = f32(acc + v)
    assert bf16_bits(acc) == c["allreduce_out"][0]
    acc = Fraction(0)
    for v in reversed(vals):
        acc = f32(acc + v)
    assert bf16_bits(acc) == c["allreduce_out_if_descending"][0]
    assert c["allreduce_out"] != c["allreduce_out_if_descending"]


def test_sum_order_oracle():
    c = FIX["sum_order"]
    R, H = c["R"], c["H"]
    parts = np.array([np.full((1, H), b, np.uint16) for b in c["partials"]])
    assert parts.shape == (R, 1, H)
    got = oracle.fused_reduce_norm(c["pattern"], parts)
    assert np.array_equal(got["allreduce_out"], np.full((1, H), c["allreduce_out"][0], np.uint16))


def _row(vals, H):
    return np.array([vals[j % len(vals)] for j in range(H)], np.uint16)


def test_mul_order_derivation():
    c = FIX["mul_order"]
    H = c["H"]
    x = [bf16_value(b) for b in _row(c["partial"], H)]
    g = [bf16_value(b) for b in _row(c["gamma"], H)]
    assert all(bf16_value(b) == 0 for b in c["residual"])
    variance = f32(sum(v * v for v in x) / H)
    scale = f32_rsqrt(variance + c["eps"])
    pages = [bf16_bits(f32(f32(x[j] * scale) * g[j])) for j in range(H)]
    other = [bf16_bits(f32(x[j] * f32(scale * g[j]))) for j in range(H)]
    assert pages == list(_row(c["norm_out"], H))
    assert other == list(_row(c["norm_out_if_scale_times_gamma_first"], H))
    assert pages != other


def test_mul_order_oracle():
    c = FIX["mul_order"]
    H = c["H"]
    part = _row(c["partial"], H).reshape(1, 1, H)
    got = oracle.fused_reduce_norm(c["pattern"], part, _row(c["residual"], H).reshape(1, H),
                                   _row(c["gamma"], H), float(c["eps"]))
    assert np.array_equal(got["norm_out"][0], _row(c["norm_out"], H))
    assert np.array_equal(got["residual_out"][0], _row(c["partial"], H))


def _add_order_exact(parts, add_in, residual, residual_first=False):
    s = Fraction(0)
    for v in parts:
        s = f32(s + v)
    if residual_first:
        return s, f32(f32(s + residual) + add_in)
    return s, f32(f32(s + add_in) + residual)


def test_add_order_derivation():
    c = FIX["add_order"]
    parts = [bf16_value(b) for b in c["partials"]]
    a, r = bf16_value(c["add_in"][0]), bf16_value(c["residual"][0])
    s, x = _add_order_exact(parts, a, r)
    assert bf16_bits(s) == c["reducescatter_out"][0]
    assert bf16_bits(x) == c["residual_out"][0]
    _, y = _add_order_exact(parts, a, r, residual_first=True)
    assert bf16_bits(y) == c["residual_out_if_residual_first"][0]
    assert c["residual_out"] != c["residual_out_if_residual_first"]


def test_add_order_oracle():
    c = FIX["add_order"]
    R, H = c["R"], c["H"]
    parts = [np.full((R, H), b, np.uint16) for b in c["partials"]]  # T = R rows, one per rank
    assert len(parts) == R
    gamma = np.full(H, 0x3F80, np.uint16)
    got = oracle.reducescatter_fused_norm(c["pattern"], parts, 0, np.full((1, H), c["add_in"][0], np.uint16),
                                          np.full((1, H), c["residual"][0], np.uint16), gamma)
    assert np.array_equal(got["residual_out"], np.full((1, H), c["residual_out"][0], np.uint16))
    assert np.array_equal(got["reducescatter_out"], np.full((1, H), c["reducescatter_out"][0], np.uint16))


def _shard_rows(c, key, H):
    """R shard rows of one token: shard 0 takes the first value, the others
    the second, in every column."""
    v0, v1 = c[key]
    return [np.full((1, H), v0 if r == 0 else v1, np.uint16) for r in range(c["R"])]


def _shard_exact(c, descending=False):
    R, H = c["R"], c["H"]
    qv = [bf16_value(c["q"][0 if r == 0 else 1]) for r in range(R)]
    means = [f32(H * v * v / H) for v in qv]  # constant rows: the mean of squares is v^2
    V = Fraction(0)
    for m in (reversed(means) if descending else means):
        V = f32(V + m)
    scale = f32_rsqrt(f32(f32(V / R) + c["eps"]))
    w = [bf16_value(c["wq"][0 if r == 0 else 1]) for r in range(R)]
    return [bf16_bits(f32(f32(qv[r] * scale) * w[r])) for r in range(R)]


def test_qk_shard_order_derivation():
    c = FIX["qk_shard_order"]
    want = [c["q_out"][0]] + [c["q_out"][1]] * (c["R"] - 1)
    other = [c["q_out_if_descending"][0]] + [c["q_out_if_descending"][1]] * (c["R"] - 1)
    assert _shard_exact(c) == want
    assert _shard_exact(c, descending=True) == other
    assert want != other


def test_qk_shard_order_oracle():
    c = FIX["qk_shard_order"]
    R, H = c["R"], c["H"]
    q, k = _shard_rows(c, "q", H), _shard_rows(c, "k", H)
    shards = [np.concatenate([q[r], k[r]], axis=1) for r in range(R)]
    wq = np.concatenate([np.full(H, c["wq"][0 if r == 0 else 1], np.uint16) for r in range(R)])
    wk = np.concatenate([np.full(H, c["wk"][0 if r == 0 else 1], np.uint16) for r in range(R)])
    q_out, k_out = oracle.qk_norm_sharded(shards, H, H, wq, wk, float(c["eps"]))
    for r in range(R):
        assert np.all(q_out[0, r * H:(r + 1) * H] == c["q_out"][0 if r == 0 else 1]), r
        assert np.all(k_out[0, r * H:(r + 1) * H] == c["k_out"][0 if r == 0 else 1]), r
    # the single-matrix form on the q columns alone
    out = oracle.rms_norm_sharded(q, H, wq, float(c["eps"]))
    assert np.array_equal(out, q_out)


def fp4_case(name):
    """The fixture's NVFP4 case: (section, exact row values, exact g).  The
    row's squares sum to H, so its norm (scale 1, gamma 1) is the row."""
    c = FIX[name]
    n = [bf16_value(b) for b in c["row"]]
    assert len(n) == c["H"] and sum(v * v for v in n) == c["H"]
    g = Fraction(float(np.array(c["scale_factor_bits"], np.uint32).view(np.float32)[0]))
    return c, n, g


def fp4_block0(n, g, g_times_amax_first=False, n_times_g_first=False):
    """SF code and packed code bytes of the first 16-value block, each product
    rounded to fp32 in the stated order."""
    amax = max(abs(v) for v in n[:16])
    s = f32(f32(g * amax) / 6) if g_times_amax_first else f32(g * f32(amax / 6))
    sf = e4m3_code(s)
    d = e4m3_code_value(sf)
    es = f32(g / d)
    nib = [e2m1_nibble(f32(f32(v * g) / d) if n_times_g_first else f32(v * es)) for v in n[:16]]
    return sf, [nib[2 * k] | (nib[2 * k + 1] << 4) for k in range(8)]


def test_fp4_order_derivations():
    c, n, g = fp4_case("fp4_sf_order")
    assert fp4_block0(n, g) == (c["sf_block0"][0], c["quant_block0"])
    assert fp4_block0(n, g, g_times_amax_first=True)[0] == c["sf_block0_if_g_times_amax_first"][0]
    c, n, g = fp4_case("fp4_element_order")
    assert fp4_block0(n, g) == (c["sf_block0"][0], c["quant_block0"])
    assert fp4_block0(n, g, n_times_g_first=True)[1] == c["quant_block0_if_n_times_g_first"]


def test_fp4_order_oracle():
    for name in ("fp4_sf_order", "fp4_element_order"):
        c, n, g = fp4_case(name)
        H = c["H"]
        part = np.array(c["row"], np.uint16).reshape(1, 1, H)
        got = oracle.fused_reduce_norm(c["pattern"], part, np.zeros((1, H), np.uint16),
                                       np.full(H, 0x3F80, np.uint16), float(c["eps"]), float(g))
        assert np.array_equal(got["residual_out"][0], np.array(c["row"], np.uint16)), name
        assert got["sf_out"][0, 0] == c["sf_block0"][0], name
        assert list(got["quant_out"][0, :8]) == c["quant_block0"], name

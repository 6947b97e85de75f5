"""Pins for the oracle's all-gather fusion with the dual MLA RMSNorm.

The gathered rows are the ranks' slices in rank order; the x and y norms are
two independent RMSNorms over their column segments (each must equal the
single-partial, zero-residual fused oracle on those columns, and a textbook
RMSNorm in double); the FP8 1x128 form quantises the x norm exactly as the
fused oracle's blockwise pattern does; the rope columns only pass through.
"""
import numpy as np
import pytest

from tests.helpers import assert_bf16_close, bf16_bits_of_f32, bf16_of_f64, f32_of_bf16

EPS = float(np.float32(1e-6))


def _inputs(orc, rng, R, T, q, kv, rope, scale=1.0):
    hidden = q + kv + rope
    full = bf16_bits_of_f32(rng.standard_normal((T, hidden)).astype(np.float32) * scale)
    slices = []
    for r in range(R):
        start, count = orc.rs_token_split(T, R, r)
        slices.append(full[start:start + count])
    xg = bf16_bits_of_f32(rng.uniform(0.5, 1.5, q).astype(np.float32))
    yg = bf16_bits_of_f32(rng.uniform(0.5, 1.5, kv).astype(np.float32))
    return full, slices, xg, yg


@pytest.mark.parametrize("R,T", [(8, 64), (3, 10), (4, 2), (1, 5)])
def test_gather_is_rank_order_concatenation(orc, R, T):
    rng = np.random.default_rng(80 + R + T)
    full, slices, xg, yg = _inputs(orc, rng, R, T, 128, 64, 16)
    for pattern in (0, 1, 2):
        o = orc.allgather_fused_norm(pattern, slices, 128, 64, xg, yg)
        assert np.array_equal(o["allgather_out"], full)


def test_segment_norms_equal_the_fused_oracle(orc):
    rng = np.random.default_rng(81)
    R, T, q, kv, rope = 4, 21, 256, 128, 64
    full, slices, xg, yg = _inputs(orc, rng, R, T, q, kv, rope)
    o = orc.allgather_fused_norm(1, slices, q, kv, xg, yg, EPS, 1e-5)
    x, y = np.ascontiguousarray(full[:, :q]), np.ascontiguousarray(full[:, q:q + kv])
    want_x = orc.fused_reduce_norm(1, [x], np.zeros_like(x), xg, EPS)["norm_out"]
    want_y = orc.fused_reduce_norm(1, [y], np.zeros_like(y), yg, 1e-5)["norm_out"]
    assert np.array_equal(o["x_norm_out"], want_x)
    assert np.array_equal(o["y_norm_out"], want_y)


def test_fp8_blockwise_of_x_equals_the_fused_oracle(orc):
    rng = np.random.default_rng(82)
    R, T, q, kv, rope = 8, 40, 1536, 512, 64  # the 2112-wide MLA row
    full, slices, xg, yg = _inputs(orc, rng, R, T, q, kv, rope)
    o = orc.allgather_fused_norm(2, slices, q, kv, xg, yg)
    x = np.ascontiguousarray(full[:, :q])
    want = orc.fused_reduce_norm(6, [x], np.zeros_like(x), xg)
    assert np.array_equal(o["quant_out"], want["quant_out"])
    assert np.array_equal(o["scale_out"], want["block_scale_out"])
    assert np.array_equal(o["x_norm_out"], want["norm_out"])


def test_textbook_norms_and_separate_eps(orc):
    """x with eps = 1.0 (large, so it shows), y with eps = 1e-6."""
    rng = np.random.default_rng(83)
    R, T, q, kv, rope = 2, 9, 128, 64, 8
    full, slices, xg, yg = _inputs(orc, rng, R, T, q, kv, rope, scale=0.5)
    o = orc.allgather_fused_norm(1, slices, q, kv, xg, yg, 1.0, EPS)
    for out, lo, hi, g, eps in ((o["x_norm_out"], 0, q, xg, 1.0), (o["y_norm_out"], q, q + kv, yg, EPS)):
        v = f32_of_bf16(full[:, lo:hi]).astype(np.float64)
        want = v / np.sqrt((v * v).mean(1, keepdims=True) + eps) * f32_of_bf16(g)
        assert_bf16_close(out, bf16_of_f64(want), 1, 0.99, "segment norm")


def test_rope_columns_do_not_enter_the_norms(orc):
    rng = np.random.default_rng(84)
    R, T, q, kv, rope = 2, 6, 128, 64, 64
    full, slices, xg, yg = _inputs(orc, rng, R, T, q, kv, rope)
    a = orc.allgather_fused_norm(1, slices, q, kv, xg, yg)
    other = [s.copy() for s in slices]
    for s in other:
        s[:, q + kv:] = bf16_bits_of_f32(rng.standard_normal((s.shape[0], rope)).astype(np.float32) * 100)
    b = orc.allgather_fused_norm(1, other, q, kv, xg, yg)
    assert np.array_equal(a["x_norm_out"], b["x_norm_out"]) and np.array_equal(a["y_norm_out"], b["y_norm_out"])


def test_rows_selection(orc):
    rng = np.random.default_rng(85)
    full, slices, xg, yg = _inputs(orc, rng, 3, 17, 128, 64, 16)
    a = orc.allgather_fused_norm(2, slices, 128, 64, xg, yg)
    rows = np.array([16, 0, 5, 6, 11])
    b = orc.allgather_fused_norm(2, slices, 128, 64, xg, yg, rows=rows)
    for k in b:
        assert np.array_equal(b[k], a[k][rows])

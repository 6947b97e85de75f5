"""Pins for the oracle's reduce-scatter fusion, restated for one GPU.

Rank w's output is the fused epilogue over its token slice.  With add_in = 0
the slices of all ranks, put back in order, are exactly the all-reduce form
over every token; the slices follow the pages' token split; add_in enters
as one more fp32 term before the residual and is not part of
reducescatter_out.
"""
import numpy as np
import pytest

from tests.helpers import assert_bf16_close, bf16_bits_of_f32, bf16_of_f64, f32_of_bf16

EPS = float(np.float32(1e-6))


def _inputs(rng, R, T, H):
    parts = [bf16_bits_of_f32(rng.standard_normal((T, H)).astype(np.float32)) for _ in range(R)]
    res = bf16_bits_of_f32(rng.standard_normal((T, H)).astype(np.float32))
    gamma = bf16_bits_of_f32(rng.uniform(0.5, 1.5, H).astype(np.float32))
    return parts, res, gamma


@pytest.mark.parametrize("T,W,want", [(10, 3, [(0, 4), (4, 3), (7, 3)]), (2, 4, [(0, 1), (1, 1), (2, 0), (2, 0)]),
                                      (8, 8, [(i, 1) for i in range(8)]), (0, 2, [(0, 0), (0, 0)])])
def test_token_split_follows_the_pages(orc, T, W, want):
    """T//W tokens per rank and one more for the first T%W ranks, in rank order."""
    assert [orc.rs_token_split(T, W, r) for r in range(W)] == want


@pytest.mark.parametrize("rs,ar", [(0, 0), (1, 1), (2, 2), (3, 3), (4, 4), (5, 5), (6, 6)])
def test_slices_reassemble_the_all_reduce_form(orc, rs, ar):
    rng = np.random.default_rng(50 + rs)
    R, T, H = 3, 11, 256
    parts, res, gamma = _inputs(rng, R, T, H)
    sf = 37.0 if ar in (2, 4) else (300.0 if ar in (3, 5) else 0.0)
    full = orc.fused_reduce_norm(ar, parts, res, gamma, EPS, sf)
    for rank in range(R):
        start, count = orc.rs_token_split(T, R, rank)
        o = orc.reducescatter_fused_norm(rs, parts, rank, None, res[start:start + count], gamma, EPS, sf)
        assert np.array_equal(o["reducescatter_out"], full["allreduce_out"][start:start + count])
        for k in ("residual_out", "norm_out", "quant_out", "block_scale_out", "sf_out"):
            if k in o and k in full:
                assert np.array_equal(o[k], full[k][start:start + count]), (rs, k)


@pytest.mark.parametrize("rs,ar", [(8, 1), (7, 6)])
def test_zero_add_in_is_the_plain_form(orc, rs, ar):
    rng = np.random.default_rng(60 + rs)
    R, T, H = 4, 9, 384
    parts, res, gamma = _inputs(rng, R, T, H)
    full = orc.fused_reduce_norm(ar, parts, res, gamma, EPS)
    for rank in range(R):
        start, count = orc.rs_token_split(T, R, rank)
        zero = np.zeros((count, H), np.uint16)
        o = orc.reducescatter_fused_norm(rs, parts, rank, zero, res[start:start + count], gamma, EPS)
        for k in o:
            ref = full["allreduce_out" if k == "reducescatter_out" else k][start:start + count]
            assert np.array_equal(o[k], ref), (rs, k)


def test_add_in_exact_sums(orc):
    """Dyadic values: residual_out = sum + add_in + residual exactly, while
    reducescatter_out is the sum of the partials alone."""
    rng = np.random.default_rng(70)
    R, T, H = 4, 12, 64
    ints = rng.integers(-16, 17, size=(R + 2, T, H))
    vals = (ints / 16.0).astype(np.float32)
    parts = [bf16_bits_of_f32(v) for v in vals[:R]]
    add_full = bf16_bits_of_f32(vals[R])
    res_full = bf16_bits_of_f32(vals[R + 1])
    gamma = bf16_bits_of_f32(np.ones(H, np.float32))
    for rank in range(R):
        start, count = orc.rs_token_split(T, R, rank)
        sl = slice(start, start + count)
        o = orc.reducescatter_fused_norm(8, parts, rank, add_full[sl], res_full[sl], gamma, EPS)
        assert np.array_equal(o["reducescatter_out"], bf16_bits_of_f32(ints[:R, sl].sum(0) / 16.0))
        assert np.array_equal(o["residual_out"], bf16_bits_of_f32(ints[:, sl].sum(0) / 16.0))


def test_add_in_enters_the_norm(orc):
    """The norm is taken over x = sum + add_in + residual: compare with the
    exact-real RMSNorm of that sum."""
    rng = np.random.default_rng(71)
    R, T, H = 2, 8, 512
    parts, res, gamma = _inputs(rng, R, T, H)
    add = bf16_bits_of_f32(rng.standard_normal((T, H)).astype(np.float32) * 2)
    start, count = orc.rs_token_split(T, R, 1)
    sl = slice(start, start + count)
    o = orc.reducescatter_fused_norm(8, parts, 1, add[sl], res[sl], gamma, EPS)
    x = sum(f32_of_bf16(p[sl]).astype(np.float64) for p in parts) + f32_of_bf16(add[sl]) + f32_of_bf16(res[sl])
    want = x / np.sqrt((x * x).mean(1, keepdims=True) + EPS) * f32_of_bf16(gamma)
    assert_bf16_close(o["norm_out"], bf16_of_f64(want), 1, 0.99, "norm with add_in")


def test_rejects_missing_add_in_and_bad_rank(orc):
    rng = np.random.default_rng(72)
    parts, res, gamma = _inputs(rng, 2, 4, 128)
    with pytest.raises(ValueError):
        orc.reducescatter_fused_norm(9, parts, 0, None, res[:2], gamma)
    with pytest.raises(Exception):
        orc.reducescatter_fused_norm(1, parts, 2, None, res[:2], gamma)

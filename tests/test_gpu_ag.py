"""GPU parity of ts_allgather_fused_norm against the CPU oracle, through the C ABI.

Tolerances: allgather_out bit-exact (a copy); x/y norms within 1 bf16 ulp,
>= 99.9 % bit-identical; FP8 codes bit-exact except <= 1 step on <= 1e-4 of
elements, block scales <= 1e-3 differing by <= 2^-7 relative; and exact
self-consistency: the oracle's encoder on the GPU's own x norm reproduces the
GPU's codes and scales bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_gb300 as pkg
from reduce_residual_rmsnorm_gb300 import workloads as wl
from tests.gpu_util import Guarded, host
from tests.helpers import assert_bf16_close, codes_close, e4m3_order, f32_of_bf16

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def _inputs(R, T, q, kv, rope, seed):
    g = torch.Generator().manual_seed(seed)
    full = torch.randn((T, q + kv + rope), generator=g).to(torch.bfloat16)
    slices = [full[s:s + c].clone() for s, c in (pkg.rs_token_split(T, R, r) for r in range(R))]
    xg = (torch.rand(q, generator=g) + 0.5).to(torch.bfloat16)
    yg = (torch.rand(kv, generator=g) + 0.5).to(torch.bfloat16)
    return full, slices, xg, yg


def _run(dev, pattern, slices, q, kv, rope, xg, yg, x_eps=EPS, y_eps=EPS, with_x=True):
    T = sum(s.shape[0] for s in slices)
    hidden = q + kv + rope
    outs = {"allgather_out": Guarded((T, hidden), torch.bfloat16, dev)}
    if pattern in (1, 2):
        if with_x:
            outs["x_norm_out"] = Guarded((T, q), torch.bfloat16, dev)
        outs["y_norm_out"] = Guarded((T, kv), torch.bfloat16, dev)
    if pattern == 2:
        outs["quant_out"] = Guarded((T, q), torch.uint8, dev)
        outs["scale_out"] = Guarded((T, q // 128), torch.float32, dev)
    pkg.ts_allgather_fused_norm(pattern, [s.to(dev) for s in slices], q, kv, rope,
                                None if pattern == 0 else xg.to(dev), None if pattern == 0 else yg.to(dev),
                                x_eps, y_eps, **{k: v.t for k, v in outs.items()})
    torch.cuda.synchronize()
    for k, v in outs.items():
        assert v.intact(), f"write outside {k}"
    return {k: host(v.t) for k, v in outs.items()}


CASES = [  # R, T, q, kv, rope
    (8, 64, 1536, 512, 64),    # the 2112-wide MLA row
    (1, 1, 128, 8, 0),
    (3, 10, 128, 64, 16),
    (4, 2, 256, 128, 64),      # ranks 2 and 3 own no token
    (2, 33, 512, 256, 32),
    (16, 100, 1024, 512, 64),
    (3, 7, 1408, 512, 64),     # x ends mid-warp (176 chunks); the last CTA part empty
    (5, 13, 1024, 8, 0),       # just past 4 chunks per lane
    (2, 5, 384, 1024, 8),      # x ends mid-warp, y wider than x
    # more than 6 and at most 16 rows per SM: one warp per segment, but the
    # wide FP8 x segment without the gammas requested ahead (4 CTAs per SM)
    (8, 2000, 1536, 512, 64),
    # more rows than half a wave (16 per SM): the row kernel instead of one
    # warp per segment
    (8, 2600, 1536, 512, 64),
    (3, 2500, 1408, 512, 64),
    (5, 2500, 384, 1024, 8),
]


@pytest.mark.parametrize("R,T,q,kv,rope", CASES, ids=[f"R{c[0]}-T{c[1]}-q{c[2]}-kv{c[3]}-r{c[4]}" for c in CASES])
@pytest.mark.parametrize("pattern", [0, 1, 2])
def test_small_shapes(dev, pattern, R, T, q, kv, rope):
    full, slices, xg, yg = _inputs(R, T, q, kv, rope, seed=R + T + q + pattern)
    got = _run(dev, pattern, slices, q, kv, rope, xg, yg, EPS, 1e-5)
    want = oracle.allgather_fused_norm(pattern, [wl.bits(s) for s in slices], q, kv, wl.bits(xg), wl.bits(yg),
                                       EPS, 1e-5)
    assert np.array_equal(got["allgather_out"], wl.bits(full))
    assert np.array_equal(got["allgather_out"], want["allgather_out"])
    if pattern == 0:
        return
    assert_bf16_close(got["x_norm_out"], want["x_norm_out"], 1, 0.999, "x_norm")
    assert_bf16_close(got["y_norm_out"], want["y_norm_out"], 1, 0.999, "y_norm")
    if pattern == 2:
        codes_close(got["quant_out"], want["quant_out"], e4m3_order, 1, 1e-4, "x e4m3")
        gs, ws = got["scale_out"], want["scale_out"]
        assert (gs != ws).mean() <= 1e-3 and (np.abs(gs - ws) <= np.abs(ws) * 2.0 ** -7).all()
        # exact self-consistency on the GPU's own x norm
        n = f32_of_bf16(got["x_norm_out"]).reshape(T, q // 128, 128)
        s = np.abs(n).max(-1).astype(np.float32) / np.float32(448.0)
        assert np.array_equal(gs, s)
        with np.errstate(divide="ignore", invalid="ignore"):
            codes = oracle.e4m3_encode((n / s[..., None]).astype(np.float32)).reshape(T, q)
        codes[np.repeat(s == 0, 128, axis=-1).reshape(T, q)] = 0
        assert np.array_equal(got["quant_out"], codes)


def test_fp8_without_x_norm_out(dev):
    full, slices, xg, yg = _inputs(8, 40, 1536, 512, 64, seed=3)
    a = _run(dev, 2, slices, 1536, 512, 64, xg, yg)
    b = _run(dev, 2, slices, 1536, 512, 64, xg, yg, with_x=False)
    for k in ("allgather_out", "y_norm_out", "quant_out", "scale_out"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.slow
def test_fp8_block_scales_across_the_range(dev):
    """x_gamma per 128-column block from 2^-130 to 2^100: block scales that are
    fp32 subnormals, below 2^-112 and large, in one row."""
    full, slices, xg, yg = _inputs(4, 9, 1024, 128, 64, seed=12)
    mult = torch.tensor([2.0 ** -130, 2.0 ** -118, 2.0 ** -112, 1.0, 2.0 ** 40, 2.0 ** 100, 2.0 ** -2, 3.0])
    xg = (xg.float() * mult.repeat_interleave(128)).to(torch.bfloat16)
    got = _run(dev, 2, slices, 1024, 128, 64, xg, yg)
    want = oracle.allgather_fused_norm(2, [wl.bits(s) for s in slices], 1024, 128, wl.bits(xg), wl.bits(yg))
    assert_bf16_close(got["x_norm_out"], want["x_norm_out"], 1, 0.999, "x_norm")
    codes_close(got["quant_out"], want["quant_out"], e4m3_order, 1, 1e-4, "x e4m3")
    n = f32_of_bf16(got["x_norm_out"]).reshape(9, 8, 128)
    s = np.abs(n).max(-1).astype(np.float32) / np.float32(448.0)
    assert np.array_equal(got["scale_out"], s)
    assert (s[:, 0] < 2.0 ** -126).all() and (s[:, 1] < 2.0 ** -112).all()
    with np.errstate(divide="ignore", invalid="ignore"):
        codes = oracle.e4m3_encode((n / s[..., None]).astype(np.float32)).reshape(9, 1024)
    codes[np.repeat(s == 0, 128, axis=-1).reshape(9, 1024)] = 0
    assert np.array_equal(got["quant_out"], codes)


def test_full_size(dev):
    """R=8, T=65536 gathered tokens of 1536 | 512 | 64: sampled rows."""
    full, slices, xg, yg = _inputs(8, 65536, 1536, 512, 64, seed=0)
    got = _run(dev, 2, slices, 1536, 512, 64, xg, yg)
    assert np.array_equal(got["allgather_out"], wl.bits(full))
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(65536 - 16, 65536), rng.integers(0, 65536, 1500)]))
    want = oracle.allgather_fused_norm(2, [wl.bits(s) for s in slices], 1536, 512, wl.bits(xg), wl.bits(yg),
                                       EPS, EPS, rows=rows)
    assert_bf16_close(got["x_norm_out"][rows], want["x_norm_out"], 1, 0.999, "x_norm")
    assert_bf16_close(got["y_norm_out"][rows], want["y_norm_out"], 1, 0.999, "y_norm")
    codes_close(got["quant_out"][rows], want["quant_out"], e4m3_order, 1, 1e-4, "x e4m3")


@pytest.mark.parametrize("q,kv,rope", [(1536, 512, 64), (1408, 512, 64), (384, 1024, 8), (128, 8, 0)])
@pytest.mark.parametrize("pattern", [1, 2])
def test_rows_do_not_depend_on_T(dev, pattern, q, kv, rope):
    """The first 40 and 2000 gathered rows in calls of their own (one warp per
    row segment; for 2000 rows of a wide FP8 x segment the instance without
    the gammas requested ahead) give the same bits as in a call over 5000 rows
    (one warp per row), also where x ends half-way through a warp."""
    R, T = 4, 5000
    full, slices, xg, yg = _inputs(R, T, q, kv, rope, seed=q + kv + pattern)
    big = _run(dev, pattern, slices, q, kv, rope, xg, yg)
    for Ts in (40, 2000):
        small_full = full[:Ts]
        small_slices = [small_full[s0:s0 + c].clone() for s0, c in (pkg.rs_token_split(Ts, R, r) for r in range(R))]
        small = _run(dev, pattern, small_slices, q, kv, rope, xg, yg)
        for k, v in small.items():
            assert np.array_equal(v, big[k][:Ts]), (Ts, k)

"""Seeded random configurations of every entry point against the oracle.

40 draws (TS_FUZZ_SEEDS in the environment sets another count) of (entry
point, pattern, R, T, widths, value scale), each checked
with the same tolerances as the targeted parity tests: sums and copies
bit-exact, bf16 norms within 1 ulp (>= 99.9 % identical), codes and scale
factors within one step on <= 1e-4 of elements (or of the groups, <= 1e-3).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_gb300 as pkg
from reduce_residual_rmsnorm_gb300 import workloads as wl
from tests.gpu_util import host
from tests.helpers import assert_bf16_close, codes_close, e2m1_nibbles, e2m1_order, e4m3_order

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def _draw(seed):
    rng = np.random.default_rng(seed)
    kind = ["fused", "fused", "fused", "rs", "qk", "single", "ag"][rng.integers(0, 7)]
    return rng, kind


def _check_fused_outputs(pattern, got, want):
    assert np.array_equal(got["residual_out"], want["residual_out"])
    if "norm_out" in got:
        assert_bf16_close(got["norm_out"], want["norm_out"], 1, 0.999, "norm")
    if pattern in (2, 4, 6, 7):
        codes_close(got["quant_out"], want["quant_out"], e4m3_order, 1, 1e-4, "e4m3")
    if pattern in (3, 5):
        codes_close(e2m1_nibbles(got["quant_out"]), e2m1_nibbles(want["quant_out"]), e2m1_order, 1, 1e-4, "e2m1")
        codes_close(got["scale_out"], want["sf_out"], e4m3_order, 1, 1e-4, "sf")
    if pattern in (6, 7):
        gs, ws = got["scale_out"], want["block_scale_out"]
        assert (gs != ws).mean() <= 1e-3 and (np.abs(gs - ws) <= np.abs(ws) * 2.0 ** -7).all()


@pytest.mark.parametrize("seed", range(int(os.environ.get("TS_FUZZ_SEEDS", "40"))))
def test_random_configuration(dev, seed):
    rng, kind = _draw(seed)
    scale = float(2.0 ** rng.integers(-8, 9))
    if kind in ("fused", "rs"):
        pattern = int(rng.integers(0, 9))
        form = {7: 6, 8: 1}.get(pattern, pattern) if kind == "rs" else pattern
        quantum = 128 if form in (6, 7) else (16 if form in (3, 5) else 8)
        H = int(quantum * rng.integers(1, 16384 // quantum + 1))
        R = int(rng.integers(1, 17))
        T = int(rng.integers(1, 300))
        inp = wl.fused_inputs(wl.FusedShape(R=R, T=T, H=H, p_std=scale), seed=seed)
        sf = {2: 40.0, 4: 40.0, 3: 300.0, 5: 300.0}.get(form)
        sfv = None if sf is None else torch.tensor([sf], dtype=torch.float32, device=dev)
        P = int(8 * rng.integers(1, H // 8 + 1)) if form in (7, 8) else 0
        if kind == "fused":
            outs = pkg.new_outputs(pattern, T, H, dev, partial_cols=P)
            pkg.ts_fused_reduce_norm(pattern, inp["partials"].to(dev), None if pattern == 0 else inp["residual"].to(dev),
                                     None if pattern == 0 else inp["gamma"].to(dev), EPS, sfv, **outs)
            torch.cuda.synchronize()
            got = {k: host(v) for k, v in outs.items()}
            want = oracle.fused_reduce_norm(pattern, [wl.bits(p) for p in inp["partials"]], wl.bits(inp["residual"]),
                                            wl.bits(inp["gamma"]), EPS, sf or 0.0, P)
            if pattern == 0:
                assert np.array_equal(got["allreduce_out"], want["allreduce_out"])
                return
            if "partial_norm_out" in got:
                assert_bf16_close(got["partial_norm_out"], want["partial_norm_out"], 1, 0.999, "partial")
            _check_fused_outputs(pattern, got, want)
        else:
            rank = int(rng.integers(-1, R))
            start, count = pkg.rs_token_split(T, R, rank)
            add_full = torch.randn((T, H), generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
            add = add_full[start:start + count] if pattern >= 7 else None
            res = inp["residual"][start:start + count]
            outs = pkg.new_outputs(form, count, H, dev)
            kw = {("reducescatter_out" if k == "allreduce_out" else k): v for k, v in outs.items()}
            pkg.ts_reducescatter_fused_norm(pattern, inp["partials"].to(dev), rank,
                                            None if add is None else add.to(dev),
                                            None if form == 0 else res.to(dev),
                                            None if form == 0 else inp["gamma"].to(dev), EPS, sfv, **kw)
            torch.cuda.synchronize()
            got = {k: host(v) for k, v in outs.items()}
            ranks = range(R) if rank < 0 else [rank]
            for r in ranks:
                s0, c0 = pkg.rs_token_split(T, R, r)
                if c0 == 0:
                    continue
                sl = slice(s0 - start, s0 - start + c0)
                want = oracle.reducescatter_fused_norm(
                    pattern, [wl.bits(p) for p in inp["partials"]], r,
                    None if add is None else wl.bits(add_full[s0:s0 + c0]), wl.bits(inp["residual"][s0:s0 + c0]),
                    wl.bits(inp["gamma"]), EPS, sf or 0.0)
                g = {k: v[sl] for k, v in got.items()}
                if form == 0:
                    assert np.array_equal(g["allreduce_out"], want["reducescatter_out"])
                    continue
                _check_fused_outputs(form, g, want)
    elif kind in ("qk", "single"):
        R = int(rng.integers(1, 17))
        T = int(rng.integers(1, 200))
        Q = int(8 * rng.integers(1, 513))
        K = int(8 * rng.integers(1, 129)) if kind == "qk" else 0
        V = int(8 * rng.integers(0, 9))
        g = torch.Generator().manual_seed(seed)
        shards = (torch.randn((R, T, Q + K + V), generator=g) * scale).to(torch.bfloat16)
        wq = (torch.rand(R * Q, generator=g) + 0.5).to(torch.bfloat16)
        if kind == "qk":
            wk = (torch.rand(R * K, generator=g) + 0.5).to(torch.bfloat16)
            q, k = pkg.ts_qk_norm_sharded(shards.to(dev), Q, K, wq.to(dev), wk.to(dev), EPS)
            torch.cuda.synchronize()
            rq, rk = oracle.qk_norm_sharded([wl.bits(s) for s in shards], Q, K, wl.bits(wq), wl.bits(wk), EPS)
            assert_bf16_close(host(q), rq, 1, 0.999, "q")
            assert_bf16_close(host(k), rk, 1, 0.999, "k")
        else:
            out = pkg.ts_rms_norm_sharded(shards.to(dev), Q, wq.to(dev), EPS)
            torch.cuda.synchronize()
            want = oracle.rms_norm_sharded([wl.bits(s) for s in shards], Q, wl.bits(wq), EPS)
            assert_bf16_close(host(out), want, 1, 0.999, "single")
    else:
        R = int(rng.integers(1, 17))
        # short calls run one warp per row segment, calls of more than 16 rows
        # per SM one warp per row: draw both
        T = int(rng.integers(1, 300)) if rng.random() < 0.7 else int(rng.integers(2500, 3200))
        q = int(128 * rng.integers(1, 13))
        kv = int(8 * rng.integers(1, (2112 - q) // 8 + 1))
        rope = int(8 * rng.integers(0, (2112 - q - kv) // 8 + 1))
        pattern = int(rng.integers(0, 3))
        g = torch.Generator().manual_seed(seed)
        full = (torch.randn((T, q + kv + rope), generator=g) * scale).to(torch.bfloat16)
        slices = [full[s0:s0 + c].clone() for s0, c in (pkg.rs_token_split(T, R, r) for r in range(R))]
        xg = (torch.rand(q, generator=g) + 0.5).to(torch.bfloat16)
        yg = (torch.rand(kv, generator=g) + 0.5).to(torch.bfloat16)
        e = lambda *sh, dt=torch.bfloat16: torch.empty(sh, dtype=dt, device=dev)  # noqa: E731
        outs = {"allgather_out": e(T, q + kv + rope)}
        if pattern:
            outs.update(x_norm_out=e(T, q), y_norm_out=e(T, kv))
        if pattern == 2:
            outs.update(quant_out=e(T, q, dt=torch.uint8), scale_out=e(T, q // 128, dt=torch.float32))
        pkg.ts_allgather_fused_norm(pattern, [s.to(dev) for s in slices], q, kv, rope, xg.to(dev), yg.to(dev),
                                    EPS, EPS, **outs)
        torch.cuda.synchronize()
        got = {k: host(v) for k, v in outs.items()}
        want = oracle.allgather_fused_norm(pattern, [wl.bits(s) for s in slices], q, kv, wl.bits(xg), wl.bits(yg),
                                           EPS, EPS)
        assert np.array_equal(got["allgather_out"], want["allgather_out"])
        if pattern:
            assert_bf16_close(got["x_norm_out"], want["x_norm_out"], 1, 0.999, "x")
            assert_bf16_close(got["y_norm_out"], want["y_norm_out"], 1, 0.999, "y")
        if pattern == 2:
            codes_close(got["quant_out"], want["quant_out"], e4m3_order, 1, 1e-4, "x e4m3")

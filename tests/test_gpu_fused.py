"""GPU parity of ts_fused_reduce_norm against the CPU oracle, through the C ABI.

Tolerances (written here, applied to every case):
  * allreduce_out, residual_out: bit-exact (fixed fp32 order, no FMA).
  * norm_out, partial_norm_out: every element within 1 bf16 ulp, >= 99.9 %
    bit-identical (the GPU's fp32 tree sum of x^2 and rsqrtf differ from the
    oracle's double sum and correctly rounded rsqrt by a few fp32 ulps).
  * FP8 / FP4 codes and E4M3 scale factors: bit-exact except where that
    difference flips a rounding decision: at most 1 code step, on at most
    1e-4 of the elements; fp32 block scales likewise within one bf16 ulp of
    amax on at most 1e-3 of the groups.
  * Exact self-consistency: the oracle's encoders applied to the GPU's own
    bf16 norm reproduce the GPU's codes and scales bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_gb300 as pkg
from reduce_residual_rmsnorm_gb300 import workloads as wl
from tests.gpu_util import guarded_outputs, host
from tests.helpers import (assert_bf16_close, codes_close, e2m1_nibbles, e2m1_order, e4m3_order,
                           f32_of_bf16, ulp_diff)

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def _inputs(R, T, H, seed, p_std=1.0, outliers=0.0):
    return wl.fused_inputs(wl.FusedShape(R=R, T=T, H=H, p_std=p_std, outlier_frac=outliers), seed=seed)


LIN, SW128, SW8 = pkg.SFLayout.LINEAR, pkg.SFLayout.SWIZZLED_128x4, pkg.SFLayout.SWIZZLED_8x4


def _swizzle(layout, sf_linear):
    return oracle.sf_swizzle_128x4(sf_linear) if layout == SW128 else oracle.sf_swizzle_8x4(sf_linear)


def _sf_offset(layout, m, k, n_sf):
    if layout == SW128:
        return oracle.sf_offset_swizzled_128x4(m, k, n_sf)
    return oracle.sf_offset_swizzled_8x4(m, k, n_sf)


def _run_gpu(dev, pattern, inp, scale=None, P=0, layout=LIN, allreduce=True, stream=None):
    parts = inp["partials"].to(dev)
    res = inp["residual"].to(dev)
    gamma = inp["gamma"].to(dev)
    T, H = res.shape
    g = guarded_outputs(pattern, T, H, dev, P, int(layout), allreduce)
    sf = None if scale is None else torch.tensor([scale], dtype=torch.float32, device=dev)
    pkg.ts_fused_reduce_norm(pattern, parts, None if pattern == 0 else res, None if pattern == 0 else gamma,
                             EPS, sf, sf_layout=layout, stream=stream, **{k: v.t for k, v in g.items()})
    torch.cuda.synchronize()
    for k, v in g.items():
        assert v.intact(), f"write outside {k}"
    return {k: host(v.t) for k, v in g.items()}


def _oracle(pattern, inp, scale=0.0, P=0, rows=None):
    return oracle.fused_reduce_norm(pattern, [wl.bits(p) for p in inp["partials"]], wl.bits(inp["residual"]),
                                    wl.bits(inp["gamma"]), EPS, scale, P, rows=rows)


def _compare(pattern, got, want, layout=LIN, T=None, rows=None):
    """got: full GPU outputs; want: oracle outputs on ``rows`` (all by default)."""
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    assert np.array_equal(sel(got["allreduce_out"]), want["allreduce_out"]), "allreduce_out"
    if pattern == 0:
        return
    assert np.array_equal(sel(got["residual_out"]), want["residual_out"]), "residual_out"
    if "norm_out" in got:
        assert_bf16_close(sel(got["norm_out"]), want["norm_out"], 1, 0.999, "norm_out")
    if "partial_norm_out" in got:
        assert_bf16_close(sel(got["partial_norm_out"]), want["partial_norm_out"], 1, 0.999, "partial_norm_out")
    if pattern in (2, 4, 6, 7):
        codes_close(sel(got["quant_out"]), want["quant_out"], e4m3_order, 1, 1e-4, "e4m3 codes")
    if pattern in (6, 7):
        gs, ws = sel(got["scale_out"]), want["block_scale_out"]
        diff = gs != ws
        assert diff.mean() <= 1e-3, f"{diff.mean():.2e} of block scales differ"
        assert (np.abs(gs - ws) <= np.abs(ws) * 2.0 ** -7).all()
    if pattern in (3, 5):
        codes_close(e2m1_nibbles(sel(got["quant_out"])), e2m1_nibbles(want["quant_out"]), e2m1_order, 1,
                    1e-4, "e2m1 codes")
        sf = got["scale_out"]
        if layout != LIN:
            lin = np.zeros_like(want["sf_out"])
            full_rows = np.arange(T) if rows is None else rows
            n_sf = want["sf_out"].shape[1]
            flat = sf.reshape(-1)
            for i, m in enumerate(full_rows):
                offs = [_sf_offset(layout, int(m), k, n_sf) for k in range(n_sf)]
                lin[i] = flat[offs]
            codes_close(lin, want["sf_out"], e4m3_order, 1, 1e-4, "SF (swizzled)")
        else:
            codes_close(sel(sf), want["sf_out"], e4m3_order, 1, 1e-4, "SF (linear)")


def _self_consistency(pattern, got, scale):
    """Oracle encoders on the GPU's own n reproduce the GPU's codes exactly."""
    n = f32_of_bf16(got["norm_ref"])
    T, H = n.shape
    if pattern in (2, 4):
        want = oracle.e4m3_encode(n * np.float32(scale))
        assert np.array_equal(got["quant_out"], want)
    elif pattern in (6, 7):
        g = n.reshape(T, H // 128, 128)
        s = np.abs(g).max(-1).astype(np.float32) / np.float32(448.0)
        assert np.array_equal(got["scale_out"], s)
        with np.errstate(divide="ignore", invalid="ignore"):
            q = oracle.e4m3_encode((g / s[..., None]).astype(np.float32)).reshape(T, H)
        q[np.repeat(s == 0, 128, axis=-1).reshape(T, H)] = 0
        assert np.array_equal(got["quant_out"], q)
    elif pattern in (3, 5):
        g = n.reshape(T, H // 16, 16)
        amax = np.abs(g).max(-1).astype(np.float32)
        sf = oracle.e4m3_encode(np.float32(scale) * (amax / np.float32(6.0)))
        d = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))[sf]
        with np.errstate(divide="ignore", invalid="ignore"):
            es = np.where(d == 0, np.float32(0), np.float32(scale) / d).astype(np.float32)
        codes = oracle.e2m1_encode((g * es[..., None]).astype(np.float32)).reshape(T, H)
        codes[np.repeat(d == 0, 16, axis=-1).reshape(T, H)] = 0
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        assert np.array_equal(got["quant_out"], packed)
        return sf
    return None


# ---------------------------------------------------------------------------
# small and ragged shapes: every row through the oracle
# ---------------------------------------------------------------------------

SHAPES = [  # (R, T, H)
    (2, 16, 4096),   # the kARResidualRMSNorm R=2 workload
    (1, 1, 8),
    (3, 5, 136),
    (8, 37, 7168),
    (16, 9, 1024),
    (5, 130, 5120),
    (4, 3, 16384),
    (7, 64, 2112),
    (1, 1300, 1024),  # R = 1 instance; T beyond one wave, so the L2 prefetch runs
    (2, 4300, 2048),  # R = 2 instance past 3.5 R waves of CTAs, so the L2 prefetch runs too
    (16, 5, 16384),   # the widest row with the most partials: 4 chunks per thread
    (8, 4, 16256),    # 4 chunks per thread with a ragged last chunk set (2032 of 2048)
    (3, 37, 1040),    # 65 NVFP4 scale factors per row: byte stores, swizzled padding columns
    (2, 130, 4112),   # 257 per row, 2 chunks per thread, ragged
]


def _ok_for(pattern, H):
    if pattern in (6, 7):
        return H % 128 == 0
    if pattern in (3, 5):
        return H % 16 == 0
    return True


@pytest.mark.parametrize("R,T,H", SHAPES, ids=[f"R{r}-T{t}-H{h}" for r, t, h in SHAPES])
@pytest.mark.parametrize("pattern", list(range(9)))
def test_small_shapes(dev, pattern, R, T, H):
    if not _ok_for(pattern, H):
        pytest.skip("H not a multiple of the quantisation group")
    inp = _inputs(R, T, H, seed=R * 1000 + T + H)
    P = min(H, 1024) // 8 * 8 if pattern in (7, 8) else 0
    base = _run_gpu(dev, 1, inp)
    amax = float(np.abs(f32_of_bf16(base["norm_out"])).max())
    scale = {2: 448.0 / amax, 4: 448.0 / amax, 3: 2688.0 / amax, 5: 2688.0 / amax}.get(pattern)
    for layout in ((LIN, SW128, SW8) if pattern in (3, 5) else (LIN,)):
        got = _run_gpu(dev, pattern, inp, scale, P, layout)
        want = _oracle(pattern, inp, scale or 0.0, P)
        _compare(pattern, got, want, layout, T)
        if pattern in (2, 3, 4, 5, 6, 7):
            got["norm_ref"] = base["norm_out"]
            sf = _self_consistency(pattern, got, scale)
            if layout != LIN:
                assert np.array_equal(got["scale_out"].reshape(-1), _swizzle(layout, sf))


def test_zero_rows(dev):
    """All-zero inputs: norm 0, block scale 0 with codes 0, SF 0 with codes 0."""
    R, T, H = 2, 3, 256
    z = torch.zeros((R, T, H), dtype=torch.bfloat16)
    inp = {"partials": z, "residual": torch.zeros((T, H), dtype=torch.bfloat16),
           "gamma": torch.ones(H, dtype=torch.bfloat16)}
    for pattern, scale in ((1, None), (2, 10.0), (3, 100.0), (6, None), (8, None)):
        got = _run_gpu(dev, pattern, inp, scale, 64 if pattern == 8 else 0)
        _compare(pattern, got, _oracle(pattern, inp, scale or 0.0, 64 if pattern == 8 else 0), T=T)
        for k, v in got.items():
            assert (v == 0).all(), (pattern, k)


def test_negative_zero_partials_reduce_to_positive_zero(dev):
    """Reading c1: the sum starts from a +0 accumulator, so partials that are
    all -0 reduce to +0 (bit pattern 0x0000), and so does x with a -0
    residual; the norm of such a row is +0 times gamma."""
    R, T, H = 3, 4, 256
    negz = torch.full((R, T, H), -0.0, dtype=torch.bfloat16)
    inp = {"partials": negz, "residual": torch.full((T, H), -0.0, dtype=torch.bfloat16),
           "gamma": torch.ones(H, dtype=torch.bfloat16)}
    got = _run_gpu(dev, 1, inp, allreduce=True)
    want = _oracle(1, inp)
    for k in ("allreduce_out", "residual_out", "norm_out"):
        assert np.array_equal(got[k], want[k]), k
        assert (got[k] == 0).all(), k


def test_saturation_and_extremes(dev):
    R, T, H = 4, 8, 512
    inp = _inputs(R, T, H, seed=7, p_std=3.0e4)  # large values: x^2 ~ 1e10 per element
    got = _run_gpu(dev, 2, inp, scale=1.0e4)  # most codes saturate to +-448
    want = _oracle(2, inp, 1.0e4)
    _compare(2, got, want, T=T)
    assert ((got["quant_out"] & 0x7F) == 0x7E).mean() > 0.5
    got = _run_gpu(dev, 3, inp, scale=1.0e6)  # SFs saturate to 448
    _compare(3, got, _oracle(3, inp, 1.0e6), T=T)


@pytest.mark.parametrize("pattern", [6, 7])
def test_fp8_blockwise_block_scales_across_the_range(dev, pattern):
    """gamma per 128-column block from 2^-130 (block scales that are fp32
    subnormals) through 2^-118 (scales below 2^-112) to 2^100, so that blocks
    of one row take every branch of the divide-free block quotient."""
    R, T, H = 3, 11, 1024
    inp = _inputs(R, T, H, seed=11)
    mult = torch.tensor([2.0 ** -130, 2.0 ** -118, 2.0 ** -112, 2.0 ** -100, 1.0, 2.0 ** 40, 2.0 ** 100, 2.0 ** -2])
    inp["gamma"] = (inp["gamma"].float() * mult.repeat_interleave(128)).to(torch.bfloat16)
    P = 256 if pattern == 7 else 0
    base = _run_gpu(dev, 1, inp)
    got = _run_gpu(dev, pattern, inp, None, P)
    _compare(pattern, got, _oracle(pattern, inp, 0.0, P), T=T)
    got["norm_ref"] = base["norm_out"]
    _self_consistency(pattern, got, None)
    s = got["scale_out"]
    assert (s[:, 0] < 2.0 ** -126).all() and (s[:, 1] < 2.0 ** -112).all() and (s[:, 6] > 2.0 ** 90).all()


def test_in_place_allreduce_and_residual(dev):
    R, T, H = 4, 33, 1024
    inp = _inputs(R, T, H, seed=8)
    want = _oracle(1, inp)
    parts = inp["partials"].to(dev).clone()
    res = inp["residual"].to(dev).clone()
    gamma = inp["gamma"].to(dev)
    norm = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    pkg.ts_fused_reduce_norm(1, parts, res, gamma, EPS, allreduce_out=parts[0], residual_out=res, norm_out=norm)
    torch.cuda.synchronize()
    assert np.array_equal(host(parts[0]), want["allreduce_out"])
    assert np.array_equal(host(res), want["residual_out"])
    assert_bf16_close(host(norm), want["norm_out"], 1, 0.999, "in-place norm")
    parts2 = inp["partials"].to(dev).clone()
    pkg.ts_fused_reduce_norm(0, parts2, allreduce_out=parts2[0])
    torch.cuda.synchronize()
    assert np.array_equal(host(parts2[0]), want["allreduce_out"])


@pytest.mark.parametrize("pattern,layout", [(1, LIN), (3, SW128), (6, LIN)])
def test_pinned_host_buffers(dev, pattern, layout):
    """Inputs and outputs in pinned host memory (the kernel reads and writes
    them across the host link): bit-identical to the same call on device
    buffers."""
    R, T, H = 4, 37, 2048
    inp = _inputs(R, T, H, seed=13)
    scale = 300.0 if pattern == 3 else None
    want = _run_gpu(dev, pattern, inp, scale, 0, layout)
    parts = [p.pin_memory() for p in inp["partials"]]
    res, gamma = inp["residual"].pin_memory(), inp["gamma"].pin_memory()
    outs = pkg.new_outputs(pattern, T, H, dev, sf_layout=layout, with_allreduce_out=True)
    outs = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
    sf = None if scale is None else torch.tensor([scale], dtype=torch.float32).pin_memory()
    pkg.ts_fused_reduce_norm(pattern, parts, res, gamma, EPS, sf, sf_layout=layout, **outs)
    torch.cuda.synchronize()
    assert set(outs) == set(want)
    for k, v in outs.items():
        assert np.array_equal(host(v).reshape(-1), want[k].reshape(-1)), k


def test_pinned_host_buffers_sharded_norm(dev):
    qs = wl.QKShape(R=8, T=21, q_shard=256, k_shard=64, v_shard=64)
    qi = wl.qk_inputs(qs, seed=14)
    q_d, k_d = pkg.ts_qk_norm_sharded(qi["shards"].to(dev), 256, 64, qi["q_weight"].to(dev), qi["k_weight"].to(dev),
                                      EPS)
    shards = [s.pin_memory() for s in qi["shards"]]
    q_h, k_h = pkg.ts_qk_norm_sharded(shards, 256, 64, qi["q_weight"].pin_memory(), qi["k_weight"].pin_memory(),
                                      EPS)
    torch.cuda.synchronize()
    assert q_h.device.type == "cpu" and q_h.is_pinned()
    assert np.array_equal(wl.bits(q_h), wl.bits(q_d.cpu())) and np.array_equal(wl.bits(k_h), wl.bits(k_d.cpu()))


def test_side_stream_and_zero_tokens(dev):
    inp = _inputs(2, 16, 4096, seed=9)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = _run_gpu(dev, 1, inp, stream=s)
    _compare(1, got, _oracle(1, inp), T=16)
    empty = torch.empty((2, 0, 4096), dtype=torch.bfloat16, device=dev)
    out = torch.empty((0, 4096), dtype=torch.bfloat16, device=dev)
    pkg.ts_fused_reduce_norm(1, empty, out, torch.ones(4096, dtype=torch.bfloat16, device=dev), EPS,
                             residual_out=torch.empty_like(out), norm_out=torch.empty_like(out))


def test_deterministic(dev):
    inp = _inputs(8, 64, 7168, seed=10)
    a = _run_gpu(dev, 6, inp)
    b = _run_gpu(dev, 6, inp)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


# ---------------------------------------------------------------------------
# full-size workloads: sampled rows through the oracle, exact self-consistency
# on every row
# ---------------------------------------------------------------------------

def _sample_rows(T, n=192, seed=0):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([np.arange(min(32, T)), np.arange(max(0, T - 32), T),
                                     rng.integers(0, T, n)]))
    return rows


@pytest.mark.slow
def test_full_size_allreduce_rmsnorm(dev):
    """kARResidualRMSNorm and kAllReduce, R=8, T=4096, H=7168: every row."""
    inp = wl.fused_inputs(wl.WORKLOADS["C2"], seed=0)
    for pattern in (1, 0):
        got = _run_gpu(dev, pattern, inp, allreduce=True)
        _compare(pattern, got, _oracle(pattern, inp))


@pytest.mark.slow
def test_full_size_in_the_benchmark_configuration(dev):
    """The headline step as bench.py times it: pattern 7 (PartialOut + FP8
    1x128) on R=8, T=8192, H=7168 with outliers, P=1024, launch_with_pdl,
    back-to-back launches on a side stream alternating between two copies of
    the inputs and outputs.  Sampled rows against the oracle, every row
    self-consistent, both copies identical.  Then the same call on pinned host
    inputs and outputs (the end-to-end form): the same bits as on device
    buffers."""
    inp = wl.fused_inputs(wl.WORKLOADS["C3"], seed=0)
    T, H = inp["residual"].shape
    P = 1024
    gamma = inp["gamma"].to(dev)
    sets = [(inp["partials"].to(dev), inp["residual"].to(dev), pkg.new_outputs(7, T, H, dev, partial_cols=P))
            for _ in range(2)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(6):
            parts, res, outs = sets[i % 2]
            pkg.ts_fused_reduce_norm(7, parts, res, gamma, EPS, launch_with_pdl=True, stream=s, **outs)
    torch.cuda.synchronize()
    got = {k: host(v) for k, v in sets[0][2].items()}
    other = {k: host(v) for k, v in sets[1][2].items()}
    for k in got:
        assert np.array_equal(got[k], other[k]), k
    rows = _sample_rows(T)
    _compare_rows(7, got, _oracle(7, inp, 0.0, P, rows=rows), rows)
    base = _run_gpu(dev, 1, inp, allreduce=False)
    assert np.array_equal(got["partial_norm_out"], base["norm_out"][:, :P])
    got["norm_ref"] = base["norm_out"]
    _self_consistency(7, got, None)

    h_outs = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in sets[0][2].items()}
    pkg.ts_fused_reduce_norm(7, inp["partials"].pin_memory(), inp["residual"].pin_memory(),
                             inp["gamma"].pin_memory(), EPS, launch_with_pdl=True, **h_outs)
    torch.cuda.synchronize()
    for k, v in h_outs.items():
        assert np.array_equal(host(v), got[k]), k


@pytest.mark.slow
def test_full_size_in_the_former_benchmark_configuration(dev):
    """kARResidualRMSNorm R=8, T=4096, H=7168, residual_out and norm_out only,
    launch_with_pdl, back-to-back launches on a side stream; every row
    against the oracle."""
    inp = wl.fused_inputs(wl.WORKLOADS["C2"], seed=0)
    T, H = inp["residual"].shape
    parts, res, gamma = inp["partials"].to(dev), inp["residual"].to(dev), inp["gamma"].to(dev)
    ro = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    no = torch.empty_like(ro)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(5):
            pkg.ts_fused_reduce_norm(1, parts, res, gamma, EPS, residual_out=ro, norm_out=no,
                                     launch_with_pdl=True, stream=s)
    torch.cuda.synchronize()
    want = _oracle(1, inp)
    assert np.array_equal(host(ro), want["residual_out"])
    assert_bf16_close(host(no), want["norm_out"], 1, 0.999, "norm_out")


@pytest.mark.slow
def test_full_size_fp8(dev):
    """FP8 per-tensor, FP8 1x128 blockwise, PartialOut (+FP8 blockwise), R=8,
    T=8192, H=7168 with 0.1 % outliers x50."""
    inp = wl.fused_inputs(wl.WORKLOADS["C3"], seed=0)
    base = _run_gpu(dev, 1, inp, allreduce=False)
    amax = float(np.abs(f32_of_bf16(base["norm_out"])).max())
    rows = _sample_rows(8192)
    sigma = float(np.float32(448.0) / np.float32(amax))
    for pattern, scale, P in ((2, sigma, 0), (6, None, 0), (7, None, 1024), (8, None, 1024)):
        got = _run_gpu(dev, pattern, inp, scale, P, allreduce=False)
        want = _oracle(pattern, inp, scale or 0.0, P, rows=rows)
        _compare_rows(pattern, got, want, rows)
        if pattern in (2, 6, 7):
            got["norm_ref"] = base["norm_out"]
            _self_consistency(pattern, got, scale)
        if pattern == 8:
            assert np.array_equal(got["partial_norm_out"], base["norm_out"][:, :1024])


def _compare_rows(pattern, got, want, rows):
    assert np.array_equal(got["residual_out"][rows], want["residual_out"]), "residual_out"
    w = want
    if "partial_norm_out" in got:
        assert_bf16_close(got["partial_norm_out"][rows], want["partial_norm_out"], 1, 0.999, "partial")
    if pattern in (2, 4, 6, 7):
        codes_close(got["quant_out"][rows], w["quant_out"], e4m3_order, 1, 1e-4, "e4m3 codes")
    if pattern in (6, 7):
        gs, ws = got["scale_out"][rows], w["block_scale_out"]
        assert (gs != ws).mean() <= 1e-3
        assert (np.abs(gs - ws) <= np.abs(ws) * 2.0 ** -7).all()


@pytest.mark.slow
def test_full_size_nvfp4(dev):
    """NVFP4, R=4, T=16384, H=5120, SF in LINEAR, SWIZZLED_128x4 and SWIZZLED_8x4."""
    inp = wl.fused_inputs(wl.WORKLOADS["C4"], seed=0)
    base = _run_gpu(dev, 1, inp, allreduce=False)
    amax = float(np.abs(f32_of_bf16(base["norm_out"])).max())
    g = float(np.float32(2688.0) / np.float32(amax))
    rows = _sample_rows(16384)
    want = _oracle(3, inp, g, rows=rows)
    lin = _run_gpu(dev, 3, inp, g, allreduce=False)
    assert np.array_equal(lin["residual_out"][rows], want["residual_out"])
    codes_close(e2m1_nibbles(lin["quant_out"][rows]), e2m1_nibbles(want["quant_out"]), e2m1_order, 1, 1e-4,
                "e2m1")
    codes_close(lin["scale_out"][rows], want["sf_out"], e4m3_order, 1, 1e-4, "SF")
    lin["norm_ref"] = base["norm_out"]
    sf = _self_consistency(3, lin, g)
    for layout in (SW128, SW8):
        swz = _run_gpu(dev, 3, inp, g, layout=layout, allreduce=False)
        assert np.array_equal(swz["quant_out"], lin["quant_out"])
        assert np.array_equal(swz["scale_out"].reshape(-1), _swizzle(layout, sf))


def test_pdl_dependent_chain_matches_plain(dev):
    """Six calls where each reads the previous call's residual_out: with the
    PDL flag every launch must still see its predecessor's writes."""
    inp = _inputs(8, 512, 7168, seed=11)
    parts = inp["partials"].to(dev)
    gamma = inp["gamma"].to(dev)

    def chain(pdl, pattern):
        res = inp["residual"].to(dev).clone()
        outs = []
        for _ in range(6):
            ro = torch.empty_like(res)
            extra = {}
            if pattern == 1:
                extra["norm_out"] = torch.empty_like(res)
            else:
                extra["quant_out"] = torch.empty(res.shape, dtype=torch.uint8, device=dev)
                extra["scale_out"] = torch.empty((res.shape[0], res.shape[1] // 128), dtype=torch.float32,
                                                 device=dev)
            pkg.ts_fused_reduce_norm(pattern, parts, res, gamma, EPS, residual_out=ro, launch_with_pdl=pdl,
                                     **extra)
            res = ro
            outs += list(extra.values())
        torch.cuda.synchronize()
        return [host(o) for o in outs] + [host(res)]

    for pattern in (1, 6):
        for x, y in zip(chain(False, pattern), chain(True, pattern)):
            assert np.array_equal(x, y)


# ---------------------------------------------------------------------------
# reduce-scatter fusion restated for one GPU (every rank's slice)
# ---------------------------------------------------------------------------

INVARIANCE = [(1, 8, 7168), (6, 8, 7168), (3, 4, 5120), (1, 8, 16384), (6, 4, 16384), (3, 2, 12288),
              (7, 3, 9216), (8, 8, 16384)]


@pytest.mark.parametrize("pattern,R,H", INVARIANCE, ids=[f"p{p}-R{r}-H{h}" for p, r, h in INVARIANCE])
def test_rows_do_not_depend_on_T(dev, pattern, R, H):
    """The first 64 rows in a call of their own (one wave of rows: paired
    threads) give the same bits as in a call over 600 rows (the ordinary
    layout of 2 or 4 chunks per thread)."""
    T, Tsmall = 600, 64
    inp = _inputs(R, T, H, seed=pattern + R + H)
    scale = {2: 40.0, 4: 40.0, 3: 300.0, 5: 300.0}.get(pattern)
    P = 1024 if pattern in (7, 8) else 0
    full = _run_gpu(dev, pattern, inp, scale, P)
    small_inp = {"partials": inp["partials"][:, :Tsmall].contiguous(),
                 "residual": inp["residual"][:Tsmall].contiguous(), "gamma": inp["gamma"]}
    small = _run_gpu(dev, pattern, small_inp, scale, P)
    for k, v in small.items():
        assert np.array_equal(v, full[k][:Tsmall]), k


RS_SHAPES = [(4, 37, 1024), (8, 64, 7168), (3, 2, 256), (2, 16, 4096),
             (1, 1300, 1024),   # R = 1 beyond one wave of CTAs: the L2 prefetch of add_in runs
             (3, 300, 9216),    # slices of 100 rows, 4 chunks a row: paired two-chunk threads, add_in
             (4, 600, 16384)]   # slices of 150 rows (at most one wave): the same with 4 partials


@pytest.mark.parametrize("R,T,H", RS_SHAPES, ids=[f"R{r}-T{t}-H{h}" for r, t, h in RS_SHAPES])
@pytest.mark.parametrize("rs", list(range(9)))
def test_reducescatter_every_rank(dev, rs, R, T, H):
    form = {7: 6, 8: 1}.get(rs, rs)
    if not _ok_for(form, H):
        pytest.skip("H not a multiple of the quantisation group")
    inp = _inputs(R, T, H, seed=100 + rs + R + T)
    g = torch.Generator().manual_seed(rs + T)
    add_full = torch.randn((T, H), generator=g).to(torch.bfloat16)
    scale = {2: 40.0, 4: 40.0, 3: 300.0, 5: 300.0}.get(form)
    parts = inp["partials"].to(dev)
    gamma = inp["gamma"].to(dev)
    for rank in range(R):
        start, count = pkg.rs_token_split(T, R, rank)
        res = inp["residual"][start:start + count]
        add = add_full[start:start + count] if rs >= 7 else None
        outs = guarded_outputs(form, count, H, dev, 0, 2, allreduce=True)
        kw = {("reducescatter_out" if k == "allreduce_out" else k): v.t for k, v in outs.items()}
        sf = None if scale is None else torch.tensor([scale], dtype=torch.float32, device=dev)
        pkg.ts_reducescatter_fused_norm(rs, parts, rank, None if add is None else add.to(dev),
                                        None if form == 0 else res.to(dev), None if form == 0 else gamma,
                                        EPS, sf, **kw)
        torch.cuda.synchronize()
        for k, v in outs.items():
            assert v.intact(), f"write outside {k}"
        if count == 0:
            continue
        got = {k: host(v.t) for k, v in outs.items()}
        want = oracle.reducescatter_fused_norm(rs, [wl.bits(p) for p in inp["partials"]], rank,
                                               None if add is None else wl.bits(add), wl.bits(res),
                                               wl.bits(inp["gamma"]), EPS, scale or 0.0)
        want["allreduce_out"] = want.pop("reducescatter_out")
        _compare(form, got, want, LIN, count)


def test_reducescatter_slices_equal_allreduce_rows(dev):
    """With no add_in, the eight rank slices of kRSResidualRMSNorm are the
    kARResidualRMSNorm rows, bit for bit (same kernel arithmetic)."""
    R, T, H = 8, 1000, 7168
    inp = _inputs(R, T, H, seed=12)
    full = _run_gpu(dev, 1, inp)
    parts = inp["partials"].to(dev)
    for rank in range(R):
        start, count = pkg.rs_token_split(T, R, rank)
        ro = torch.empty((count, H), dtype=torch.bfloat16, device=dev)
        no = torch.empty_like(ro)
        rso = torch.empty_like(ro)
        pkg.ts_reducescatter_fused_norm(1, parts, rank, None, inp["residual"][start:start + count].to(dev),
                                        inp["gamma"].to(dev), EPS, reducescatter_out=rso, residual_out=ro,
                                        norm_out=no)
        torch.cuda.synchronize()
        assert np.array_equal(host(rso), full["allreduce_out"][start:start + count])
        assert np.array_equal(host(ro), full["residual_out"][start:start + count])
        assert np.array_equal(host(no), full["norm_out"][start:start + count])


def test_sum_of_squares_overflow(dev):
    """Rows whose fp32 sum of squares overflows normalise to +-0 (as the fp32
    sum on the pages does); a row just below the range keeps its closed form."""
    R, T, H = 2, 4, 7168
    vals = np.zeros((R, T, H), np.float32)
    vals[0, 0] = 1.5e19   # c^2 fits fp32, the sum of 7168 squares does not
    vals[0, 1] = -1.5e19
    vals[0, 2] = 1e17     # sum of squares 7.2e37: finite
    vals[0, 3] = np.random.default_rng(0).standard_normal(H)
    inp = {"partials": torch.from_numpy(vals).to(torch.bfloat16),
           "residual": torch.zeros((T, H), dtype=torch.bfloat16),
           "gamma": torch.full((H,), 1.25, dtype=torch.bfloat16)}
    for pattern in (1, 6):
        got = _run_gpu(dev, pattern, inp)
        want = _oracle(pattern, inp)
        _compare(pattern, got, want, T=T)
        if pattern == 1:
            assert (got["norm_out"][0] == 0x0000).all() and (got["norm_out"][1] == 0x8000).all()


@pytest.mark.parametrize("R,T,H", [(8, 1000, 7168), (2, 8600, 1024), (3, 450, 9216), (4, 600, 16384)])
def test_reducescatter_all_ranks_in_one_launch(dev, R, T, H):
    """rank = -1: every rank's slice in one launch equals the per-rank calls
    (with R = 2 over 8600 rows the one launch prefetches into L2, the per-rank
    calls of 4300 rows do not; with 3 or 4 partials and 4 chunks a row the
    per-rank calls of at most one wave of rows run paired two-chunk threads
    that take add_in one chunk at a time, the one launch the unpaired four-chunk
    layout)."""
    inp = _inputs(R, T, H, seed=13)
    g = torch.Generator().manual_seed(5)
    add = torch.randn((T, H), generator=g).to(torch.bfloat16).to(dev)
    parts, res, gamma = inp["partials"].to(dev), inp["residual"].to(dev), inp["gamma"].to(dev)
    for rs, form in ((8, 1), (7, 6)):
        whole = pkg.new_outputs(form, T, H, dev)
        pkg.ts_reducescatter_fused_norm(rs, parts, -1, add, res, gamma, EPS, **whole)
        for rank in range(R):
            start, count = pkg.rs_token_split(T, R, rank)
            one = pkg.new_outputs(form, count, H, dev)
            pkg.ts_reducescatter_fused_norm(rs, parts, rank, add[start:start + count], res[start:start + count],
                                            gamma, EPS, **one)
            torch.cuda.synchronize()
            for k, v in one.items():
                assert np.array_equal(host(v), host(whole[k][start:start + count])), (rs, rank, k)


# the instances of the two flags (2-8 partials, one or two chunks a thread,
# more rows than SMs), and shapes where a flag is accepted and changes nothing
EARLY_SHAPES = [(8, 600, 7168), (5, 300, 2048), (8, 400, 4096), (4, 400, 7168), (3, 500, 4096),
                (2, 600, 8192), (2, 300, 4096), (4, 100, 7168), (3, 50, 16384), (1, 1300, 1024)]


@pytest.mark.parametrize("flag", ["early", "independent"])
@pytest.mark.parametrize("R,T,H", EARLY_SHAPES, ids=[f"R{r}-T{t}-H{h}" for r, t, h in EARLY_SHAPES])
@pytest.mark.parametrize("pattern,layout", [(1, LIN), (3, SW128), (6, LIN), (7, LIN), (0, LIN)])
def test_early_read_gives_the_same_bits(dev, pattern, layout, R, T, H, flag):
    """TS_FLAG_PDL_EARLY_READ (inputs read before the dependency wait) and
    TS_FLAG_PDL_INDEPENDENT (the wait just before exit): a chain of
    launch_with_pdl calls with the flag on one stream, each on its own outputs,
    gives the bits of a plain call: where the flag has its own instances (one
    and two chunks a thread, the padding rows of a swizzled SF buffer) and
    where it changes nothing (the paired, four-chunk and prefetching
    layouts)."""
    inp = _inputs(R, T, H, seed=pattern + R + T)
    scale = 300.0 if pattern == 3 else None
    P = 512 if pattern == 7 else 0
    want = _run_gpu(dev, pattern, inp, scale, P, layout)
    parts = inp["partials"].to(dev)
    res = None if pattern == 0 else inp["residual"].to(dev)
    gamma = None if pattern == 0 else inp["gamma"].to(dev)
    sf = None if scale is None else torch.tensor([scale], dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    outs = [pkg.new_outputs(pattern, T, H, dev, partial_cols=P, sf_layout=layout, with_allreduce_out=True)
            for _ in range(3)]
    with torch.cuda.stream(s):
        for o in outs:
            pkg.ts_fused_reduce_norm(pattern, parts, res, gamma, EPS, sf, sf_layout=layout, launch_with_pdl=True,
                                     pdl_early_read=flag == "early", pdl_independent=flag == "independent",
                                     stream=s, **o)
    torch.cuda.synchronize()
    for o in outs:
        for k, v in o.items():
            assert np.array_equal(host(v), want[k]), k


@pytest.mark.parametrize("flag", ["early", "independent"])
@pytest.mark.parametrize("rs,form", [(7, 6), (8, 1)])
def test_reducescatter_rank_chain_with_early_read(dev, rs, form, flag):
    """The per-rank calls of one reduce-scatter, back to back on one stream with
    launch_with_pdl and TS_FLAG_PDL_EARLY_READ or TS_FLAG_PDL_INDEPENDENT (no
    call writes another's inputs or touches its outputs), equal the one launch
    over every rank's slice; and a kernel after the chain on the same stream
    (a copy of every slice's residual_out) sees every call's results."""
    R, T, H = 8, 3000, 7168
    inp = _inputs(R, T, H, seed=40 + rs)
    g = torch.Generator().manual_seed(41)
    add = torch.randn((T, H), generator=g).to(torch.bfloat16).to(dev)
    parts, res, gamma = inp["partials"].to(dev), inp["residual"].to(dev), inp["gamma"].to(dev)
    whole = pkg.new_outputs(form, T, H, dev)
    pkg.ts_reducescatter_fused_norm(rs, parts, -1, add, res, gamma, EPS, **whole)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    per = []
    with torch.cuda.stream(s):
        for rank in range(R):
            start, count = pkg.rs_token_split(T, R, rank)
            one = pkg.new_outputs(form, count, H, dev)
            pkg.ts_reducescatter_fused_norm(rs, parts, rank, add[start:start + count], res[start:start + count],
                                            gamma, EPS, launch_with_pdl=True, pdl_early_read=flag == "early",
                                            pdl_independent=flag == "independent", stream=s, **one)
            per.append((start, count, one))
        copies = [one["residual_out"].clone() for _, _, one in per]
    torch.cuda.synchronize()
    for (start, count, one), c in zip(per, copies):
        for k, v in one.items():
            assert np.array_equal(host(v), host(whole[k][start:start + count])), k
        assert np.array_equal(host(c), host(whole["residual_out"][start:start + count]))


def test_golden_sum_order(dev):
    """The hand-derived example of tests/golden/rounding_order.txt in which the
    order of the peers' fp32 additions decides the bf16 result: ascending from
    a zero accumulator gives 1.0, descending would give 1.0078125.  Bit for bit
    through the C ABI, for kAllReduce and for the allreduce_out and
    residual_out (zero residual) of kARResidualRMSNorm."""
    from tests.golden_util import read_fixture

    c = read_fixture("rounding_order.txt")["sum_order"]
    R, H, want = c["R"], c["H"], c["allreduce_out"][0]
    parts = torch.tensor(np.array([np.full((1, H), b, np.uint16) for b in c["partials"]]).view(np.int16)) \
        .view(torch.bfloat16).to(dev)
    assert parts.shape == (R, 1, H)
    out = torch.empty((1, H), dtype=torch.bfloat16, device=dev)
    pkg.ts_fused_reduce_norm(0, parts, None, None, EPS, allreduce_out=out)
    res = torch.zeros((1, H), dtype=torch.bfloat16, device=dev)
    gamma = torch.ones(H, dtype=torch.bfloat16, device=dev)
    o1 = pkg.new_outputs(1, 1, H, dev, with_allreduce_out=True)
    pkg.ts_fused_reduce_norm(1, parts, res, gamma, EPS, **o1)
    torch.cuda.synchronize()
    for t in (out, o1["allreduce_out"], o1["residual_out"]):
        assert np.array_equal(host(t), np.full((1, H), want, np.uint16))


def test_golden_add_order(dev):
    """The hand-derived reduce-scatter Add example of
    tests/golden/rounding_order.txt: x = ((sum of partials) + add_in) +
    residual gives bf16 1.0 where adding the residual first would give
    1.0078125.  Bit for bit through the C ABI, for rank 0 and for the one
    launch over every rank."""
    from tests.golden_util import read_fixture

    c = read_fixture("rounding_order.txt")["add_order"]
    R, H = c["R"], c["H"]

    def bf(vals, shape):
        return torch.tensor(np.full(shape, vals, np.uint16).view(np.int16)).view(torch.bfloat16).to(dev)

    parts = torch.stack([bf(b, (R, H)) for b in c["partials"]])  # T = R rows, one per rank
    gamma = bf(0x3F80, (H,))
    for rank, rows in ((0, 1), (-1, R)):
        outs = {k: torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
                for k in ("reducescatter_out", "residual_out", "norm_out")}
        pkg.ts_reducescatter_fused_norm(c["pattern"], parts, rank, bf(c["add_in"][0], (rows, H)),
                                        bf(c["residual"][0], (rows, H)), gamma, EPS, **outs)
        torch.cuda.synchronize()
        assert np.array_equal(host(outs["residual_out"]), np.full((rows, H), c["residual_out"][0], np.uint16))
        assert np.array_equal(host(outs["reducescatter_out"]),
                              np.full((rows, H), c["reducescatter_out"][0], np.uint16))


@pytest.mark.parametrize("name", ["fp4_sf_order", "fp4_element_order"])
def test_golden_fp4_order(dev, name):
    """The hand-derived NVFP4 examples of tests/golden/rounding_order.txt, in
    which the order of the scale products decides an E4M3 scale factor (g *
    (amax / 6)) or an E2M1 code (n * (g / value(SF))): bit for bit through the
    C ABI (the row's mean of squares is exactly 1, so the norm is the row)."""
    from tests.golden_util import read_fixture

    c = read_fixture("rounding_order.txt")[name]
    H = c["H"]
    row = np.array(c["row"], np.uint16)
    g = float(np.array(c["scale_factor_bits"], np.uint32).view(np.float32)[0])
    part = torch.tensor(row.reshape(1, 1, H).view(np.int16)).view(torch.bfloat16).to(dev)
    res = torch.zeros((1, H), dtype=torch.bfloat16, device=dev)
    gamma = torch.ones(H, dtype=torch.bfloat16, device=dev)
    outs = pkg.new_outputs(3, 1, H, dev)
    pkg.ts_fused_reduce_norm(3, part, res, gamma, float(c["eps"]), torch.tensor([g], device=dev), **outs)
    torch.cuda.synchronize()
    assert np.array_equal(host(outs["residual_out"])[0], row)
    assert int(host(outs["scale_out"])[0, 0]) == c["sf_block0"][0]
    assert list(host(outs["quant_out"])[0, :8]) == c["quant_block0"]

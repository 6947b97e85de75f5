"""GPU parity of ts_qk_norm_sharded against the CPU oracle, through the C ABI.

Tolerance: every output within 1 bf16 ulp of the oracle and >= 99.9 %
bit-identical (the GPU sums squares in an fp32 tree and uses rsqrtf; the
oracle sums in double and rounds rsqrt correctly).  Output columns beyond
R*Q (or R*K) of a padded leading dimension must stay untouched.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_gb300 as pkg
from reduce_residual_rmsnorm_gb300 import workloads as wl
from tests.gpu_util import FILL, Guarded, host
from tests.helpers import assert_bf16_close

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def _run(dev, inp, Q, K, ldq=None, ldk=None):
    sh = inp["shards"]
    R, T, _ = sh.shape
    ldq = ldq or R * Q
    ldk = ldk or R * K
    gq = Guarded((T, ldq), torch.bfloat16, dev)
    gk = Guarded((T, ldk), torch.bfloat16, dev)
    pkg.ts_qk_norm_sharded(sh.to(dev), Q, K, inp["q_weight"].to(dev), inp["k_weight"].to(dev), EPS,
                           q_out=gq.t, k_out=gk.t)
    torch.cuda.synchronize()
    assert gq.intact() and gk.intact(), "write outside the outputs"
    q, k = host(gq.t), host(gk.t)
    pad = np.uint16(FILL | (FILL << 8))
    assert (q[:, R * Q:] == pad).all() and (k[:, R * K:] == pad).all(), "padding columns written"
    return q[:, :R * Q], k[:, :R * K]


def _oracle(inp, Q, K, rows=None):
    return oracle.qk_norm_sharded([wl.bits(s) for s in inp["shards"]], Q, K, wl.bits(inp["q_weight"]),
                                  wl.bits(inp["k_weight"]), EPS, rows=rows)


CASES = [  # R, T, Q, K, V, ldq pad, ldk pad
    (8, 33, 1024, 128, 128, 0, 0),    # the MiniMax shard shape
    (1, 1, 8, 8, 0, 0, 0),
    (2, 9, 768, 128, 128, 8, 16),
    (3, 17, 136, 24, 40, 0, 8),
    (4, 64, 1536, 256, 256, 0, 0),
    (16, 5, 384, 64, 64, 0, 0),
    (8, 3, 4096, 1024, 8, 64, 64),
    (5, 130, 256, 512, 0, 0, 0),
    (2, 6000, 256, 64, 16, 0, 0),    # two tokens per warp; T beyond one wave, so the L2 prefetch runs
    (3, 40, 512, 512, 64, 8, 0),      # 2 + 2 chunks per lane: weights loaded before the barrier
    (2, 21, 256, 1024, 0, 0, 8),      # 1 + 4 chunks per lane, likewise
]


@pytest.mark.parametrize("R,T,Q,K,V,pq,pk", CASES, ids=[f"R{c[0]}-T{c[1]}-Q{c[2]}-K{c[3]}" for c in CASES])
def test_small_shapes(dev, R, T, Q, K, V, pq, pk):
    inp = wl.qk_inputs(wl.QKShape(R=R, T=T, q_shard=Q, k_shard=K, v_shard=V), seed=R + T + Q)
    q, k = _run(dev, inp, Q, K, R * Q + pq, R * K + pk)
    wq, wk = _oracle(inp, Q, K)
    assert_bf16_close(q, wq, 1, 0.999, "q_out")
    assert_bf16_close(k, wk, 1, 0.999, "k_out")


def test_strided_views(dev):
    """q|k|v taken as views of one wider [T, 2*stride] buffer per shard."""
    R, T, Q, K, V = 4, 21, 256, 64, 64
    inp = wl.qk_inputs(wl.QKShape(R=R, T=T, q_shard=Q, k_shard=K, v_shard=V), seed=5)
    stride = Q + K + V
    wide = torch.zeros((R, T, 2 * stride), dtype=torch.bfloat16)
    wide[:, :, :stride] = inp["shards"]
    wd = wide.to(dev)
    views = [wd[r, :, :stride] for r in range(R)]
    q_out, k_out = pkg.ts_qk_norm_sharded(views, Q, K, inp["q_weight"].to(dev), inp["k_weight"].to(dev), EPS)
    torch.cuda.synchronize()
    wq, wk = _oracle(inp, Q, K)
    assert_bf16_close(host(q_out), wq, 1, 0.999, "q strided")
    assert_bf16_close(host(k_out), wk, 1, 0.999, "k strided")


def test_zero_tokens(dev):
    sh = torch.empty((8, 0, 1280), dtype=torch.bfloat16, device=dev)
    q, k = pkg.ts_qk_norm_sharded(sh, 1024, 128, torch.ones(8192, dtype=torch.bfloat16, device=dev),
                                  torch.ones(1024, dtype=torch.bfloat16, device=dev), EPS)
    assert q.shape == (0, 8192) and k.shape == (0, 1024)


@pytest.mark.slow
def test_full_size_minimax(dev):
    """R=8 shards [T=32768, q 1024 | k 128 | v 128]: 4096 sampled tokens
    (first and last 64 and a seeded random draw) through the oracle."""
    inp = wl.qk_inputs(wl.WORKLOADS["C5"], seed=0)
    q, k = _run(dev, inp, 1024, 128)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(32768 - 64, 32768),
                                     rng.integers(0, 32768, 4000)]))
    wq, wk = _oracle(inp, 1024, 128, rows=rows)
    assert_bf16_close(q[rows], wq, 1, 0.999, "q_out")
    assert_bf16_close(k[rows], wk, 1, 0.999, "k_out")


# ---------------------------------------------------------------------------
# single-matrix sharded RMSNorm (ts_rms_norm_sharded)
# ---------------------------------------------------------------------------

def _rms_inputs(R, T, W, extra, seed):
    g = torch.Generator().manual_seed(seed)
    shards = torch.randn((R, T, W + extra), generator=g).to(torch.bfloat16)
    w = (torch.rand(R * W, generator=g) + 0.5).to(torch.bfloat16)
    return shards, w


RMS_CASES = [(8, 33, 768, 0, 0), (1, 1, 8, 0, 0), (2, 9, 3072, 0, 0), (3, 17, 136, 24, 8),
             (16, 5, 384, 64, 0), (5, 130, 4096, 8, 16), (4, 64, 1024, 0, 64), (8, 3000, 768, 0, 0)]


@pytest.mark.parametrize("R,T,W,extra,pad", RMS_CASES, ids=[f"R{c[0]}-T{c[1]}-W{c[2]}" for c in RMS_CASES])
def test_single_matrix_small_shapes(dev, R, T, W, extra, pad):
    shards, w = _rms_inputs(R, T, W, extra, seed=R * 7 + T)
    g = Guarded((T, R * W + pad), torch.bfloat16, dev)
    pkg.ts_rms_norm_sharded(shards.to(dev), W, w.to(dev), EPS, out=g.t)
    torch.cuda.synchronize()
    assert g.intact()
    out = host(g.t)
    assert (out[:, R * W:] == np.uint16(FILL | (FILL << 8))).all()
    want = oracle.rms_norm_sharded([wl.bits(s) for s in shards], W, wl.bits(w), EPS)
    assert_bf16_close(out[:, :R * W], want, 1, 0.999, "single-matrix")


def test_single_matrix_agrees_with_qk_q_segment(dev):
    inp = wl.qk_inputs(wl.QKShape(R=8, T=64, q_shard=1024, k_shard=128, v_shard=128), seed=12)
    sh = inp["shards"].to(dev)
    q, _ = pkg.ts_qk_norm_sharded(sh, 1024, 128, inp["q_weight"].to(dev), inp["k_weight"].to(dev), EPS)
    single = pkg.ts_rms_norm_sharded(sh, 1024, inp["q_weight"].to(dev), EPS)
    torch.cuda.synchronize()
    assert np.array_equal(host(q), host(single))


@pytest.mark.slow
def test_single_matrix_full_size(dev):
    """R=8 shards of [T=32768, 768] (MiniMax-M2's 6144-wide q split 8 ways)."""
    shards, w = _rms_inputs(8, 32768, 768, 0, seed=0)
    out = pkg.ts_rms_norm_sharded(shards.to(dev), 768, w.to(dev), EPS)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(32), np.arange(32768 - 32, 32768), rng.integers(0, 32768, 2000)]))
    want = oracle.rms_norm_sharded([wl.bits(s) for s in shards], 768, wl.bits(w), EPS, rows=rows)
    assert_bf16_close(host(out)[rows], want, 1, 0.999, "single-matrix full size")


def test_pdl_qk_matches_plain(dev):
    inp = wl.qk_inputs(wl.QKShape(R=8, T=300, q_shard=1024, k_shard=128, v_shard=128), seed=13)
    sh = inp["shards"].to(dev)
    wq, wk = inp["q_weight"].to(dev), inp["k_weight"].to(dev)
    a = pkg.ts_qk_norm_sharded(sh, 1024, 128, wq, wk, EPS)
    b = pkg.ts_qk_norm_sharded(sh, 1024, 128, wq, wk, EPS, launch_with_pdl=True)
    c = pkg.ts_rms_norm_sharded(sh, 1024, wq, EPS, launch_with_pdl=True)
    torch.cuda.synchronize()
    assert np.array_equal(host(a[0]), host(b[0])) and np.array_equal(host(a[1]), host(b[1]))
    assert np.array_equal(host(a[0]), host(c))

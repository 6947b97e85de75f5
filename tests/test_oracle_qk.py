"""Pins for the oracle of the sharded MiniMax QK-RMSNorm.

The sharded definition (per-shard means of squares, summed over the shards,
divided by R inside the rsqrt) must agree with the unsharded RMSNorm over the
concatenated q (and k) when the shards have equal widths, reduce to a textbook
RMSNorm for R = 1, give the closed form on constant rows, ignore the v
columns, and match an exact-real evaluation on tiny inputs.
"""
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch

from tests.helpers import assert_bf16_close, bf16_bits_of_f32, bf16_of_f64, f32_of_bf16

EPS = float(np.float32(1e-6))


def _qk_inputs(rng, R, T, Q, K, V, std=1.0):
    stride = Q + K + V
    shards = [bf16_bits_of_f32(rng.standard_normal((T, stride)).astype(np.float32) * std)
              for _ in range(R)]
    wq = bf16_bits_of_f32(rng.uniform(0.5, 1.5, R * Q).astype(np.float32))
    wk = bf16_bits_of_f32(rng.uniform(0.5, 1.5, R * K).astype(np.float32))
    return shards, wq, wk


def test_equal_shards_equal_unsharded_rmsnorm(orc):
    """(1/R) sum_r (1/Q) sum_j x^2 = (1/(RQ)) sum over the concatenated row, so
    the sharded norm equals a plain RMSNorm of the concatenation (evaluated
    here by the fused oracle with one partial and a zero residual)."""
    rng = np.random.default_rng(30)
    R, T, Q, K, V = 4, 12, 256, 64, 64
    shards, wq, wk = _qk_inputs(rng, R, T, Q, K, V)
    q_out, k_out = orc.qk_norm_sharded(shards, Q, K, wq, wk, eps=EPS)
    q_cat = np.concatenate([s[:, :Q] for s in shards], axis=1)
    k_cat = np.concatenate([s[:, Q:Q + K] for s in shards], axis=1)
    zq = np.zeros_like(q_cat)
    zk = np.zeros_like(k_cat)
    want_q = orc.fused_reduce_norm(1, [q_cat], zq, wq, eps=EPS)["norm_out"]
    want_k = orc.fused_reduce_norm(1, [k_cat], zk, wk, eps=EPS)["norm_out"]
    assert_bf16_close(q_out, want_q, 1, 0.99, "q vs unsharded")
    assert_bf16_close(k_out, want_k, 1, 0.99, "k vs unsharded")


def test_single_shard_is_plain_rmsnorm(orc):
    rng = np.random.default_rng(31)
    T, Q, K, V = 9, 128, 32, 8
    shards, wq, wk = _qk_inputs(rng, 1, T, Q, K, V)
    q_out, k_out = orc.qk_norm_sharded(shards, Q, K, wq, wk, eps=EPS)
    for out, lo, hi, w in ((q_out, 0, Q, wq), (k_out, Q, Q + K, wk)):
        x = f32_of_bf16(shards[0][:, lo:hi]).astype(np.float64)
        want = x / np.sqrt((x * x).mean(1, keepdims=True) + EPS) * f32_of_bf16(w)
        assert_bf16_close(out, bf16_of_f64(want), 1, 0.99, "R=1")


def test_constant_rows_closed_form(orc):
    """Shard r holds the constant c_r: the global mean of squares is
    mean_r(c_r^2), so out = w * c_r / sqrt(mean_r(c_r^2) + eps)."""
    R, T, Q, K, V = 4, 2, 64, 16, 16
    cs = [0.5, -0.25, 2.0 ** -10, 1.5]
    shards = [bf16_bits_of_f32(np.full((T, Q + K + V), c, np.float32)) for c in cs]
    rng = np.random.default_rng(32)
    wq = bf16_bits_of_f32(rng.uniform(0.5, 1.5, R * Q).astype(np.float32))
    wk = bf16_bits_of_f32(rng.uniform(0.5, 1.5, R * K).astype(np.float32))
    q_out, k_out = orc.qk_norm_sharded(shards, Q, K, wq, wk, eps=EPS)
    ms = float(np.mean(np.square(cs)))
    for out, width, w in ((q_out, Q, wq), (k_out, K, wk)):
        c_row = np.repeat(cs, width)
        want = bf16_of_f64(f32_of_bf16(w).astype(np.float64) * c_row / np.sqrt(ms + EPS))
        assert_bf16_close(out, np.broadcast_to(want, out.shape), 1, 0.99, "constant")


def test_v_columns_are_ignored(orc):
    rng = np.random.default_rng(33)
    R, T, Q, K, V = 3, 5, 64, 32, 32
    shards, wq, wk = _qk_inputs(rng, R, T, Q, K, V)
    a = orc.qk_norm_sharded(shards, Q, K, wq, wk)
    other = [s.copy() for s in shards]
    for s in other:
        s[:, Q + K:] = bf16_bits_of_f32(rng.standard_normal((T, V)).astype(np.float32) * 100)
    b = orc.qk_norm_sharded(other, Q, K, wq, wk)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_shard_order_and_weight_slices(orc):
    """Swapping two shards (and their weight slices) swaps the output blocks;
    the shared mean of squares is unchanged up to fp32 summation order."""
    rng = np.random.default_rng(34)
    R, T, Q, K, V = 2, 6, 64, 16, 16
    shards, wq, wk = _qk_inputs(rng, R, T, Q, K, V)
    q0, k0 = orc.qk_norm_sharded(shards, Q, K, wq, wk)
    wq_s = np.concatenate([wq[Q:], wq[:Q]])
    wk_s = np.concatenate([wk[K:], wk[:K]])
    q1, k1 = orc.qk_norm_sharded(shards[::-1], Q, K, wq_s, wk_s)
    assert_bf16_close(q1, np.concatenate([q0[:, Q:], q0[:, :Q]], 1), 1, 0.999, "q swap")
    assert_bf16_close(k1, np.concatenate([k0[:, K:], k0[:, :K]], 1), 1, 0.999, "k swap")


def test_brute_force_exact_reals(orc):
    getcontext().prec = 50
    rng = np.random.default_rng(35)
    R, T, Q, K, V = 2, 4, 8, 8, 8
    ints = rng.integers(-64, 65, size=(R, T, Q + K + V))
    shards = [bf16_bits_of_f32((i / 32.0).astype(np.float32)) for i in ints]
    wq = bf16_bits_of_f32(rng.uniform(0.5, 1.5, R * Q).astype(np.float32))
    wk = bf16_bits_of_f32(rng.uniform(0.5, 1.5, R * K).astype(np.float32))
    q_out, k_out = orc.qk_norm_sharded(shards, Q, K, wq, wk, eps=EPS)
    for out, lo, width, w in ((q_out, 0, Q, wq), (k_out, Q, K, wk)):
        wf = f32_of_bf16(w)
        want = np.empty(out.shape)
        for t in range(T):
            xs = [[Fraction(int(ints[r, t, lo + j]), 32) for j in range(width)] for r in range(R)]
            m = sum(sum(v * v for v in row) / width for row in xs) / R + Fraction(EPS)
            inv = Decimal(1) / (Decimal(m.numerator) / Decimal(m.denominator)).sqrt()
            for r in range(R):
                for j in range(width):
                    v = xs[r][j]
                    want[t, r * width + j] = float(Decimal(v.numerator) / Decimal(v.denominator)
                                                   * inv * Decimal(float(wf[r * width + j])))
        assert_bf16_close(out, bf16_of_f64(want), 1, 0.95, "QK brute force")


def test_agrees_with_eager_torch_definition(orc):
    """A cross-check (not a pin): the eager fp32 torch formulation of the
    sharded norm, with the all-reduce of the [T, 2] variance written as a sum
    over the shards."""
    rng = np.random.default_rng(36)
    R, T, Q, K, V = 4, 16, 128, 32, 32
    shards, wq, wk = _qk_inputs(rng, R, T, Q, K, V)
    q_out, k_out = orc.qk_norm_sharded(shards, Q, K, wq, wk, eps=EPS)
    var = torch.zeros(T, 2)
    xs = []
    for s in shards:
        t = torch.from_numpy(f32_of_bf16(s))
        q, k = t[:, :Q], t[:, Q:Q + K]
        xs.append((q, k))
        var += torch.cat([q.pow(2).mean(-1, keepdim=True), k.pow(2).mean(-1, keepdim=True)], -1)
    var = var / R
    qv, kv = var.chunk(2, -1)
    wqf = torch.from_numpy(f32_of_bf16(wq)).view(R, Q)
    wkf = torch.from_numpy(f32_of_bf16(wk)).view(R, K)
    q_ref = torch.cat([xs[r][0] * torch.rsqrt(qv + EPS) * wqf[r] for r in range(R)], 1)
    k_ref = torch.cat([xs[r][1] * torch.rsqrt(kv + EPS) * wkf[r] for r in range(R)], 1)
    to_bits = lambda x: x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    assert_bf16_close(q_out, to_bits(q_ref), 1, 0.99, "eager q")
    assert_bf16_close(k_out, to_bits(k_ref), 1, 0.99, "eager k")


# ---------------------------------------------------------------------------
# single-matrix sharded RMSNorm (one segment instead of q and k)
# ---------------------------------------------------------------------------

def test_single_matrix_equals_unsharded_rmsnorm(orc):
    rng = np.random.default_rng(40)
    R, T, W = 8, 10, 96
    shards = [bf16_bits_of_f32(rng.standard_normal((T, W + 16)).astype(np.float32)) for _ in range(R)]
    w = bf16_bits_of_f32(rng.uniform(0.5, 1.5, R * W).astype(np.float32))
    out = orc.rms_norm_sharded(shards, W, w, eps=EPS)
    cat = np.concatenate([s[:, :W] for s in shards], axis=1)
    want = orc.fused_reduce_norm(1, [cat], np.zeros_like(cat), w, eps=EPS)["norm_out"]
    assert_bf16_close(out, want, 1, 0.99, "single-matrix vs unsharded")


def test_single_matrix_is_the_q_segment_of_qk(orc):
    """With the same shards, the single-matrix norm of the first W columns is
    the QK norm's q output (the k segment does not enter q's variance)."""
    rng = np.random.default_rng(41)
    R, T, Q, K = 3, 7, 64, 16
    shards, wq, wk = _qk_inputs(rng, R, T, Q, K, 8)
    q_out, _ = orc.qk_norm_sharded(shards, Q, K, wq, wk, eps=EPS)
    assert np.array_equal(orc.rms_norm_sharded(shards, Q, wq, eps=EPS), q_out)


def test_single_matrix_single_shard_textbook(orc):
    rng = np.random.default_rng(42)
    T, W = 5, 256
    sh = [bf16_bits_of_f32(rng.standard_normal((T, W)).astype(np.float32) * 3)]
    w = bf16_bits_of_f32(rng.uniform(0.5, 1.5, W).astype(np.float32))
    out = orc.rms_norm_sharded(sh, W, w, eps=EPS)
    x = f32_of_bf16(sh[0]).astype(np.float64)
    want = x / np.sqrt((x * x).mean(1, keepdims=True) + EPS) * f32_of_bf16(w)
    assert_bf16_close(out, bf16_of_f64(want), 1, 0.99, "single shard")


def test_single_matrix_constant_rows(orc):
    R, T, W = 4, 2, 32
    cs = [0.75, -0.5, 2.0 ** -11, 3.0]
    sh = [bf16_bits_of_f32(np.full((T, W), c, np.float32)) for c in cs]
    rng = np.random.default_rng(43)
    w = bf16_bits_of_f32(rng.uniform(0.5, 1.5, R * W).astype(np.float32))
    out = orc.rms_norm_sharded(sh, W, w, eps=EPS)
    ms = float(np.mean(np.square(cs)))
    want = bf16_of_f64(f32_of_bf16(w).astype(np.float64) * np.repeat(cs, W) / np.sqrt(ms + EPS))
    assert_bf16_close(out, np.broadcast_to(want, out.shape), 1, 0.99, "constant")

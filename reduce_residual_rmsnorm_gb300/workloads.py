"""Seeded synthetic inputs for the fused reduce/residual/RMSNorm path and the
sharded QK-RMSNorm.

This module only draws random numbers: it holds none of the method's
arithmetic, so both the CUDA path's tests/benchmark and the CPU oracle can be
fed from it.  Every tensor is drawn on the host with a seeded
``torch.Generator`` in a fixed order (partials r = 0..R-1, then the residual,
then gamma; for QK the R shards, then q_weight, then k_weight), drawn in fp32
and rounded to bf16 by PyTorch's conversion.

Named workloads (the shapes and value distributions the method is measured on):

=====  ======================================  ==========================================
name   what                                    shapes / distributions
=====  ======================================  ==========================================
C1     kARResidualRMSNorm, R=2                 T=16, H=4096; p,res ~N(0,1); gamma ~U(.5,1.5)
C2     kARResidualRMSNorm and kAllReduce, R=8  T=4096, H=7168; p ~N(0,0.5^2); res ~N(0,1)
C3     FP8 per-tensor / 1x128 blockwise /      T=8192, H=7168, R=8; as C2 plus 0.1% of the
       PartialOut(P=1024)                      entries of every partial and the residual x50
C4     NVFP4, R=4, LINEAR and SWIZZLED_128x4   T=16384, H=5120; p,res ~N(0,1)
C5     MiniMax sharded QK-RMSNorm, R=8         T=32768, shard row q 1024 | k 128 | v 128
                                               (stride 1280); x ~N(0,1); weights ~U(.5,1.5)
=====  ======================================  ==========================================

"N(0, 0.5)" in the C2/C3 description is read as a standard deviation of 0.5.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

BF16 = torch.bfloat16


@dataclass(frozen=True)
class FusedShape:
    R: int
    T: int
    H: int
    p_std: float = 1.0
    res_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_mul: float = 50.0


@dataclass(frozen=True)
class QKShape:
    R: int
    T: int
    q_shard: int
    k_shard: int
    v_shard: int

    @property
    def row_stride(self) -> int:
        return self.q_shard + self.k_shard + self.v_shard


WORKLOADS = {
    "C1": FusedShape(R=2, T=16, H=4096),
    "C2": FusedShape(R=8, T=4096, H=7168, p_std=0.5),
    "C3": FusedShape(R=8, T=8192, H=7168, p_std=0.5, outlier_frac=1e-3),
    "C4": FusedShape(R=4, T=16384, H=5120),
    "C5": QKShape(R=8, T=32768, q_shard=1024, k_shard=128, v_shard=128),
}


def _normal(shape, std, g, outlier_frac=0.0, outlier_mul=50.0):
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=g.device)
    if std != 1.0:
        x.mul_(std)
    if outlier_frac > 0.0:
        numel = x.numel()
        k = int(round(outlier_frac * numel))
        idx = torch.randint(0, numel, (k,), generator=g, device=g.device)
        x.view(-1)[idx] *= outlier_mul
    return x.to(BF16)


def _uniform(shape, lo, hi, g):
    return (torch.rand(shape, generator=g, dtype=torch.float32, device=g.device) * (hi - lo) + lo).to(BF16)


def fused_inputs(shape: FusedShape, seed: int = 0, device="cpu") -> dict:
    """bf16 tensors ``partials`` [R, T, H], ``residual`` [T, H], ``gamma`` [H].

    Drawn with a generator on ``device`` (host by default; the host and a
    CUDA generator give different, equally seeded, numbers)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    R, T, H = shape.R, shape.T, shape.H
    partials = torch.empty((R, T, H), dtype=BF16, device=device)
    for r in range(R):
        partials[r] = _normal((T, H), shape.p_std, g, shape.outlier_frac, shape.outlier_mul)
    residual = _normal((T, H), shape.res_std, g, shape.outlier_frac, shape.outlier_mul)
    gamma = _uniform((H,), 0.5, 1.5, g)
    return {"partials": partials, "residual": residual, "gamma": gamma}


def qk_inputs(shape: QKShape, seed: int = 0, device="cpu") -> dict:
    """bf16 tensors ``shards`` [R, T, row_stride], ``q_weight`` [R*q_shard],
    ``k_weight`` [R*k_shard], drawn with a generator on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    R, T = shape.R, shape.T
    shards = torch.empty((R, T, shape.row_stride), dtype=BF16, device=device)
    for r in range(R):
        shards[r] = _normal((T, shape.row_stride), 1.0, g)
    q_weight = _uniform((R * shape.q_shard,), 0.5, 1.5, g)
    k_weight = _uniform((R * shape.k_shard,), 0.5, 1.5, g)
    return {"shards": shards, "q_weight": q_weight, "k_weight": k_weight}


def bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a host bf16 tensor, as a numpy array (no copy)."""
    assert t.dtype == BF16 and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def row_split(T: int, world_size: int, rank: int) -> tuple[int, int]:
    """Rows [start, start+count) of rank ``rank`` when T independent rows are
    split over ``world_size`` GPUs: T//W rows each, the first T%W ranks one
    more (the token split of tokenspeed's `rsag_get_token_dist`)."""
    base, extra = divmod(T, world_size)
    count = base + (1 if rank < extra else 0)
    start = rank * base + min(rank, extra)
    return start, count

"""ctypes binding of ``libts_fused_norm.so`` (include/ts_fused_norm.h).

Argument marshalling only: tensors (CUDA, or pinned host tensors the kernels
address across the host link) become pointers, the stream is
PyTorch's current stream, and a non-zero status becomes a ``TsError``.  Every
step of the computation runs in the library's CUDA kernels; there is no
Python or CPU fallback, and calling without the built library raises.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading
from typing import Sequence

import torch

from .build import LIB_PATH

_lock = threading.Lock()
_lib = None


class Pattern(enum.IntEnum):
    """`AllReduceFusionPattern` codes (tokenspeed trtllm.py)."""
    kAllReduce = 0
    kARResidualRMSNorm = 1
    kARResidualRMSNormFP8Quant = 2
    kARResidualRMSNormFP4Quant = 3
    kARResidualRMSNormOutFP8Quant = 4
    kARResidualRMSNormOutFP4Quant = 5
    kARResidualRMSNormFP8BlockWiseQuant = 6
    kARResidualRMSNormPartialOutFP8BlockWiseQuant = 7
    kARResidualRMSNormPartialOut = 8


class RSPattern(enum.IntEnum):
    """`ReduceScatterFusionPattern` codes (tokenspeed trtllm.py)."""
    kReduceScatter = 0
    kRSResidualRMSNorm = 1
    kRSResidualRMSNormFP8Quant = 2
    kRSResidualRMSNormFP4Quant = 3
    kRSResidualRMSNormOutFP8Quant = 4
    kRSResidualRMSNormOutFP4Quant = 5
    kRSResidualRMSNormFP8BlockWiseQuant = 6
    kRSAddResidualRMSNormFP8BlockWiseQuant = 7
    kRSAddResidualRMSNorm = 8


class AGPattern(enum.IntEnum):
    """`AllGatherFusionPattern` codes (tokenspeed trtllm.py)."""
    kAllGather = 0
    kAllGatherfusedRMS = 1
    kAllGatherfusedRMSFP8BlockWiseQuant = 2


class SFLayout(enum.IntEnum):
    """`QuantizationSFLayout` codes (tokenspeed trtllm.py)."""
    SWIZZLED_128x4 = 0
    SWIZZLED_8x4 = 1
    LINEAR = 2


class TsError(RuntimeError):
    def __init__(self, status: int, name: str, detail: str):
        super().__init__(f"{name}: {detail}")
        self.status = status
        self.name = name
        self.detail = detail


class TsOuts(ctypes.Structure):
    _fields_ = [
        ("allreduce_out", ctypes.c_void_p),
        ("residual_out", ctypes.c_void_p),
        ("norm_out", ctypes.c_void_p),
        ("partial_norm_out", ctypes.c_void_p),
        ("partial_cols", ctypes.c_int64),
        ("quant_out", ctypes.c_void_p),
        ("scale_out", ctypes.c_void_p),
        ("sf_layout", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


EXPORTS = ("ts_fused_reduce_norm", "ts_reducescatter_fused_norm", "ts_allgather_fused_norm", "ts_qk_norm_sharded",
           "ts_rms_norm_sharded", "ts_status_string", "ts_last_error_detail")

TS_FLAG_PDL = 1
TS_FLAG_PDL_EARLY_READ = 2
TS_FLAG_PDL_INDEPENDENT = 4


def _fused_flags(launch_with_pdl: bool, pdl_early_read: bool, pdl_independent: bool) -> int:
    return ((TS_FLAG_PDL if launch_with_pdl else 0) | (TS_FLAG_PDL_EARLY_READ if pdl_early_read else 0) |
            (TS_FLAG_PDL_INDEPENDENT if pdl_independent else 0))


def library(path: str | None = None):
    """Load the CUDA library (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        u32 = ctypes.c_uint32
        lib.ts_fused_reduce_norm.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.c_int, vp, vp,
                                             ctypes.c_float, vp, i64, i64, ctypes.POINTER(TsOuts), u32, vp]
        lib.ts_fused_reduce_norm.restype = ctypes.c_int
        lib.ts_reducescatter_fused_norm.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int,
                                                    vp, vp, vp, ctypes.c_float, vp, i64, i64,
                                                    ctypes.POINTER(TsOuts), u32, vp]
        lib.ts_reducescatter_fused_norm.restype = ctypes.c_int
        lib.ts_allgather_fused_norm.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.c_int, i64, i64, i64, i64,
                                                i64, vp, vp, ctypes.c_float, ctypes.c_float, vp, vp, vp, vp, vp,
                                                u32, vp]
        lib.ts_allgather_fused_norm.restype = ctypes.c_int
        lib.ts_qk_norm_sharded.argtypes = [ctypes.POINTER(vp), ctypes.c_int, i64, i64, i64, i64, vp, vp,
                                           ctypes.c_float, vp, i64, vp, i64, u32, vp]
        lib.ts_qk_norm_sharded.restype = ctypes.c_int
        lib.ts_rms_norm_sharded.argtypes = [ctypes.POINTER(vp), ctypes.c_int, i64, i64, i64, vp,
                                            ctypes.c_float, vp, i64, u32, vp]
        lib.ts_rms_norm_sharded.restype = ctypes.c_int
        lib.ts_status_string.argtypes = [ctypes.c_int]
        lib.ts_status_string.restype = ctypes.c_char_p
        lib.ts_last_error_detail.argtypes = []
        lib.ts_last_error_detail.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _check(status: int) -> None:
    if status != 0:
        lib = library()
        raise TsError(status, lib.ts_status_string(status).decode(),
                      lib.ts_last_error_detail().decode())


def ts_status_string(status: int) -> str:
    return library().ts_status_string(int(status)).decode()


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    """A tensor the kernels can address: on the GPU, or in page-locked host
    memory (read and written by the kernel across the host link)."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or (t.device.type == "cpu" and t.is_pinned())):
        raise TypeError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _empty_like_place(shape, dtype, like: torch.Tensor) -> torch.Tensor:
    """A new tensor where ``like`` lives: the same GPU, or pinned host memory."""
    if like.is_cuda:
        return torch.empty(shape, dtype=dtype, device=like.device)
    return torch.empty(shape, dtype=dtype).pin_memory()


def _scalar_like_place(value: float, like: torch.Tensor) -> torch.Tensor:
    """One fp32 value where ``like`` lives, written before this returns (a
    blocking host-to-device copy, or a pinned host tensor)."""
    if like.is_cuda:
        return torch.tensor([value], dtype=torch.float32, device=like.device)
    return torch.tensor([value], dtype=torch.float32).pin_memory()


def _partials(partials) -> tuple[list[int], int, int, torch.Tensor]:
    """Pointers, T, H and one of the partials: R contiguous bf16 [T, H] tensors,
    or one contiguous [R, T, H] tensor (whose rows are addressed without
    making R views)."""
    if isinstance(partials, torch.Tensor):
        _dev(partials, "partials", torch.bfloat16)
        if partials.dim() != 3:
            raise ValueError("partials as one tensor must be [R, T, H]")
        if partials.is_contiguous():
            R, T, H = partials.shape
            base, step = partials.data_ptr(), T * H * 2
            return [base + r * step for r in range(R)], T, H, partials
        partials = list(partials.unbind(0))
    parts = [_dev(p, "partials[%d]" % i, torch.bfloat16) for i, p in enumerate(partials)]
    if not parts:
        raise ValueError("partials is empty")
    T, H = parts[0].shape
    for p in parts:
        if p.shape != (T, H) or not p.is_contiguous():
            raise ValueError("every partial must be a contiguous [T, H] tensor")
    return [p.data_ptr() for p in parts], T, H, parts[0]


def _rows(ts: torch.Tensor | Sequence[torch.Tensor], name: str) -> list[torch.Tensor]:
    if isinstance(ts, torch.Tensor):
        if ts.dim() != 3:
            raise ValueError(f"{name} as one tensor must be [R, T, H]")
        ts = list(ts.unbind(0))
    return list(ts)


def sf_shape(T: int, H: int, sf_layout: int = SFLayout.LINEAR) -> tuple[int, int]:
    """Shape of the NVFP4 scale-factor buffer for [T, H] values in ``sf_layout``
    (the swizzled layouts pad rows to 128 or 8 and columns to 4)."""
    layout = int(sf_layout)
    if layout == SFLayout.LINEAR:
        return T, H // 16
    tile = 128 if layout == SFLayout.SWIZZLED_128x4 else 8
    return (T + tile - 1) // tile * tile, (H // 16 + 3) // 4 * 4


def sf_swizzled_shape(T: int, H: int) -> tuple[int, int]:
    """Shape of the padded SWIZZLED_128x4 scale-factor buffer for [T, H] values."""
    return sf_shape(T, H, SFLayout.SWIZZLED_128x4)


def new_outputs(pattern: int, T: int, H: int, device="cuda", partial_cols: int = 0,
                sf_layout: int = SFLayout.LINEAR, with_allreduce_out: bool = False) -> dict:
    """Allocate (torch.empty) the required outputs of a pattern."""
    p = int(pattern)
    e = lambda *s, dt=torch.bfloat16: torch.empty(s, dtype=dt, device=device)  # noqa: E731
    out = {}
    if p == 0 or with_allreduce_out:
        out["allreduce_out"] = e(T, H)
    if p != 0:
        out["residual_out"] = e(T, H)
    if p in (1, 4, 5):
        out["norm_out"] = e(T, H)
    if p in (7, 8):
        out["partial_norm_out"] = e(T, partial_cols)
    if p in (2, 4, 6, 7):
        out["quant_out"] = e(T, H, dt=torch.uint8)
    if p in (3, 5):
        out["quant_out"] = e(T, H // 2, dt=torch.uint8)
        out["scale_out"] = e(*sf_shape(T, H, sf_layout), dt=torch.uint8)
    if p in (6, 7):
        out["scale_out"] = e(T, H // 128, dt=torch.float32)
    return out


def ts_fused_reduce_norm(pattern: int, partials, residual: torch.Tensor | None = None,
                         gamma: torch.Tensor | None = None, eps: float = 1e-6,
                         scale_factor: torch.Tensor | float | None = None, *,
                         allreduce_out: torch.Tensor | None = None,
                         residual_out: torch.Tensor | None = None,
                         norm_out: torch.Tensor | None = None,
                         partial_norm_out: torch.Tensor | None = None,
                         quant_out: torch.Tensor | None = None,
                         scale_out: torch.Tensor | None = None,
                         sf_layout: int = SFLayout.LINEAR, launch_with_pdl: bool = False,
                         pdl_early_read: bool = False, pdl_independent: bool = False, stream=None) -> None:
    """Run one AllReduceFusionPattern (see include/ts_fused_norm.h).

    ``partials``: R CUDA bf16 tensors [T, H] (or one [R, T, H] tensor).
    ``scale_factor``: device fp32 tensor of one element, or a Python float
    (then copied to the device first, as trtllm.py's wrapper does).
    ``partial_norm_out``'s width gives partial_cols.
    ``launch_with_pdl``: programmatic dependent launch (TS_FLAG_PDL).
    ``pdl_early_read``: with it, read the first inputs before waiting for the
    previous kernel (TS_FLAG_PDL_EARLY_READ; only when that kernel writes none
    of this call's inputs).
    ``pdl_independent``: with it, run without waiting for the kernels before it
    and wait only before finishing (TS_FLAG_PDL_INDEPENDENT; only when none of
    the kernels of the run of such calls, nor the one just before the run,
    writes this call's inputs or touches its outputs).
    """
    ptrs, T, H, part0 = _partials(partials)
    for name, t in (("residual", residual), ("gamma", gamma), ("allreduce_out", allreduce_out),
                    ("residual_out", residual_out), ("norm_out", norm_out),
                    ("partial_norm_out", partial_norm_out), ("quant_out", quant_out),
                    ("scale_out", scale_out)):
        if t is not None:
            _dev(t, name)
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
    if scale_factor is not None and not isinstance(scale_factor, torch.Tensor):
        scale_factor = _scalar_like_place(float(scale_factor), part0)
    if scale_factor is not None:
        _dev(scale_factor, "scale_factor", torch.float32)
    outs = TsOuts(_ptr(allreduce_out), _ptr(residual_out), _ptr(norm_out), _ptr(partial_norm_out),
                  0 if partial_norm_out is None else int(partial_norm_out.shape[-1]),
                  _ptr(quant_out), _ptr(scale_out), int(sf_layout), 0)
    arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
    _check(library().ts_fused_reduce_norm(int(pattern), arr, len(ptrs), _ptr(residual), _ptr(gamma),
                                          float(eps), _ptr(scale_factor), int(T), int(H),
                                          ctypes.byref(outs),
                                          _fused_flags(launch_with_pdl, pdl_early_read, pdl_independent),
                                          _stream(stream)))


def rs_token_split(T: int, world: int, rank: int) -> tuple[int, int]:
    """(start, count) of rank ``rank``'s token slice: T//world tokens each, the
    first T % world ranks one more (tokenspeed triton.py `rsag_get_token_dist`).
    Rank -1 stands for every rank's slice: (0, T)."""
    if rank < 0:
        return 0, T
    base, extra = divmod(T, world)
    return rank * base + min(rank, extra), base + (1 if rank < extra else 0)


def ts_reducescatter_fused_norm(rs_pattern: int, partials, rank: int, add_in: torch.Tensor | None = None,
                                residual: torch.Tensor | None = None, gamma: torch.Tensor | None = None,
                                eps: float = 1e-6, scale_factor: torch.Tensor | float | None = None, *,
                                reducescatter_out: torch.Tensor | None = None,
                                residual_out: torch.Tensor | None = None,
                                norm_out: torch.Tensor | None = None,
                                quant_out: torch.Tensor | None = None,
                                scale_out: torch.Tensor | None = None,
                                sf_layout: int = SFLayout.LINEAR, launch_with_pdl: bool = False,
                                pdl_early_read: bool = False, pdl_independent: bool = False, stream=None) -> None:
    """Rank ``rank``'s reduce-scatter fusion output (see include/ts_fused_norm.h).

    ``partials``: R CUDA bf16 tensors [T, H] holding every token; ``add_in``,
    ``residual`` and the outputs have the rank's ``count`` rows
    (``rs_token_split(T, R, rank)``); ``rank=-1`` computes every rank's slice
    in one launch (all T rows).
    """
    ptrs, T, H, part0 = _partials(partials)
    for name, t in (("add_in", add_in), ("residual", residual), ("gamma", gamma),
                    ("reducescatter_out", reducescatter_out), ("residual_out", residual_out),
                    ("norm_out", norm_out), ("quant_out", quant_out), ("scale_out", scale_out)):
        if t is not None:
            _dev(t, name)
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
    if scale_factor is not None and not isinstance(scale_factor, torch.Tensor):
        scale_factor = _scalar_like_place(float(scale_factor), part0)
    if scale_factor is not None:
        _dev(scale_factor, "scale_factor", torch.float32)
    outs = TsOuts(_ptr(reducescatter_out), _ptr(residual_out), _ptr(norm_out), None, 0, _ptr(quant_out),
                  _ptr(scale_out), int(sf_layout), 0)
    arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
    _check(library().ts_reducescatter_fused_norm(int(rs_pattern), arr, len(ptrs), int(rank), _ptr(add_in),
                                                 _ptr(residual), _ptr(gamma), float(eps), _ptr(scale_factor),
                                                 int(T), int(H), ctypes.byref(outs),
                                                 _fused_flags(launch_with_pdl, pdl_early_read, pdl_independent),
                                                 _stream(stream)))


def ts_allgather_fused_norm(ag_pattern: int, inputs, q_lora_rank: int, kv_lora_rank: int,
                            qk_rope_head_dim: int, x_gamma: torch.Tensor | None = None,
                            y_gamma: torch.Tensor | None = None, x_eps: float = 1e-6, y_eps: float = 1e-6, *,
                            allgather_out: torch.Tensor, x_norm_out: torch.Tensor | None = None,
                            y_norm_out: torch.Tensor | None = None, quant_out: torch.Tensor | None = None,
                            scale_out: torch.Tensor | None = None, launch_with_pdl: bool = False,
                            stream=None) -> None:
    """All-gather fusion with the dual MLA RMSNorm (see include/ts_fused_norm.h).

    ``inputs``: R CUDA bf16 tensors, rank r's token slice [count_r, hidden]
    with the counts of ``rs_token_split(T, R, r)``; the outputs have T rows.
    """
    ins = [_dev(x, "inputs[%d]" % i, torch.bfloat16) for i, x in enumerate(inputs)]
    R = len(ins)
    hidden = q_lora_rank + kv_lora_rank + qk_rope_head_dim
    T = sum(int(x.shape[0]) for x in ins)
    for r, x in enumerate(ins):
        if x.dim() != 2 or x.shape != (rs_token_split(T, R, r)[1], hidden) or not x.is_contiguous():
            raise ValueError("inputs[r] must be a contiguous [count_r, hidden] slice (rs_token_split counts)")
    for name, t in (("x_gamma", x_gamma), ("y_gamma", y_gamma), ("allgather_out", allgather_out),
                    ("x_norm_out", x_norm_out), ("y_norm_out", y_norm_out), ("quant_out", quant_out),
                    ("scale_out", scale_out)):
        if t is not None:
            _dev(t, name)
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
    arr = (ctypes.c_void_p * R)(*[x.data_ptr() for x in ins])
    _check(library().ts_allgather_fused_norm(int(ag_pattern), arr, R, T, hidden, q_lora_rank, kv_lora_rank,
                                             qk_rope_head_dim, _ptr(x_gamma), _ptr(y_gamma), float(x_eps),
                                             float(y_eps), _ptr(allgather_out), _ptr(x_norm_out),
                                             _ptr(y_norm_out), _ptr(quant_out), _ptr(scale_out),
                                             TS_FLAG_PDL if launch_with_pdl else 0, _stream(stream)))


def ts_qk_norm_sharded(shards, q_shard: int, k_shard: int, q_weight: torch.Tensor,
                       k_weight: torch.Tensor, eps: float = 1e-6, q_out: torch.Tensor | None = None,
                       k_out: torch.Tensor | None = None, launch_with_pdl: bool = False, stream=None):
    """Sharded MiniMax QK-RMSNorm (see include/ts_fused_norm.h).

    ``shards``: R CUDA bf16 tensors [T, >= q_shard + k_shard] with unit column
    stride (row stride taken from ``stride(0)``), or one [R, T, row] tensor.
    Returns (q_out [T, R*q_shard], k_out [T, R*k_shard]), allocated if None.
    """
    sh = [_dev(s, "shards[%d]" % i, torch.bfloat16) for i, s in enumerate(_rows(shards, "shards"))]
    T = sh[0].shape[0]
    stride = sh[0].stride(0)
    for s in sh:
        if s.dim() != 2 or s.shape[0] != T or s.stride(1) != 1 or s.stride(0) != stride:
            raise ValueError("shards must share T and the row stride, with unit column stride")
        if s.shape[1] < q_shard + k_shard:
            raise ValueError("a shard row is narrower than q_shard + k_shard")
    R = len(sh)
    _dev(q_weight, "q_weight", torch.bfloat16)
    _dev(k_weight, "k_weight", torch.bfloat16)
    if q_out is None:
        q_out = _empty_like_place((T, R * q_shard), torch.bfloat16, sh[0])
    if k_out is None:
        k_out = _empty_like_place((T, R * k_shard), torch.bfloat16, sh[0])
    for name, t in (("q_out", q_out), ("k_out", k_out)):
        _dev(t, name, torch.bfloat16)
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{name} must be 2-D with unit column stride")
    arr = (ctypes.c_void_p * R)(*[s.data_ptr() for s in sh])
    _check(library().ts_qk_norm_sharded(arr, R, int(T), int(stride), int(q_shard), int(k_shard),
                                        _ptr(q_weight), _ptr(k_weight), float(eps), _ptr(q_out),
                                        int(q_out.stride(0)), _ptr(k_out), int(k_out.stride(0)),
                                        TS_FLAG_PDL if launch_with_pdl else 0, _stream(stream)))
    return q_out, k_out


def ts_rms_norm_sharded(shards, width: int, weight: torch.Tensor, eps: float = 1e-6,
                        out: torch.Tensor | None = None, launch_with_pdl: bool = False, stream=None):
    """Single-matrix sharded RMSNorm (see include/ts_fused_norm.h).

    ``shards``: R CUDA bf16 tensors [T, >= width] with unit column stride and a
    common row stride (or one [R, T, row] tensor); ``weight``: bf16 [R*width].
    Returns ``out`` [T, R*width] (allocated if None).
    """
    sh = [_dev(s, "shards[%d]" % i, torch.bfloat16) for i, s in enumerate(_rows(shards, "shards"))]
    T = sh[0].shape[0]
    stride = sh[0].stride(0)
    for s in sh:
        if s.dim() != 2 or s.shape[0] != T or s.stride(1) != 1 or s.stride(0) != stride:
            raise ValueError("shards must share T and the row stride, with unit column stride")
        if s.shape[1] < width:
            raise ValueError("a shard row is narrower than width")
    R = len(sh)
    _dev(weight, "weight", torch.bfloat16)
    if out is None:
        out = _empty_like_place((T, R * width), torch.bfloat16, sh[0])
    _dev(out, "out", torch.bfloat16)
    if out.dim() != 2 or out.stride(1) != 1:
        raise ValueError("out must be 2-D with unit column stride")
    arr = (ctypes.c_void_p * R)(*[s.data_ptr() for s in sh])
    _check(library().ts_rms_norm_sharded(arr, R, int(T), int(stride), int(width), _ptr(weight), float(eps),
                                         _ptr(out), int(out.stride(0)), TS_FLAG_PDL if launch_with_pdl else 0,
                                         _stream(stream)))
    return out

"""CPU oracle for the fused reduce -> residual -> RMSNorm (-> FP8/NVFP4) path and
the sharded MiniMax QK-RMSNorm.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only users.  The product library never
imports this package, and this package never imports the product.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, fp32 steps in
the pages' order, compiled without FMA contraction or fast-math).  This module
only compiles it (``build()``) and marshals numpy arrays to it.  bf16 tensors
are passed as their raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PATTERNS = {
    "kAllReduce": 0,
    "kARResidualRMSNorm": 1,
    "kARResidualRMSNormFP8Quant": 2,
    "kARResidualRMSNormFP4Quant": 3,
    "kARResidualRMSNormOutFP8Quant": 4,
    "kARResidualRMSNormOutFP4Quant": 5,
    "kARResidualRMSNormFP8BlockWiseQuant": 6,
    "kARResidualRMSNormPartialOutFP8BlockWiseQuant": 7,
    "kARResidualRMSNormPartialOut": 8,
}

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (no FMA, no fast-math)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle library and declare its symbols."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        # ORACLE_LIB lets the mutation tests load a deliberately broken copy
        lib = ctypes.CDLL(path or os.environ.get("ORACLE_LIB") or build())
        c_u16p = ctypes.POINTER(ctypes.c_uint16)
        c_u8p = ctypes.POINTER(ctypes.c_uint8)
        c_f32p = ctypes.POINTER(ctypes.c_float)
        c_i64p = ctypes.POINTER(ctypes.c_int64)
        lib.orc_bf16_encode.argtypes = [ctypes.c_float]
        lib.orc_bf16_encode.restype = ctypes.c_uint16
        lib.orc_bf16_decode.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_decode.restype = ctypes.c_float
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = ctypes.c_float
        lib.orc_e2m1_encode.argtypes = [ctypes.c_float]
        lib.orc_e2m1_encode.restype = ctypes.c_uint8
        lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e2m1_decode.restype = ctypes.c_float
        for name, outp in (("orc_bf16_encode_n", c_u16p), ("orc_e4m3_encode_n", c_u8p),
                           ("orc_e2m1_encode_n", c_u8p)):
            fn = getattr(lib, name)
            fn.argtypes = [c_f32p, ctypes.c_int64, outp]
            fn.restype = None
        lib.orc_sf_swizzled_cols.argtypes = [ctypes.c_int64]
        lib.orc_sf_swizzled_cols.restype = ctypes.c_int64
        lib.orc_sf_swizzled_rows.argtypes = [ctypes.c_int64]
        lib.orc_sf_swizzled_rows.restype = ctypes.c_int64
        lib.orc_sf_offset_swizzled_128x4.argtypes = [ctypes.c_int64] * 3
        lib.orc_sf_offset_swizzled_128x4.restype = ctypes.c_int64
        lib.orc_sf_swizzle_128x4.argtypes = [c_u8p, ctypes.c_int64, ctypes.c_int64, c_u8p]
        lib.orc_sf_swizzle_128x4.restype = None
        lib.orc_sf_swizzled8_rows.argtypes = [ctypes.c_int64]
        lib.orc_sf_swizzled8_rows.restype = ctypes.c_int64
        lib.orc_sf_offset_swizzled_8x4.argtypes = [ctypes.c_int64] * 3
        lib.orc_sf_offset_swizzled_8x4.restype = ctypes.c_int64
        lib.orc_sf_swizzle_8x4.argtypes = [c_u8p, ctypes.c_int64, ctypes.c_int64, c_u8p]
        lib.orc_sf_swizzle_8x4.restype = None
        lib.orc_fused_reduce_norm_rows.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.POINTER(c_u16p), c_u16p, c_u16p,
            ctypes.c_float, ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
            c_i64p, ctypes.c_int64, c_u16p, c_u16p, c_u16p, c_u16p, c_u8p, c_f32p, c_u8p]
        lib.orc_fused_reduce_norm_rows.restype = ctypes.c_int
        lib.orc_rs_token_split.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, c_i64p, c_i64p]
        lib.orc_rs_token_split.restype = None
        lib.orc_reducescatter_fused_norm.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.POINTER(c_u16p), ctypes.c_int64, ctypes.c_int, c_u16p, c_u16p,
            c_u16p, ctypes.c_float, ctypes.c_float, ctypes.c_int64, c_u16p, c_u16p, c_u16p, c_u8p, c_f32p, c_u8p]
        lib.orc_reducescatter_fused_norm.restype = ctypes.c_int
        lib.orc_allgather_fused_norm_rows.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.POINTER(c_u16p), ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, c_u16p, c_u16p, ctypes.c_float, ctypes.c_float, c_i64p, ctypes.c_int64, c_u16p,
            c_u16p, c_u16p, c_u8p, c_f32p]
        lib.orc_allgather_fused_norm_rows.restype = ctypes.c_int
        lib.orc_qk_norm_sharded_rows.argtypes = [
            ctypes.c_int, ctypes.POINTER(c_u16p), ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, c_u16p, c_u16p, ctypes.c_float, c_i64p, ctypes.c_int64,
            c_u16p, c_u16p]
        lib.orc_qk_norm_sharded_rows.restype = ctypes.c_int
        lib.orc_rms_norm_sharded_rows.argtypes = [
            ctypes.c_int, ctypes.POINTER(c_u16p), ctypes.c_int64, ctypes.c_int64, c_u16p,
            ctypes.c_float, c_i64p, ctypes.c_int64, c_u16p]
        lib.orc_rms_norm_sharded_rows.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 operands are passed as uint16 bit patterns"
    return a


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def bf16_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    load().orc_bf16_encode_n(_ptr(x, ctypes.c_float), x.size, _ptr(out, ctypes.c_uint16))
    return out


def bf16_decode(b) -> np.ndarray:
    lib = load()
    b = np.asarray(b, dtype=np.uint16)
    return np.array([lib.orc_bf16_decode(int(v)) for v in b.ravel()], np.float32).reshape(b.shape)


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    load().orc_e4m3_encode_n(_ptr(x, ctypes.c_float), x.size, _ptr(out, ctypes.c_uint8))
    return out


def e4m3_decode(c) -> np.ndarray:
    lib = load()
    c = np.asarray(c, dtype=np.uint8)
    return np.array([lib.orc_e4m3_decode(int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


def e2m1_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    load().orc_e2m1_encode_n(_ptr(x, ctypes.c_float), x.size, _ptr(out, ctypes.c_uint8))
    return out


def e2m1_decode(c) -> np.ndarray:
    lib = load()
    c = np.asarray(c, dtype=np.uint8)
    return np.array([lib.orc_e2m1_decode(int(v)) for v in c.ravel()], np.float32).reshape(c.shape)


# --------------------------------------------------------------------------
# NVFP4 scale-factor layouts
# --------------------------------------------------------------------------

def sf_swizzled_shape(rows: int, n_sf_cols: int) -> tuple[int, int]:
    lib = load()
    return int(lib.orc_sf_swizzled_rows(rows)), int(lib.orc_sf_swizzled_cols(n_sf_cols))


def sf_offset_swizzled_128x4(m: int, k: int, n_sf_cols: int) -> int:
    return int(load().orc_sf_offset_swizzled_128x4(m, k, n_sf_cols))


def sf_swizzle_128x4(linear: np.ndarray) -> np.ndarray:
    linear = np.ascontiguousarray(linear, dtype=np.uint8)
    rows, cols = linear.shape
    pr, pc = sf_swizzled_shape(rows, cols)
    out = np.empty(pr * pc, np.uint8)
    load().orc_sf_swizzle_128x4(_ptr(linear, ctypes.c_uint8), rows, cols, _ptr(out, ctypes.c_uint8))
    return out


def sf_swizzled8_shape(rows: int, n_sf_cols: int) -> tuple[int, int]:
    lib = load()
    return int(lib.orc_sf_swizzled8_rows(rows)), int(lib.orc_sf_swizzled_cols(n_sf_cols))


def sf_offset_swizzled_8x4(m: int, k: int, n_sf_cols: int) -> int:
    return int(load().orc_sf_offset_swizzled_8x4(m, k, n_sf_cols))


def sf_swizzle_8x4(linear: np.ndarray) -> np.ndarray:
    linear = np.ascontiguousarray(linear, dtype=np.uint8)
    rows, cols = linear.shape
    pr, pc = sf_swizzled8_shape(rows, cols)
    out = np.empty(pr * pc, np.uint8)
    load().orc_sf_swizzle_8x4(_ptr(linear, ctypes.c_uint8), rows, cols, _ptr(out, ctypes.c_uint8))
    return out


# --------------------------------------------------------------------------
# the operations
# --------------------------------------------------------------------------

def fused_reduce_norm(pattern: int, partials, residual=None, gamma=None, eps: float = 1e-6,
                      scale_factor: float = 0.0, partial_cols: int = 0, rows=None) -> dict:
    """Evaluate one AllReduceFusionPattern on the listed rows (all rows by default).

    ``partials``: uint16 array [R, T, H] or a list of R arrays [T, H] (bf16 bits).
    ``residual``: uint16 [T, H] (patterns 1-8); ``gamma``: uint16 [H].
    Returns a dict of compact outputs, one row per listed row:
    ``allreduce_out``, ``residual_out``, ``norm_out`` (uint16 [n, H]),
    ``partial_norm_out`` (uint16 [n, P]), ``quant_out`` (uint8 [n, H] e4m3 or
    [n, H/2] packed e2m1), ``block_scale_out`` (float32 [n, H/128]) and
    ``sf_out`` (uint8 LINEAR [n, H/16]), for the outputs the pattern defines.
    """
    parts = [_u16(p) for p in partials]
    R = len(parts)
    T, H = parts[0].shape
    for p in parts:
        assert p.shape == (T, H)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    if pattern != 0:
        residual = _u16(residual)
        gamma = _u16(gamma)
        assert residual.shape == (T, H) and gamma.shape == (H,)
    out = {"allreduce_out": np.empty((n, H), np.uint16)}
    if pattern != 0:
        out["residual_out"] = np.empty((n, H), np.uint16)
        out["norm_out"] = np.empty((n, H), np.uint16)
    if pattern in (7, 8):
        assert 0 < partial_cols <= H
        out["partial_norm_out"] = np.empty((n, partial_cols), np.uint16)
    if pattern in (2, 4, 6, 7):
        out["quant_out"] = np.empty((n, H), np.uint8)
    if pattern in (3, 5):
        out["quant_out"] = np.empty((n, H // 2), np.uint8)
        out["sf_out"] = np.empty((n, H // 16), np.uint8)
    if pattern in (6, 7):
        out["block_scale_out"] = np.empty((n, H // 128), np.float32)

    arr = (ctypes.POINTER(ctypes.c_uint16) * R)(*[_ptr(p, ctypes.c_uint16) for p in parts])
    g = lambda k, ct: _ptr(out.get(k), ct)  # noqa: E731
    rc = load().orc_fused_reduce_norm_rows(
        int(pattern), R, arr, _ptr(residual, ctypes.c_uint16), _ptr(gamma, ctypes.c_uint16),
        float(eps), float(scale_factor), H, int(partial_cols), _ptr(rows, ctypes.c_int64), n,
        g("allreduce_out", ctypes.c_uint16), g("residual_out", ctypes.c_uint16),
        g("norm_out", ctypes.c_uint16), g("partial_norm_out", ctypes.c_uint16),
        g("quant_out", ctypes.c_uint8), g("block_scale_out", ctypes.c_float),
        g("sf_out", ctypes.c_uint8))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (pattern %d, H %d)" % (pattern, H))
    return out


def qk_norm_sharded(shards, q_shard: int, k_shard: int, q_weight, k_weight, eps: float = 1e-6,
                    rows=None) -> tuple[np.ndarray, np.ndarray]:
    """Sharded MiniMax QK-RMSNorm on the listed tokens.

    ``shards``: R uint16 arrays [T, row_stride] (q | k | v per row).
    ``q_weight``: uint16 [R*q_shard]; ``k_weight``: uint16 [R*k_shard].
    Returns (q_out uint16 [n, R*q_shard], k_out uint16 [n, R*k_shard]).
    """
    sh = [_u16(s) for s in shards]
    R = len(sh)
    T, stride = sh[0].shape
    for s in sh:
        assert s.shape == (T, stride)
    wq, wk = _u16(q_weight), _u16(k_weight)
    assert wq.shape == (R * q_shard,) and wk.shape == (R * k_shard,)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    q_out = np.empty((n, R * q_shard), np.uint16)
    k_out = np.empty((n, R * k_shard), np.uint16)
    arr = (ctypes.POINTER(ctypes.c_uint16) * R)(*[_ptr(s, ctypes.c_uint16) for s in sh])
    rc = load().orc_qk_norm_sharded_rows(
        R, arr, stride, q_shard, k_shard, _ptr(wq, ctypes.c_uint16), _ptr(wk, ctypes.c_uint16),
        float(eps), _ptr(rows, ctypes.c_int64), n, _ptr(q_out, ctypes.c_uint16),
        _ptr(k_out, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("oracle rejected the QK arguments")
    return q_out, k_out


def rms_norm_sharded(shards, width: int, weight, eps: float = 1e-6, rows=None) -> np.ndarray:
    """Single-matrix sharded RMSNorm on the listed tokens.

    ``shards``: R uint16 arrays [T, row_stride] (the first ``width`` columns are
    the shard's slice of the hidden dim); ``weight``: uint16 [R*width].
    Returns uint16 [n, R*width] (shard r at columns r*width...).
    """
    sh = [_u16(s) for s in shards]
    R = len(sh)
    T, stride = sh[0].shape
    for s in sh:
        assert s.shape == (T, stride)
    w = _u16(weight)
    assert w.shape == (R * width,)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, R * width), np.uint16)
    arr = (ctypes.POINTER(ctypes.c_uint16) * R)(*[_ptr(s, ctypes.c_uint16) for s in sh])
    rc = load().orc_rms_norm_sharded_rows(R, arr, stride, width, _ptr(w, ctypes.c_uint16), float(eps),
                                          _ptr(rows, ctypes.c_int64), rows.size,
                                          _ptr(out, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("oracle rejected the sharded RMSNorm arguments")
    return out


RS_PATTERNS = {
    "kReduceScatter": 0,
    "kRSResidualRMSNorm": 1,
    "kRSResidualRMSNormFP8Quant": 2,
    "kRSResidualRMSNormFP4Quant": 3,
    "kRSResidualRMSNormOutFP8Quant": 4,
    "kRSResidualRMSNormOutFP4Quant": 5,
    "kRSResidualRMSNormFP8BlockWiseQuant": 6,
    "kRSAddResidualRMSNormFP8BlockWiseQuant": 7,
    "kRSAddResidualRMSNorm": 8,
}


def rs_token_split(T: int, world: int, rank: int) -> tuple[int, int]:
    start, count = ctypes.c_int64(), ctypes.c_int64()
    load().orc_rs_token_split(T, world, rank, ctypes.byref(start), ctypes.byref(count))
    return start.value, count.value


def reducescatter_fused_norm(rs_pattern: int, partials, rank: int, add_in=None, residual=None, gamma=None,
                             eps: float = 1e-6, scale_factor: float = 0.0) -> dict:
    """Rank ``rank``'s reduce-scatter fusion output, all R partials local.

    ``partials``: R uint16 arrays [T, H]; ``add_in``/``residual``: uint16 [count, H]
    for the rank's token slice; returns compact outputs ``reducescatter_out``,
    ``residual_out``, ``norm_out``, ``quant_out``, ``block_scale_out``, ``sf_out``
    (those the pattern defines) with ``count`` rows.
    """
    parts = [_u16(p) for p in partials]
    R = len(parts)
    T, H = parts[0].shape
    start, count = rs_token_split(T, R, rank)
    form = {7: 6, 8: 1}.get(rs_pattern, rs_pattern)
    out = {"reducescatter_out": np.empty((count, H), np.uint16)}
    if form != 0:
        residual = _u16(residual)
        gamma = _u16(gamma)
        assert residual.shape == (count, H) and gamma.shape == (H,)
        out["residual_out"] = np.empty((count, H), np.uint16)
        out["norm_out"] = np.empty((count, H), np.uint16)
    if rs_pattern in (7, 8):
        add_in = _u16(add_in)
        assert add_in.shape == (count, H)
    else:
        add_in = None
    if form in (2, 4, 6):
        out["quant_out"] = np.empty((count, H), np.uint8)
    if form in (3, 5):
        out["quant_out"] = np.empty((count, H // 2), np.uint8)
        out["sf_out"] = np.empty((count, H // 16), np.uint8)
    if form == 6:
        out["block_scale_out"] = np.empty((count, H // 128), np.float32)
    arr = (ctypes.POINTER(ctypes.c_uint16) * R)(*[_ptr(p, ctypes.c_uint16) for p in parts])
    g = lambda k, ct: _ptr(out.get(k), ct)  # noqa: E731
    rc = load().orc_reducescatter_fused_norm(
        int(rs_pattern), R, arr, T, int(rank), _ptr(add_in, ctypes.c_uint16), _ptr(residual, ctypes.c_uint16),
        _ptr(gamma, ctypes.c_uint16), float(eps), float(scale_factor), H,
        g("reducescatter_out", ctypes.c_uint16), g("residual_out", ctypes.c_uint16),
        g("norm_out", ctypes.c_uint16), g("quant_out", ctypes.c_uint8), g("block_scale_out", ctypes.c_float),
        g("sf_out", ctypes.c_uint8))
    if rc != 0:
        raise ValueError("oracle rejected the reduce-scatter arguments")
    return out


AG_PATTERNS = {"kAllGather": 0, "kAllGatherfusedRMS": 1, "kAllGatherfusedRMSFP8BlockWiseQuant": 2}


def allgather_fused_norm(pattern: int, inputs, q_lora_rank: int, kv_lora_rank: int, x_gamma=None, y_gamma=None,
                         x_eps: float = 1e-6, y_eps: float = 1e-6, rows=None) -> dict:
    """All-gather fusion with the dual MLA RMSNorm on the listed gathered rows.

    ``inputs``: R uint16 arrays [count_r, hidden] (rank r's token slice, the
    counts of ``rs_token_split``).  Returns compact ``allgather_out`` [n, hidden]
    and, by pattern, ``x_norm_out`` [n, q], ``y_norm_out`` [n, kv], ``quant_out``
    uint8 [n, q], ``scale_out`` float32 [n, q/128].
    """
    ins = [_u16(x) for x in inputs]
    R = len(ins)
    hidden = ins[0].shape[1]
    T = sum(x.shape[0] for x in ins)
    for r, x in enumerate(ins):
        assert x.shape == (rs_token_split(T, R, r)[1], hidden)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    q, kv = q_lora_rank, kv_lora_rank
    out = {"allgather_out": np.empty((n, hidden), np.uint16)}
    if pattern in (1, 2):
        x_gamma, y_gamma = _u16(x_gamma), _u16(y_gamma)
        assert x_gamma.shape == (q,) and y_gamma.shape == (kv,)
        out["x_norm_out"] = np.empty((n, q), np.uint16)
        out["y_norm_out"] = np.empty((n, kv), np.uint16)
    if pattern == 2:
        out["quant_out"] = np.empty((n, q), np.uint8)
        out["scale_out"] = np.empty((n, q // 128), np.float32)
    arr = (ctypes.POINTER(ctypes.c_uint16) * R)(*[_ptr(x, ctypes.c_uint16) for x in ins])
    g = lambda k, ct: _ptr(out.get(k), ct)  # noqa: E731
    rc = load().orc_allgather_fused_norm_rows(
        int(pattern), R, arr, T, hidden, q, kv, _ptr(x_gamma, ctypes.c_uint16), _ptr(y_gamma, ctypes.c_uint16),
        float(x_eps), float(y_eps), _ptr(rows, ctypes.c_int64), n, g("allgather_out", ctypes.c_uint16),
        g("x_norm_out", ctypes.c_uint16), g("y_norm_out", ctypes.c_uint16), g("quant_out", ctypes.c_uint8),
        g("scale_out", ctypes.c_float))
    if rc != 0:
        raise ValueError("oracle rejected the all-gather arguments")
    return out

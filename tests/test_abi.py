"""The C ABI without a GPU: the library loads, exports every function the header
declares, and rejects bad arguments on the host before any launch.

Every negative case below carries exactly one defect that the host checks
catch, so no kernel is ever launched (the pointers are fake addresses that are
never dereferenced).  The one accepted case has T = 0, which validates and
returns without launching.
"""
import ctypes
import os
import re

import pytest

import reduce_residual_rmsnorm_gb300 as pkg
from reduce_residual_rmsnorm_gb300 import build as libbuild
from reduce_residual_rmsnorm_gb300._binding import TsOuts

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TS_OK, BAD_PATTERN, NULL, SHAPE, ALIGN, UNSUPPORTED, ALIAS = 0, -1, -2, -3, -4, -5, -6
MiB = 1 << 20


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return pkg.library()


def _header_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\bTS_API\s+[\w\s\*]*?\b(ts_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_api():
    assert _header_functions() == sorted(pkg.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in ((0, "TS_OK"), (-1, "TS_ERR_BAD_PATTERN"), (-2, "TS_ERR_NULL"), (-3, "TS_ERR_SHAPE"),
                       (-4, "TS_ERR_ALIGN"), (-5, "TS_ERR_UNSUPPORTED"), (-6, "TS_ERR_ALIAS"),
                       (-7, "TS_ERR_LAUNCH"), (-99, "TS_ERR_UNKNOWN")):
        assert lib.ts_status_string(code).decode() == name


# ---------------------------------------------------------------------------
# ts_fused_reduce_norm
# ---------------------------------------------------------------------------

class Fake:
    """Distinct, 16-byte aligned, non-overlapping fake device addresses."""

    def __init__(self):
        self.next = 0x7F0000000000

    def __call__(self, nbytes=64 * MiB):
        p = self.next
        self.next += (nbytes + 4095) // 4096 * 4096 + 4096
        return p


def _fused_call(lib, pattern=1, R=2, T=16, H=256, P=0, sf_layout=2, flags=0, mutate=None):
    f = Fake()
    parts = [f() for _ in range(R)]
    args = dict(pattern=pattern, partials=parts, R=R, residual=f(), gamma=f(), eps=1e-6,
                scale_factor=f(), T=T, H=H, flags=flags)
    table = {0: "R-----", 1: "oRR---", 2: "oR--R-", 3: "oR--RR", 4: "oRR-R-", 5: "oRR-RR",
             6: "oR--RR", 7: "oR-RRR", 8: "oRoR--"}
    row = table.get(pattern, "oRR---")
    keys = ["allreduce_out", "residual_out", "norm_out", "partial_norm_out", "quant_out", "scale_out"]
    outs = {k: (f() if row[i] == "R" else None) for i, k in enumerate(keys)}
    outs["partial_cols"] = P
    outs["sf_layout"] = sf_layout
    outs["reserved"] = 0
    if mutate:
        mutate(args, outs)
    o = TsOuts(outs["allreduce_out"], outs["residual_out"], outs["norm_out"], outs["partial_norm_out"],
               outs["partial_cols"], outs["quant_out"], outs["scale_out"], outs["sf_layout"], outs["reserved"])
    parts = args["partials"]
    arr = None if parts is None else (ctypes.c_void_p * len(parts))(*parts)
    st = lib.ts_fused_reduce_norm(args["pattern"], arr, args["R"], args["residual"], args["gamma"],
                                  args["eps"], args["scale_factor"], args["T"], args["H"],
                                  ctypes.byref(o), args["flags"], None)
    return st, lib.ts_last_error_detail().decode()


def test_zero_rows_is_a_valid_no_op(lib):
    for pattern, H, P in ((0, 256, 0), (1, 256, 0), (2, 256, 0), (3, 256, 0), (5, 256, 0), (6, 256, 0),
                          (7, 256, 128), (8, 256, 64)):
        st, detail = _fused_call(lib, pattern=pattern, T=0, H=H, P=P)
        assert st == TS_OK, (pattern, detail)


def _set(path, value):
    def m(args, outs):
        (args if path in args else outs)[path] = value
    return m


NEG_FUSED = [
    ("pattern -1", dict(pattern=-1), BAD_PATTERN),
    ("pattern 9", dict(pattern=9), BAD_PATTERN),
    ("R = 0", dict(mutate=lambda a, o: a.update(R=0)), SHAPE),
    ("R = 17", dict(R=17), SHAPE),
    ("T < 0", dict(T=-1), SHAPE),
    ("H = 0", dict(H=0), SHAPE),
    ("H % 8", dict(H=100), SHAPE),
    ("H too large", dict(H=16392), UNSUPPORTED),
    ("blockwise H % 128", dict(pattern=6, H=192), SHAPE),
    ("fp4 H % 16", dict(pattern=3, H=200), SHAPE),
    ("partials NULL", dict(mutate=_set("partials", None)), NULL),
    ("a partial NULL", dict(mutate=lambda a, o: a["partials"].__setitem__(1, None)), NULL),
    ("partial misaligned", dict(mutate=lambda a, o: a["partials"].__setitem__(0, a["partials"][0] + 2)), ALIGN),
    ("residual NULL", dict(mutate=_set("residual", None)), NULL),
    ("gamma NULL", dict(mutate=_set("gamma", None)), NULL),
    ("gamma misaligned", dict(mutate=lambda a, o: a.update(gamma=a["gamma"] + 8)), ALIGN),
    ("scale NULL fp8", dict(pattern=2, mutate=_set("scale_factor", None)), NULL),
    ("scale NULL fp4", dict(pattern=3, mutate=_set("scale_factor", None)), NULL),
    ("scale misaligned", dict(pattern=2, mutate=lambda a, o: a.update(scale_factor=a["scale_factor"] + 2)), ALIGN),
    ("residual_out NULL", dict(mutate=_set("residual_out", None)), NULL),
    ("norm_out NULL", dict(mutate=_set("norm_out", None)), NULL),
    ("allreduce_out NULL p0", dict(pattern=0, mutate=_set("allreduce_out", None)), NULL),
    ("quant_out NULL", dict(pattern=6, mutate=_set("quant_out", None)), NULL),
    ("scale_out NULL", dict(pattern=3, mutate=_set("scale_out", None)), NULL),
    ("partial_out NULL", dict(pattern=8, P=64, mutate=_set("partial_norm_out", None)), NULL),
    ("norm_out given to p2", dict(pattern=2, mutate=_set("norm_out", 0x10000)), UNSUPPORTED),
    ("residual_out given to p0", dict(pattern=0, mutate=_set("residual_out", 0x10000)), UNSUPPORTED),
    ("quant_out given to p1", dict(pattern=1, mutate=_set("quant_out", 0x10000)), UNSUPPORTED),
    ("out misaligned", dict(mutate=lambda a, o: o.update(norm_out=o["norm_out"] + 4)), ALIGN),
    ("scale_out misaligned", dict(pattern=6, mutate=lambda a, o: o.update(scale_out=o["scale_out"] + 2)), ALIGN),
    ("partial_cols 0", dict(pattern=8, P=0), SHAPE),
    ("partial_cols > H", dict(pattern=8, P=264), SHAPE),
    ("partial_cols % 8", dict(pattern=7, P=100), SHAPE),
    ("sf layout 7", dict(pattern=5, sf_layout=7), BAD_PATTERN),
    ("reserved", dict(mutate=_set("reserved", 1)), UNSUPPORTED),
    ("unknown flag", dict(flags=8), UNSUPPORTED),
    ("outputs overlap", dict(mutate=lambda a, o: o.update(norm_out=o["residual_out"] + 16)), ALIAS),
    ("output overlaps partial", dict(mutate=lambda a, o: o.update(norm_out=a["partials"][1])), ALIAS),
    ("allreduce_out inside partial 0", dict(pattern=0, mutate=lambda a, o: o.update(
        allreduce_out=a["partials"][0] + 256)), ALIAS),
    ("allreduce_out == partials[1]", dict(pattern=0, mutate=lambda a, o: o.update(
        allreduce_out=a["partials"][1])), ALIAS),
    ("norm_out == residual", dict(mutate=lambda a, o: o.update(norm_out=a["residual"])), ALIAS),
    ("output overlaps gamma", dict(mutate=lambda a, o: o.update(residual_out=a["gamma"])), ALIAS),
]


@pytest.mark.parametrize("name,kw,want", NEG_FUSED, ids=[c[0] for c in NEG_FUSED])
def test_fused_rejects(lib, name, kw, want):
    st, detail = _fused_call(lib, **kw)
    assert st == want, (name, st, detail)
    assert detail, "a failure must explain itself"


def test_zero_rows_accepts_null_row_buffers(lib):
    def nullify(a, o):
        a["partials"] = [None] * len(a["partials"])
        a["residual"] = None
        for k in ("allreduce_out", "residual_out", "norm_out", "quant_out", "scale_out"):
            o[k] = None
    st, d = _fused_call(lib, pattern=1, T=0, mutate=nullify)
    assert st == TS_OK, d
    st, d = _fused_call(lib, pattern=1, T=1, mutate=nullify)
    assert st == NULL, d
    st, d = _qk_call(lib, T=0, mutate=lambda a: a.update(shards=[None] * 8, q_out=None, k_out=None))
    assert st == TS_OK, d
    st, d = _qk_call(lib, T=0, mutate=lambda a: a.update(wq=None))
    assert st == NULL, d


def test_in_place_aliases_are_accepted(lib):
    # allreduce_out == partials[0] and residual_out == residual pass validation
    # (checked with T = 0 so nothing launches)
    st, d = _fused_call(lib, pattern=0, T=0, mutate=lambda a, o: o.update(allreduce_out=a["partials"][0]))
    assert st == TS_OK, d
    st, d = _fused_call(lib, pattern=1, T=0, mutate=lambda a, o: o.update(residual_out=a["residual"]))
    assert st == TS_OK, d


# ---------------------------------------------------------------------------
# ts_qk_norm_sharded
# ---------------------------------------------------------------------------

def _qk_call(lib, R=8, T=4, stride=1280, Q=1024, K=128, ldq=None, ldk=None, flags=0, mutate=None):
    f = Fake()
    a = dict(shards=[f() for _ in range(R)], R=R, T=T, stride=stride, Q=Q, K=K, wq=f(), wk=f(),
             q_out=f(), ldq=R * Q if ldq is None else ldq, k_out=f(), ldk=R * K if ldk is None else ldk,
             flags=flags)
    if mutate:
        mutate(a)
    arr = None if a["shards"] is None else (ctypes.c_void_p * len(a["shards"]))(*a["shards"])
    st = lib.ts_qk_norm_sharded(arr, a["R"], a["T"], a["stride"], a["Q"], a["K"], a["wq"], a["wk"], 1e-6,
                                a["q_out"], a["ldq"], a["k_out"], a["ldk"], a["flags"], None)
    return st, lib.ts_last_error_detail().decode()


def _rms_call(lib, R=8, T=4, stride=768, W=768, ldo=None, flags=0, mutate=None):
    f = Fake()
    a = dict(shards=[f() for _ in range(R)], R=R, T=T, stride=stride, W=W, w=f(), out=f(),
             ldo=R * W if ldo is None else ldo, flags=flags)
    if mutate:
        mutate(a)
    arr = None if a["shards"] is None else (ctypes.c_void_p * len(a["shards"]))(*a["shards"])
    st = lib.ts_rms_norm_sharded(arr, a["R"], a["T"], a["stride"], a["W"], a["w"], 1e-6, a["out"], a["ldo"],
                                 a["flags"], None)
    return st, lib.ts_last_error_detail().decode()


def test_qk_zero_tokens_is_valid(lib):
    assert _qk_call(lib, T=0)[0] == TS_OK


NEG_QK = [
    ("shards NULL", dict(mutate=lambda a: a.update(shards=None)), NULL),
    ("R 0", dict(mutate=lambda a: a.update(R=0)), SHAPE),
    ("R 17", dict(R=17, stride=1280), SHAPE),
    ("T < 0", dict(T=-5), SHAPE),
    ("Q % 8", dict(Q=1020), SHAPE),
    ("K 0", dict(K=0), SHAPE),
    ("Q too big", dict(Q=4104, stride=8192), UNSUPPORTED),
    ("K too big", dict(K=1032, stride=8192), UNSUPPORTED),
    ("stride small", dict(stride=1144), SHAPE),
    ("stride % 8", dict(stride=1284), SHAPE),
    ("ldq small", dict(ldq=1024 * 8 - 8), SHAPE),
    ("ldk % 8", dict(ldk=128 * 8 + 4), SHAPE),
    ("shard NULL", dict(mutate=lambda a: a["shards"].__setitem__(3, None)), NULL),
    ("shard misaligned", dict(mutate=lambda a: a["shards"].__setitem__(3, a["shards"][3] + 8)), ALIGN),
    ("wq NULL", dict(mutate=lambda a: a.update(wq=None)), NULL),
    ("k_out misaligned", dict(mutate=lambda a: a.update(k_out=a["k_out"] + 2)), ALIGN),
    ("q_out overlaps k_out", dict(mutate=lambda a: a.update(k_out=a["q_out"] + 64)), ALIAS),
    ("q_out overlaps a shard", dict(mutate=lambda a: a.update(q_out=a["shards"][2] + 1024)), ALIAS),
    ("k_out overlaps wk", dict(mutate=lambda a: a.update(k_out=a["wk"])), ALIAS),
    ("K 0 (use the single-matrix call)", dict(K=0), SHAPE),
    ("unknown flag", dict(flags=4), UNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,want", NEG_QK, ids=[c[0] for c in NEG_QK])
def test_qk_rejects(lib, name, kw, want):
    st, detail = _qk_call(lib, **kw)
    assert st == want, (name, st, detail)
    assert detail


def test_binding_requires_cuda_or_pinned_tensors():
    """Pageable host tensors are refused (only GPU and pinned host memory are
    addressable by the kernels); pinned host tensors are accepted (on a GPU
    box, tests/test_gpu_fused.py runs them)."""
    import torch

    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    assert not x.is_pinned()
    with pytest.raises(TypeError, match="pinned host tensor"):
        pkg.ts_fused_reduce_norm(0, [x], allreduce_out=x)
    with pytest.raises(TypeError):
        pkg.ts_rms_norm_sharded([x], 64, x[0], 1e-6)


def test_rms_zero_tokens_is_valid(lib):
    assert _rms_call(lib, T=0)[0] == TS_OK
    assert _rms_call(lib, T=0, mutate=lambda a: a.update(shards=[None] * 8, out=None))[0] == TS_OK


NEG_RMS = [
    ("shards NULL", dict(mutate=lambda a: a.update(shards=None)), NULL),
    ("R 0", dict(mutate=lambda a: a.update(R=0)), SHAPE),
    ("W % 8", dict(W=100, stride=104), SHAPE),
    ("W too big", dict(W=4104, stride=4104), UNSUPPORTED),
    ("stride < W", dict(stride=760), SHAPE),
    ("ldo small", dict(ldo=768 * 8 - 8), SHAPE),
    ("weight NULL", dict(mutate=lambda a: a.update(w=None)), NULL),
    ("out NULL", dict(mutate=lambda a: a.update(out=None)), NULL),
    ("out misaligned", dict(mutate=lambda a: a.update(out=a["out"] + 2)), ALIGN),
    ("out overlaps a shard", dict(mutate=lambda a: a.update(out=a["shards"][0])), ALIAS),
    ("out overlaps weight", dict(mutate=lambda a: a.update(out=a["w"] - 64)), ALIAS),
    ("unknown flag", dict(flags=8), UNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,want", NEG_RMS, ids=[c[0] for c in NEG_RMS])
def test_rms_rejects(lib, name, kw, want):
    st, detail = _rms_call(lib, **kw)
    assert st == want, (name, st, detail)
    assert detail


def test_pdl_flag_accepted(lib):
    assert _fused_call(lib, T=0, flags=1)[0] == TS_OK
    assert _qk_call(lib, T=0, flags=1)[0] == TS_OK
    assert _rms_call(lib, T=0, flags=1)[0] == TS_OK


def test_early_read_flag_only_on_the_fused_forms(lib):
    """TS_FLAG_PDL_EARLY_READ (2) and TS_FLAG_PDL_INDEPENDENT (4) belong to the
    fused and reduce-scatter entry points; the sharded norms reject them."""
    assert _fused_call(lib, T=0, flags=3)[0] == TS_OK
    assert _fused_call(lib, T=0, flags=2)[0] == TS_OK
    assert _fused_call(lib, T=0, flags=5)[0] == TS_OK
    assert _rs_call(lib, T=0, flags=3)[0] == TS_OK
    assert _rs_call(lib, T=0, flags=5)[0] == TS_OK
    assert _qk_call(lib, T=0, flags=3)[0] == UNSUPPORTED
    assert _rms_call(lib, T=0, flags=2)[0] == UNSUPPORTED
    assert _qk_call(lib, T=0, flags=5)[0] == UNSUPPORTED
    assert _fused_call(lib, T=0, flags=8)[0] == UNSUPPORTED


# ---------------------------------------------------------------------------
# ts_reducescatter_fused_norm
# ---------------------------------------------------------------------------

def _rs_call(lib, rs=8, R=4, rank=0, T=16, H=256, add=True, flags=0, mutate=None):
    f = Fake()
    parts = [f() for _ in range(R)]
    a = dict(rs=rs, partials=parts, R=R, rank=rank, add_in=f() if add else None, residual=f(), gamma=f(),
             sf=f(), T=T, H=H, flags=flags)
    form = {7: 6, 8: 1}.get(rs, rs)
    table = {0: "R-----", 1: "oRR---", 2: "oR--R-", 3: "oR--RR", 4: "oRR-R-", 5: "oRR-RR", 6: "oR--RR"}
    row = table.get(form, "oRR---")
    keys = ["allreduce_out", "residual_out", "norm_out", "partial_norm_out", "quant_out", "scale_out"]
    outs = {k: (f() if row[i] == "R" else None) for i, k in enumerate(keys)}
    if mutate:
        mutate(a, outs)
    o = TsOuts(outs["allreduce_out"], outs["residual_out"], outs["norm_out"], outs["partial_norm_out"], 0,
               outs["quant_out"], outs["scale_out"], 2, 0)
    arr = None if a["partials"] is None else (ctypes.c_void_p * len(a["partials"]))(*a["partials"])
    st = lib.ts_reducescatter_fused_norm(a["rs"], arr, a["R"], a["rank"], a["add_in"], a["residual"], a["gamma"],
                                         1e-6, a["sf"], a["T"], a["H"], ctypes.byref(o), a["flags"], None)
    return st, lib.ts_last_error_detail().decode()


def test_rs_valid_empty_calls(lib):
    assert _rs_call(lib, T=0)[0] == TS_OK
    assert _rs_call(lib, T=0, rank=-1)[0] == TS_OK
    assert _rs_call(lib, T=2, R=4, rank=3)[0] == TS_OK  # rank 3 of 4 owns no token of 2


NEG_RS = [
    ("rs pattern 9", dict(rs=9), BAD_PATTERN),
    ("rank -2", dict(rank=-2), SHAPE),
    ("rank == R", dict(rank=4), SHAPE),
    ("add_in missing for 8", dict(add=False), NULL),
    ("add_in missing for 7", dict(rs=7, add=False), NULL),
    ("add_in given for 1", dict(rs=1, add=True), UNSUPPORTED),
    ("add_in misaligned", dict(mutate=lambda a, o: a.update(add_in=a["add_in"] + 4)), ALIGN),
    ("partial out given", dict(mutate=lambda a, o: o.update(partial_norm_out=0x10000)), UNSUPPORTED),
    ("output overlaps add_in", dict(mutate=lambda a, o: o.update(norm_out=a["add_in"])), ALIAS),
    ("H % 8", dict(H=100), SHAPE),
    ("partials NULL", dict(mutate=lambda a, o: a.update(partials=None)), NULL),
]


@pytest.mark.parametrize("name,kw,want", NEG_RS, ids=[c[0] for c in NEG_RS])
def test_rs_rejects(lib, name, kw, want):
    st, detail = _rs_call(lib, **kw)
    assert st == want, (name, st, detail)
    assert detail


# ---------------------------------------------------------------------------
# ts_allgather_fused_norm
# ---------------------------------------------------------------------------

def _ag_call(lib, pat=1, R=8, T=64, q=1536, kv=512, rope=64, hidden=None, flags=0, mutate=None):
    f = Fake()
    a = dict(pat=pat, inputs=[f() for _ in range(R)], R=R, T=T, hidden=q + kv + rope if hidden is None else hidden,
             q=q, kv=kv, rope=rope, xg=f(), yg=f(), flags=flags)
    table = {0: "R----", 1: "RRR--", 2: "RoRRR"}
    keys = ["allgather_out", "x_norm_out", "y_norm_out", "quant_out", "scale_out"]
    outs = {k: (f() if table.get(pat, "RRR--")[i] == "R" else None) for i, k in enumerate(keys)}
    if mutate:
        mutate(a, outs)
    arr = None if a["inputs"] is None else (ctypes.c_void_p * len(a["inputs"]))(*a["inputs"])
    st = lib.ts_allgather_fused_norm(a["pat"], arr, a["R"], a["T"], a["hidden"], a["q"], a["kv"], a["rope"],
                                     a["xg"], a["yg"], 1e-6, 1e-6, *[outs[k] for k in keys], a["flags"], None)
    return st, lib.ts_last_error_detail().decode()


def test_ag_valid_empty_calls(lib):
    for pat in (0, 1, 2):
        assert _ag_call(lib, pat=pat, T=0)[0] == TS_OK
    st, d = _ag_call(lib, pat=1, T=0, mutate=lambda a, o: (a.update(inputs=[None] * 8),
                                                          o.update(allgather_out=None, x_norm_out=None,
                                                                   y_norm_out=None)))
    assert st == TS_OK, d


NEG_AG = [
    ("pattern 3", dict(pat=3), BAD_PATTERN),
    ("inputs NULL", dict(mutate=lambda a, o: a.update(inputs=None)), NULL),
    ("R 17", dict(R=17), SHAPE),
    ("q % 128", dict(q=1544, hidden=1544 + 512 + 64), SHAPE),
    ("kv % 8", dict(kv=500, hidden=1536 + 500 + 64), SHAPE),
    ("segments != hidden", dict(hidden=2104), SHAPE),
    ("hidden > 2112", dict(q=1664, hidden=1664 + 512 + 64), SHAPE),
    ("an input NULL", dict(mutate=lambda a, o: a["inputs"].__setitem__(2, None)), NULL),
    ("input misaligned", dict(mutate=lambda a, o: a["inputs"].__setitem__(2, a["inputs"][2] + 8)), ALIGN),
    ("x_gamma NULL", dict(mutate=lambda a, o: a.update(xg=None)), NULL),
    ("allgather_out NULL", dict(mutate=lambda a, o: o.update(allgather_out=None)), NULL),
    ("y_norm_out NULL p2", dict(pat=2, mutate=lambda a, o: o.update(y_norm_out=None)), NULL),
    ("quant_out given to p1", dict(mutate=lambda a, o: o.update(quant_out=0x10000)), UNSUPPORTED),
    ("x_norm_out given to p0", dict(pat=0, mutate=lambda a, o: o.update(x_norm_out=0x10000)), UNSUPPORTED),
    ("scale_out misaligned", dict(pat=2, mutate=lambda a, o: o.update(scale_out=o["scale_out"] + 2)), ALIGN),
    ("x_norm overlaps y_norm", dict(mutate=lambda a, o: o.update(y_norm_out=o["x_norm_out"] + 64)), ALIAS),
    ("output overlaps an input", dict(mutate=lambda a, o: o.update(allgather_out=a["inputs"][3])), ALIAS),
    ("unknown flag", dict(flags=2), UNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,want", NEG_AG, ids=[c[0] for c in NEG_AG])
def test_ag_rejects(lib, name, kw, want):
    st, detail = _ag_call(lib, **kw)
    assert st == want, (name, st, detail)
    assert detail

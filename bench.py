"""Throughput of the fused reduce -> residual -> RMSNorm (+quant) path on GB300.

One step = one ``ts_fused_reduce_norm`` call of
kARResidualRMSNormPartialOutFP8BlockWiseQuant (pattern 7: residual_out, the
first 1024 columns of the bf16 norm, FP8 E4M3 codes and fp32 1x128 block
scales) over the largest workload, R=8, T=8192, H=7168 (bf16 partials
N(0, 0.5^2), residual N(0, 1), 0.1 % of the partial and residual entries x50,
gamma U(0.5, 1.5), seed 0), inputs resident in HBM, launched with the pages'
``launch_with_pdl`` option (programmatic dependent launch: each call still
waits for the previous one to complete before touching memory).  Consecutive
steps alternate between two copies of the inputs and outputs, so no step
touches a cache line the step before it touched.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``value`` is tokens (rows) per second over all ranks (each rank runs the
same per-GPU workload: weak scaling, no collective on the data path).
``--gpus N`` without torchrun starts N ranks itself through
torch.distributed.run; under torchrun it must equal WORLD_SIZE.  The line
also carries the roofline of the kernel (algorithmic bytes / CUDA-event time
against the measured HBM copy bandwidth), an end-to-end figure through the
C ABI with host buffers (the call given pinned host inputs and outputs, which
the kernel reads and writes across the host link; the staged-copy form beside
it), the host time of one C-ABI call from a C caller, the CPU oracle timed on
a bounded sample of rows, the SM clocks sampled during the timed region, and
``rows``: the other patterns and workloads timed the same way (kAllReduce and
kARResidualRMSNorm on R=8, T=4096; FP8 per-tensor, FP8 1x128 blockwise,
PartialOut on R=8, T=8192; NVFP4 on R=4, T=16384, H=5120 in the three SF
layouts; tensor-parallel degrees 1, 2 and 4 on T=16384, H=5120; the
reduce-scatter and all-gather forms; the sharded MiniMax QK-norm and
single-matrix norm on R=8, T=32768; and the R=2, T=16 latency case).  Rows
launch with ``launch_with_pdl`` too, except those labelled "(plain launch)"
and the reduce-scatter calls on concurrent streams.

Every timed region starts behind a short spin kernel queued on the stream, so
that the host has enqueued the region's launches before its start event
runs: the region then measures the GPU executing them back to back, not the
host's enqueue latency of its first call.

``--impl reference`` times the CPU oracle instead (host cores, bounded samples
of the same workload per step); under torchrun only rank 0 runs it.
``--sweep-t`` prints only the per-call time of single fused calls against T,
with the inputs cold in L2 (one JSON line per shape and T).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused reduce+RMSNorm(+quant) tokens/s and achieved HBM GB/s vs 8 TB/s, 1×GB300"
HEADLINE = {"key": "C3", "pattern": 7, "partial_cols": 1024}
WORKLOAD = ("kARResidualRMSNormPartialOutFP8BlockWiseQuant R=8 T=8192 H=7168 P=1024: bf16 partials "
            "~N(0,0.5^2), residual ~N(0,1), 0.1% of partial and residual entries x50, gamma ~U(0.5,1.5), "
            "eps 1e-6, seed 0")
NSETS = 2  # copies of each workload's buffers, alternated between consecutive launches
EPS = 1e-6
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 10 ** 6


# ---------------------------------------------------------------------------
# algorithmic bytes (reads of R partials + residual, gamma once, all outputs)
# ---------------------------------------------------------------------------

def fused_bytes(pattern: int, R: int, T: int, H: int, P: int = 0, sf_layout: int = 2,
                allreduce_out: bool = False) -> int:
    p = int(pattern)
    rb = T * R * H * 2
    wb = 0
    if p == 0 or allreduce_out:
        wb += T * H * 2
    if p != 0:
        rb += T * H * 2 + H * 2  # residual, gamma
        wb += T * H * 2          # residual_out
    if 2 <= p <= 5:
        rb += 4                  # scale_factor
    if p in (1, 4, 5):
        wb += T * H * 2          # norm_out
    if p in (7, 8):
        wb += T * P * 2          # partial_norm_out
    if p in (2, 4, 6, 7):
        wb += T * H              # e4m3 codes
    if p in (6, 7):
        wb += T * (H // 128) * 4
    if p in (3, 5):
        wb += T * H // 2
        if sf_layout == 2:  # LINEAR
            wb += T * (H // 16)
        else:               # SWIZZLED_128x4 / SWIZZLED_8x4, padding included
            tile = 128 if sf_layout == 0 else 8
            wb += ((T + tile - 1) // tile * tile) * ((H // 16 + 3) // 4 * 4)
    return rb + wb


def qk_bytes(R: int, T: int, Q: int, K: int) -> int:
    return T * R * (Q + K) * 2 * 2 + R * (Q + K) * 2


def rs_add_bytes(R: int, T: int, H: int, fp8_block: bool = False) -> int:
    """kRSAddResidualRMSNorm(FP8BlockWise) over all R ranks' slices (R calls):
    the partials' rows, add_in, residual, gamma once per call, and the outputs."""
    rb = T * R * H * 2 + 2 * T * H * 2 + R * H * 2
    wb = T * H * 2 + (T * H + T * (H // 128) * 4 if fp8_block else T * H * 2)
    return rb + wb


def ag_bytes(pattern: int, T: int, q: int, kv: int, rope: int) -> int:
    """All-gather dual norm: read every row once, write the gathered copy and the
    pattern's outputs (pattern 2 here without the optional bf16 x norm)."""
    hidden = q + kv + rope
    b = T * hidden * 2 * 2
    if pattern == 1:
        b += T * (q + kv) * 2 + (q + kv) * 2
    elif pattern == 2:
        b += T * kv * 2 + T * q + T * (q // 128) * 4 + (q + kv) * 2
    return b


def rms_sharded_bytes(R: int, T: int, W: int) -> int:
    return T * R * W * 2 * 2 + R * W * 2


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def read_peaks() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = ("ag_norm.cu", "device_util.cuh", "fused_rows.cu", "int_div.h", "launch.h", "qk_norm.cu",
                  "sf_layout.cuh")
# the device sources each kernel family is built from
KERNEL_FAMILIES = {
    "fused_rows": ("device_util.cuh", "fused_rows.cu", "launch.h", "sf_layout.cuh"),
    "qk_norm": ("device_util.cuh", "int_div.h", "launch.h", "qk_norm.cu"),
    "ag_norm": ("ag_norm.cu", "device_util.cuh", "int_div.h", "launch.h"),
}


def _code_tokens(text: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed, so
    that rewording a comment does not change the hash (string and character
    literals are kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif text[i] in "\"'":
            j = i + 1
            while j < n and text[j] != text[i]:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(files=KERNEL_SOURCES, read=None) -> str:
    """Hash of device sources (by default all of them; not the host-side
    argument checks), comments and layout excluded.  ``read(name)`` returns a
    file's text (default: the file under csrc/)."""
    csrc = os.path.join(ROOT, "reduce_residual_rmsnorm_gb300", "csrc")
    if read is None:
        def read(fn):
            with open(os.path.join(csrc, fn), encoding="utf-8") as f:
                return f.read()
    h = hashlib.sha256()
    for fn in sorted(files):
        h.update(fn.encode() + b"\0" + _code_tokens(read(fn)).encode())
    return h.hexdigest()[:16]


def row_family(key: str) -> str:
    """Kernel family a benchmark row (a ``_case_builders`` name) runs."""
    if key.startswith("ag-"):
        return "ag_norm"
    if key in ("c5-qk", "single-768"):
        return "qk_norm"
    return "fused_rows"


def recorded_traffic(key: str):
    """dram read+write bytes per step of the benchmark row ``key`` from the
    committed ncu captures, if they were taken on that row's kernel as it is
    now (same hash of its family's sources); else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    row = rec.get("rows", {}).get(key)
    if row is None or row.get("kernel_hash") != kernel_source_hash(KERNEL_FAMILIES[row_family(key)]):
        return None
    return int(row["bytes"])


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index, self.period_ms, self.proc = index, period_ms, None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let the first sample land
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest ``value`` over all ranks (every rank gets it)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline, never a target)
# ---------------------------------------------------------------------------

def oracle_rows_per_second(inp_host: dict, seconds: float, pattern: int = 1, partial_cols: int = 0):
    import numpy as np

    import oracle
    from reduce_residual_rmsnorm_gb300 import workloads as wl

    parts = [wl.bits(p) for p in inp_host["partials"]]
    res, gamma = wl.bits(inp_host["residual"]), wl.bits(inp_host["gamma"])
    T = res.shape[0]
    done, start, row = 0, time.perf_counter(), 0
    chunk = 8
    while True:
        rows = (np.arange(chunk) + row) % T
        oracle.fused_reduce_norm(pattern, parts, res, gamma, EPS, partial_cols=partial_cols, rows=rows)
        done += chunk
        row = (row + chunk) % T
        el = time.perf_counter() - start
        if el >= seconds:
            return done / el, done, el


def _oracle_worker(args):
    """One process of the all-cores baseline: memory-map the bf16 inputs the
    parent wrote, then run the oracle on this worker's rows for ``seconds``."""
    path, R, T, H, first, stride, seconds, pattern, partial_cols = args
    import numpy as np

    import oracle

    data = np.memmap(path, dtype=np.uint16, mode="r", shape=(R + 1, T, H))
    gamma = np.memmap(path + ".gamma", dtype=np.uint16, mode="r", shape=(H,))
    parts = [np.asarray(data[r]) for r in range(R)]
    res = np.asarray(data[R])
    gamma = np.asarray(gamma)
    done, row, start = 0, first, time.perf_counter()
    while True:
        rows = (np.arange(8) * stride + row) % T
        oracle.fused_reduce_norm(pattern, parts, res, gamma, EPS, partial_cols=partial_cols, rows=rows)
        done += 8
        row = (row + 8 * stride) % T
        el = time.perf_counter() - start
        if el >= seconds:
            return done, el


def oracle_rows_per_second_all_cores(inp_host: dict, seconds: float, pattern: int = 1, partial_cols: int = 0):
    """The same oracle, one spawned process per host core, each on its own rows
    (a reported baseline only); returns (rows/s, cores)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import tempfile

    import numpy as np

    from reduce_residual_rmsnorm_gb300 import workloads as wl

    cores = os.cpu_count() or 1
    R, T, H = inp_host["partials"].shape
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "inputs.bf16")
        mm = np.memmap(path, dtype=np.uint16, mode="w+", shape=(R + 1, T, H))
        for r in range(R):
            mm[r] = wl.bits(inp_host["partials"][r])
        mm[R] = wl.bits(inp_host["residual"])
        mm.flush()
        del mm
        wl.bits(inp_host["gamma"]).tofile(path + ".gamma")
        # spawned (not forked) workers; a worker that dies raises instead of hanging
        with cf.ProcessPoolExecutor(cores, mp_context=mp.get_context("spawn")) as ex:
            futs = [ex.submit(_oracle_worker, (path, R, T, H, i, cores, seconds, pattern, partial_cols))
                    for i in range(cores)]
            res = [f.result(timeout=seconds + 300) for f in futs]
    return sum(done / el for done, el in res), cores


def headline_config(world: int) -> dict:
    """The ``config`` of the JSON line; both arms print the same one."""
    from reduce_residual_rmsnorm_gb300 import workloads as wl

    shape = wl.WORKLOADS[HEADLINE["key"]]
    nbytes = headline_bytes()
    return {"workload": WORKLOAD, "pattern": HEADLINE["pattern"], "R": shape.R, "T": shape.T, "H": shape.H,
            "partial_cols": HEADLINE["partial_cols"], "launch_with_pdl": True, "bytes_per_step": nbytes,
            "l2": (f"inputs larger than L2 ({nbytes / 1e6:.0f} MB per step > 129 MB), and {NSETS} copies of "
                   "the inputs and outputs alternated between steps; no flush"),
            "parallelism": f"replicas x{world} (rows are independent; no collective)"}


def headline_bytes() -> int:
    from reduce_residual_rmsnorm_gb300 import workloads as wl

    shape = wl.WORKLOADS[HEADLINE["key"]]
    return fused_bytes(HEADLINE["pattern"], shape.R, shape.T, shape.H, HEADLINE["partial_cols"])


# ---------------------------------------------------------------------------
# the reference arm: the oracle on host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from reduce_residual_rmsnorm_gb300 import workloads as wl

    shape = wl.WORKLOADS[HEADLINE["key"]]
    pattern, P = HEADLINE["pattern"], HEADLINE["partial_cols"]
    inp = wl.fused_inputs(shape, seed=0)
    parts = [wl.bits(p) for p in inp["partials"]]
    res, gamma = wl.bits(inp["residual"]), wl.bits(inp["gamma"])

    def rows_call(rows):
        oracle.fused_reduce_norm(pattern, parts, res, gamma, EPS, partial_cols=P, rows=rows)

    t0 = time.perf_counter()
    rows_call(np.arange(4))
    per_row = (time.perf_counter() - t0) / 4
    budget = 120.0  # seconds for warm-up + timed steps together
    rows_per_step = int(max(1, min(shape.T, budget / max(1, args.steps + args.warmup) / per_row)))
    step_rows = lambda i: (np.arange(rows_per_step) + i * rows_per_step) % shape.T  # noqa: E731
    for i in range(args.warmup):
        rows_call(step_rows(i))
    t0 = time.perf_counter()
    for i in range(args.steps):
        rows_call(step_rows(args.warmup + i))
    el = time.perf_counter() - t0
    value = rows_per_step * args.steps / el
    sample = (f"{rows_per_step} of the {shape.T} rows per step (pattern {pattern}, R={shape.R}, H={shape.H}, "
              f"P={P}), single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": headline_config(world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

# Host time the Python binding takes to enqueue one call (measured 9-16 us on
# the Grace host); the gate in front of a timed region lasts long enough for
# the host to enqueue that many calls.
GATE_US_PER_LAUNCH = 25.0
GATE_MAX_LAUNCHES = 512
SLEEP_CYCLES_PER_US = 2100  # torch.cuda._sleep counts SM clock cycles (at most 2070 MHz here)


def gate(stream, launches: int) -> float:
    """Queue a spin kernel on ``stream`` that keeps the GPU busy while the host
    enqueues the next ``launches`` calls, so that a start event recorded after
    it is followed by launches already in the queue.  Returns its nominal
    length in microseconds."""
    import torch

    us = min(launches, GATE_MAX_LAUNCHES) * GATE_US_PER_LAUNCH + 100.0
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * SLEEP_CYCLES_PER_US))
    return us


def time_launches(calls, iters: int, stream, warmup: int = 3, launches_per_call: int = 1) -> float:
    """Average ms per call, CUDA events on ``stream`` around ``iters`` calls.

    ``calls``: one callable, or a list of callables (one per copy of the
    buffers) taken in turn, so that consecutive calls touch different memory.
    The region starts behind ``gate``."""
    import torch

    seq = list(calls) if isinstance(calls, (list, tuple)) else [calls]
    n = len(seq)
    for i in range(warmup):
        seq[i % n]()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gate(stream, iters * launches_per_call)
    s.record(stream)
    for i in range(iters):
        seq[(warmup + i) % n]()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / iters


def roofline_entry(nbytes: int, ms: float, peak: float) -> dict:
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"us": ms * 1e3, "bytes": nbytes, "gbs": gbs, "frac": gbs / peak}


def _copies(make, nsets: int = NSETS) -> list:
    """``nsets`` calls of one workload, call i built by ``make(i)`` on its own
    copy of the inputs and outputs (copy 0 may use the original tensors)."""
    return [make(i) for i in range(nsets)]


def _case_builders():
    """name -> (label, builder).  builder(dev, stream) returns
    (calls, algorithmic bytes per call, launches per call); ``calls`` holds one
    call per copy of the buffers (inputs drawn on the GPU)."""
    import torch

    import reduce_residual_rmsnorm_gb300 as pkg
    from reduce_residual_rmsnorm_gb300 import workloads as wl

    def clone_if(t, i):
        return t if i == 0 else t.clone()

    def fused(key, pattern, P=0, pdl=True, layout=2, R=None, T=None, H=None, early=False, indep=False):
        """One AllReduceFusionPattern on a named workload (or an R/T/H variant of
        it); FP8 per-tensor and NVFP4 scales from the workload's own norm."""
        def build(dev, stream):
            shape = wl.WORKLOADS[key]
            if R is not None:
                shape = wl.FusedShape(R=R, T=T, H=H, p_std=shape.p_std, res_std=shape.res_std,
                                      outlier_frac=shape.outlier_frac)
            inp = wl.fused_inputs(shape, seed=0, device=dev)
            Tn, Hn = shape.T, shape.H
            sf = None
            if pattern in (2, 3, 4, 5):
                norm = torch.empty((Tn, Hn), dtype=torch.bfloat16, device=dev)
                pkg.ts_fused_reduce_norm(1, inp["partials"], inp["residual"], inp["gamma"], EPS,
                                         residual_out=torch.empty_like(norm), norm_out=norm, stream=stream)
                top = 2688.0 if pattern in (3, 5) else 448.0
                sf = (top / norm.float().abs().max()).reshape(1).to(torch.float32)
                del norm

            def make(i):
                parts = clone_if(inp["partials"], i)
                res = None if pattern == 0 else clone_if(inp["residual"], i)
                gam = None if pattern == 0 else inp["gamma"]
                outs = pkg.new_outputs(pattern, Tn, Hn, dev, partial_cols=P, sf_layout=layout)
                extra = {"sf_layout": layout} if pattern in (3, 5) else {}
                return lambda: pkg.ts_fused_reduce_norm(pattern, parts, res, gam, EPS, sf,  # noqa: E731
                                                        launch_with_pdl=pdl, pdl_early_read=early,
                                                        pdl_independent=indep, stream=stream, **extra, **outs)
            return _copies(make), fused_bytes(pattern, shape.R, Tn, Hn, P, sf_layout=layout), 1
        return build

    def rs_add(rs_pattern, all_ranks=False, concurrent=False, early=False, indep=False):
        """R per-rank calls one after the other (launch_with_pdl), one call over
        every rank's slice (rank -1), or, ``concurrent``, the R per-rank calls
        on R streams forked from and joined back to ``stream`` (the ranks run
        at the same time, as on R GPUs), captured once in a CUDA graph that
        each step replays."""
        def build(dev, stream):
            shape = wl.WORKLOADS["C3"]
            inp = wl.fused_inputs(shape, seed=0, device=dev)
            R, T, H = shape.R, shape.T, shape.H
            gen = torch.Generator(device=dev)
            gen.manual_seed(1)
            add = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
            ranks = [-1] if all_ranks else list(range(R))

            def make(i):
                parts, a_all, r_all = clone_if(inp["partials"], i), clone_if(add, i), clone_if(inp["residual"], i)
                calls = []
                for rank in ranks:
                    start, count = pkg.rs_token_split(T, R, rank)
                    form = 6 if rs_pattern == 7 else 1
                    outs = pkg.new_outputs(form, count, H, dev)
                    calls.append((rank, a_all[start:start + count], r_all[start:start + count], outs))

                def call():
                    # with indep, rank 0's call is made without the flag: it
                    # waits for the step before, so a run of calls made with it
                    # never spans two steps (which share buffers)
                    for rank, a_in, res, outs in calls:
                        pkg.ts_reducescatter_fused_norm(rs_pattern, parts, rank, a_in, res, inp["gamma"], EPS,
                                                        launch_with_pdl=True, pdl_early_read=early,
                                                        pdl_independent=indep and rank > 0, stream=stream,
                                                        **outs)
                if not concurrent:
                    return call
                side = [torch.cuda.Stream(device=dev) for _ in calls]
                graph = torch.cuda.CUDAGraph()
                torch.cuda.synchronize()
                with torch.cuda.graph(graph, stream=stream):
                    for s2, (rank, a_in, res, outs) in zip(side, calls):
                        s2.wait_stream(stream)
                        pkg.ts_reducescatter_fused_norm(rs_pattern, parts, rank, a_in, res, inp["gamma"], EPS,
                                                        stream=s2, **outs)
                    for s2 in side:
                        stream.wait_stream(s2)
                return graph.replay
            nbytes = rs_add_bytes(R, T, H, rs_pattern == 7) - (R - 1) * H * 2 * (1 if all_ranks else 0)
            return _copies(make), nbytes, 1 if concurrent else len(ranks)
        return build

    def ag(pattern):
        def build(dev, stream):
            R, T, q, kv, rope = 8, 65536, 1536, 512, 64
            gen = torch.Generator(device=dev)
            gen.manual_seed(0)
            full = torch.randn((T, q + kv + rope), generator=gen, device=dev).to(torch.bfloat16)
            slices = [full[s:s + c].clone() for s, c in (pkg.rs_token_split(T, R, r) for r in range(R))]
            del full
            xg = (torch.rand(q, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
            yg = (torch.rand(kv, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
            e = lambda *sh, dt=torch.bfloat16: torch.empty(sh, dtype=dt, device=dev)  # noqa: E731

            def make(i):
                ins = [clone_if(x, i) for x in slices]
                outs = {"allgather_out": e(T, q + kv + rope)}
                if pattern == 1:
                    outs.update(x_norm_out=e(T, q), y_norm_out=e(T, kv))
                elif pattern == 2:
                    outs.update(y_norm_out=e(T, kv), quant_out=e(T, q, dt=torch.uint8),
                                scale_out=e(T, q // 128, dt=torch.float32))
                return lambda: pkg.ts_allgather_fused_norm(pattern, ins, q, kv, rope, xg, yg, EPS, EPS,  # noqa
                                                           launch_with_pdl=True, stream=stream, **outs)
            return _copies(make), ag_bytes(pattern, T, q, kv, rope), 1
        return build

    def c5(dev, stream):
        qs = wl.WORKLOADS["C5"]
        qi = wl.qk_inputs(qs, seed=0, device=dev)

        def make(i):
            sh = clone_if(qi["shards"], i)
            qo = torch.empty((qs.T, qs.R * qs.q_shard), dtype=torch.bfloat16, device=dev)
            ko = torch.empty((qs.T, qs.R * qs.k_shard), dtype=torch.bfloat16, device=dev)
            return lambda: pkg.ts_qk_norm_sharded(sh, qs.q_shard, qs.k_shard, qi["q_weight"],  # noqa: E731
                                                  qi["k_weight"], EPS, qo, ko, launch_with_pdl=True,
                                                  stream=stream)
        return _copies(make), qk_bytes(qs.R, qs.T, qs.q_shard, qs.k_shard), 1

    def single(dev, stream):
        gen = torch.Generator(device=dev)
        gen.manual_seed(0)
        sh0 = torch.randn((8, 32768, 768), generator=gen, device=dev).to(torch.bfloat16)
        w = (torch.rand(8 * 768, generator=gen, device=dev) + 0.5).to(torch.bfloat16)

        def make(i):
            sh = clone_if(sh0, i)
            so = torch.empty((32768, 8 * 768), dtype=torch.bfloat16, device=dev)
            return lambda: pkg.ts_rms_norm_sharded(sh, 768, w, EPS, so, launch_with_pdl=True,  # noqa: E731
                                                   stream=stream)
        return _copies(make), rms_sharded_bytes(8, 32768, 768), 1

    def c1(dev, stream):
        shape = wl.WORKLOADS["C1"]
        inp = wl.fused_inputs(shape, seed=0, device=dev)
        outs = pkg.new_outputs(1, 16, 4096, dev)

        def call(pdl=False, early=False):
            pkg.ts_fused_reduce_norm(1, inp["partials"], inp["residual"], inp["gamma"], EPS, stream=stream,
                                     launch_with_pdl=pdl, pdl_early_read=early, **outs)
        return [call], fused_bytes(1, 2, 16, 4096), 1

    tp = lambda pattern, R: fused("C4", pattern, R=R, T=16384, H=5120)  # noqa: E731
    return {
        "c3-p7": ("kARResidualRMSNormPartialOutFP8BlockWiseQuant R=8 T=8192 H=7168 P=1024",
                  fused("C3", 7, 1024)),
        "c3-p7-nopdl": ("kARResidualRMSNormPartialOutFP8BlockWiseQuant R=8 T=8192 H=7168 P=1024 (plain launch)",
                        fused("C3", 7, 1024, pdl=False)),
        "c3-p7-early": ("kARResidualRMSNormPartialOutFP8BlockWiseQuant R=8 T=8192 H=7168 P=1024 (inputs read "
                        "before the wait)", fused("C3", 7, 1024, early=True)),
        "c2-p1": ("kARResidualRMSNorm R=8 T=4096 H=7168", fused("C2", 1)),
        "c2-p0": ("kAllReduce R=8 T=4096 H=7168", fused("C2", 0)),
        "c3-p2": ("kARResidualRMSNormFP8Quant R=8 T=8192 H=7168", fused("C3", 2)),
        "c3-p6": ("kARResidualRMSNormFP8BlockWiseQuant R=8 T=8192 H=7168", fused("C3", 6)),
        "c3-p8": ("kARResidualRMSNormPartialOut R=8 T=8192 H=7168 P=1024", fused("C3", 8, 1024)),
        "c4-p3-linear": ("kARResidualRMSNormFP4Quant R=4 T=16384 H=5120 SF LINEAR", fused("C4", 3, layout=2)),
        "c4-p3-swizzled": ("kARResidualRMSNormFP4Quant R=4 T=16384 H=5120 SF SWIZZLED_128x4",
                           fused("C4", 3, layout=0)),
        "c4-p3-swizzled8": ("kARResidualRMSNormFP4Quant R=4 T=16384 H=5120 SF SWIZZLED_8x4",
                            fused("C4", 3, layout=1)),
        "rs-add": ("kRSAddResidualRMSNorm R=8 T=8192 H=7168, all 8 rank slices (8 PDL calls)", rs_add(8)),
        "rs-add-all": ("kRSAddResidualRMSNorm R=8 T=8192 H=7168, rank -1 (one call)", rs_add(8, True)),
        "rs-add-fp8b": ("kRSAddResidualRMSNormFP8BlockWiseQuant R=8 T=8192 H=7168, all 8 rank slices (8 PDL calls)",
                        rs_add(7)),
        "rs-add-early": ("kRSAddResidualRMSNorm R=8 T=8192 H=7168, all 8 rank slices (8 PDL calls, inputs read "
                         "before the wait)", rs_add(8, early=True)),
        "rs-add-fp8b-early": ("kRSAddResidualRMSNormFP8BlockWiseQuant R=8 T=8192 H=7168, all 8 rank slices (8 PDL "
                              "calls, inputs read before the wait)", rs_add(7, early=True)),
        "rs-add-indep": ("kRSAddResidualRMSNorm R=8 T=8192 H=7168, all 8 rank slices (8 PDL calls, ranks 1-7 "
                         "waiting only before they exit)", rs_add(8, indep=True)),
        "rs-add-fp8b-indep": ("kRSAddResidualRMSNormFP8BlockWiseQuant R=8 T=8192 H=7168, all 8 rank slices (8 PDL "
                              "calls, ranks 1-7 waiting only before they exit)", rs_add(7, indep=True)),
        "rs-add-fp8b-streams": ("kRSAddResidualRMSNormFP8BlockWiseQuant R=8 T=8192 H=7168, all 8 rank slices "
                                "(8 calls on 8 streams, one CUDA graph)", rs_add(7, concurrent=True)),
        "rs-add-streams": ("kRSAddResidualRMSNorm R=8 T=8192 H=7168, all 8 rank slices (8 calls on 8 streams, "
                           "one CUDA graph)", rs_add(8, concurrent=True)),
        "rs-add-fp8b-all": ("kRSAddResidualRMSNormFP8BlockWiseQuant R=8 T=8192 H=7168, rank -1 (one call)",
                            rs_add(7, True)),
        "ag-rms": ("kAllGatherfusedRMS R=8 T=65536 1536|512|64", ag(1)),
        "ag-rms-fp8b": ("kAllGatherfusedRMSFP8BlockWiseQuant R=8 T=65536 1536|512|64", ag(2)),
        "c5-qk": ("MiniMax QK-RMSNorm R=8 T=32768 Q=1024 K=128", c5),
        "single-768": ("single-matrix sharded RMSNorm R=8 T=32768 W=768", single),
        "tp1-p1": ("kARResidualRMSNorm R=1 T=16384 H=5120", tp(1, 1)),
        "tp2-p1": ("kARResidualRMSNorm R=2 T=16384 H=5120", tp(1, 2)),
        "tp2-p3": ("kARResidualRMSNormFP4Quant R=2 T=16384 H=5120 SF LINEAR", tp(3, 2)),
        "tp2-p6": ("kARResidualRMSNormFP8BlockWiseQuant R=2 T=16384 H=5120", tp(6, 2)),
        "tp4-p6": ("kARResidualRMSNormFP8BlockWiseQuant R=4 T=16384 H=5120", tp(6, 4)),
        "c1-p1": ("kARResidualRMSNorm R=2 T=16 H=4096 (latency, inputs warm in L2)", c1),
    }


def measure_rows(dev, stream, peak: float, iters: int, only=None) -> dict:
    import torch

    rows = {}
    for key, (label, build) in _case_builders().items():
        if key == "c3-p7" or (only is not None and key not in only):
            continue  # the headline step, timed in run_ours
        with torch.cuda.stream(stream):
            calls, nbytes, per_call = build(dev, stream)
            if key == "c1-p1":  # L2-resident latency case: stream launches and a CUDA graph
                call = calls[0]
                ms_stream = time_launches(call, max(iters, 200), stream)
                graph = torch.cuda.CUDAGraph()
                call()
                torch.cuda.synchronize()
                with torch.cuda.graph(graph, stream=stream):
                    for _ in range(100):
                        call()
                ms_graph = time_launches(graph.replay, 20, stream) / 100
                del graph
                pdl_graph = torch.cuda.CUDAGraph()  # the same chain with launch_with_pdl
                with torch.cuda.graph(pdl_graph, stream=stream):
                    for _ in range(100):
                        call(pdl=True)
                ms_pdl = time_launches(pdl_graph.replay, 20, stream) / 100
                del pdl_graph
                # and with TS_FLAG_PDL_EARLY_READ: no call of the chain writes another's inputs
                early_graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(early_graph, stream=stream):
                    for _ in range(100):
                        call(pdl=True, early=True)
                ms_early = time_launches(early_graph.replay, 20, stream) / 100
                del early_graph
                rows[label] = {"us_stream_launch": ms_stream * 1e3, "us_in_cuda_graph": ms_graph * 1e3,
                               "us_in_cuda_graph_pdl": ms_pdl * 1e3,
                               "us_in_cuda_graph_pdl_early_read": ms_early * 1e3, "bytes": nbytes}
            else:
                ms = time_launches(calls, iters, stream, launches_per_call=per_call)
                rows[label] = roofline_entry(nbytes, ms, peak)
                rows[label]["traffic"] = recorded_traffic(key)
        del calls
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return rows


def profile_case(key: str, launches: int) -> None:
    """Set up one named workload and launch it ``launches`` times (for ncu)."""
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    import __graft_entry__

    __graft_entry__.build()
    label, build = _case_builders()[key]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        calls, nbytes, _ = build(dev, stream)
        torch.cuda.synchronize()
        for i in range(launches):
            calls[i % len(calls)]()
    torch.cuda.synchronize()
    print(json.dumps({"case": key, "label": label, "launches": launches, "bytes_per_launch": nbytes}))


# (pattern, R, H) and T values of the per-call table: single calls with the inputs cold in L2
SWEEP_SHAPES = ((1, 8, 7168), (6, 8, 7168), (3, 4, 5120), (1, 2, 4096))
SWEEP_TOKENS = (1, 16, 64, 256, 1024, 4096, 16384)
# the other entry points in the same table: all-gather pattern 2 over R=8 slices
# of 1536 | 512 | 64 rows, and the MiniMax QK norm on R=8 shards of q 1024 | k 128
SWEEP_OTHER = ("allgather-fp8", "qk")


def sweep_t(reps: int = 40) -> None:
    """Per-call time of single calls (launch_with_pdl) against T, with the
    inputs cold in L2: a CUDA graph of ``reps`` x (copy a 256 MB buffer, call),
    minus a graph of ``reps`` copies alone.  One JSON line per (shape, T).
    A copy rather than a read-only pass: after a long read-only kernel every
    kernel that writes, PyTorch's own copy included, starts several
    microseconds slower (a 69 MB copy: 22.6 us after a 256 MB copy, 30.7 us
    after a 256 MB reduction), which would not be this library's cost."""
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    import __graft_entry__

    __graft_entry__.build()
    import reduce_residual_rmsnorm_gb300 as pkg
    from reduce_residual_rmsnorm_gb300 import workloads as wl

    peak, peak_kind = read_peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush_dst = torch.empty_like(flush)

    def flush_l2():
        flush_dst.copy_(flush)

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    fn()
        return g

    def per_call_ms(g):
        with torch.cuda.stream(stream):
            return min(time_launches(g.replay, 5, stream) for _ in range(3)) / reps

    def report(call, nbytes, **key):
        def both():
            flush_l2()
            call()
        g = graph_of(both)
        ms = per_call_ms(g) - per_call_ms(g_flush)
        print(json.dumps({**key, "us": ms * 1e3, "frac": nbytes / (ms * 1e-3) / 1e9 / peak,
                          "peak_kind": peak_kind}), flush=True)
        del g
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    g_flush = graph_of(flush_l2)
    print(json.dumps({"flush_us": per_call_ms(g_flush) * 1e3}), flush=True)
    for p, R, H in SWEEP_SHAPES:
        for T in SWEEP_TOKENS:
            inp = wl.fused_inputs(wl.FusedShape(R=R, T=T, H=H), seed=0, device=dev)
            outs = pkg.new_outputs(p, T, H, dev)
            sf = torch.tensor([100.0], device=dev) if p in (2, 3, 4, 5) else None
            report(lambda: pkg.ts_fused_reduce_norm(p, inp["partials"], inp["residual"], inp["gamma"],  # noqa
                                                    EPS, sf, stream=stream, launch_with_pdl=True, **outs),
                   fused_bytes(p, R, T, H), pattern=p, R=R, T=T, H=H)
            del inp, outs
    R, q, kv, rope = 8, 1536, 512, 64
    for T in SWEEP_TOKENS:
        gen = torch.Generator(device=dev)
        gen.manual_seed(0)
        full = torch.randn((T, q + kv + rope), generator=gen, device=dev).to(torch.bfloat16)
        ins = [full[s0:s0 + c].clone() for s0, c in (pkg.rs_token_split(T, R, r) for r in range(R))]
        xg = (torch.rand(q, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
        yg = (torch.rand(kv, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
        e = lambda *sh, dt=torch.bfloat16: torch.empty(sh, dtype=dt, device=dev)  # noqa: E731
        outs = dict(allgather_out=e(T, q + kv + rope), y_norm_out=e(T, kv), quant_out=e(T, q, dt=torch.uint8),
                    scale_out=e(T, q // 128, dt=torch.float32))
        report(lambda: pkg.ts_allgather_fused_norm(2, ins, q, kv, rope, xg, yg, EPS, EPS,  # noqa: E731
                                                   launch_with_pdl=True, stream=stream, **outs),
               ag_bytes(2, T, q, kv, rope), entry="allgather-fp8", R=R, T=T, hidden=q + kv + rope)
        del full, ins, outs
    qs = wl.QKShape(R=8, T=1, q_shard=1024, k_shard=128, v_shard=128)
    for T in SWEEP_TOKENS:
        qi = wl.qk_inputs(wl.QKShape(R=qs.R, T=T, q_shard=qs.q_shard, k_shard=qs.k_shard, v_shard=qs.v_shard),
                          seed=0, device=dev)
        qo = torch.empty((T, qs.R * qs.q_shard), dtype=torch.bfloat16, device=dev)
        ko = torch.empty((T, qs.R * qs.k_shard), dtype=torch.bfloat16, device=dev)
        report(lambda: pkg.ts_qk_norm_sharded(qi["shards"], qs.q_shard, qs.k_shard, qi["q_weight"],  # noqa: E731
                                              qi["k_weight"], EPS, qo, ko, launch_with_pdl=True, stream=stream),
               qk_bytes(qs.R, T, qs.q_shard, qs.k_shard), entry="qk", R=qs.R, T=T)
        del qi, qo, ko


def c_abi_call_cost():
    """Host microseconds per C-ABI call from a C99 caller (tests/c_call_cost.c),
    or a dict with the reason it could not be measured."""
    import tempfile

    from reduce_residual_rmsnorm_gb300 import build as libbuild

    try:
        lib = libbuild.build()
        cuda = os.path.dirname(os.path.dirname(libbuild.nvcc()))
        libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")) if os.path.isdir(d)]
        with tempfile.TemporaryDirectory() as d:
            exe = os.path.join(d, "c_call_cost")
            subprocess.check_call(["gcc", "-std=c99", "-O2", "-I", os.path.join(ROOT, "include"), "-isystem",
                                   os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_call_cost.c"),
                                   "-o", exe, lib, *[f"-L{x}" for x in libdirs], "-lcudart",
                                   "-Wl,-rpath," + os.path.dirname(lib), *[f"-Wl,-rpath,{x}" for x in libdirs]])
            r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
        if r.returncode != 0:
            return {"unavailable": (r.stdout + r.stderr).strip()[-300:]}
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, RuntimeError) as exc:
        return {"unavailable": str(exc)[-300:]}


def run_ours(args):
    import statistics as st

    import torch

    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import __graft_entry__

    __graft_entry__.build()
    import reduce_residual_rmsnorm_gb300 as pkg
    from reduce_residual_rmsnorm_gb300 import workloads as wl

    peak, peak_kind = read_peaks()
    shape = wl.WORKLOADS[HEADLINE["key"]]
    pattern, P = HEADLINE["pattern"], HEADLINE["partial_cols"]
    R, T, H = shape.R, shape.T, shape.H
    host_inp = wl.fused_inputs(shape, seed=0)
    gamma = host_inp["gamma"].to(dev)
    sets = []
    for i in range(NSETS):  # step i uses copy i % NSETS of the inputs and outputs
        sets.append((host_inp["partials"].to(dev), host_inp["residual"].to(dev),
                     pkg.new_outputs(pattern, T, H, dev, partial_cols=P)))
    stream = torch.cuda.Stream(device=dev)
    nbytes = headline_bytes()

    def step(i):
        parts, res, outs = sets[i % NSETS]
        pkg.ts_fused_reduce_norm(pattern, parts, res, gamma, EPS, launch_with_pdl=True, stream=stream, **outs)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    with sampler:
        barrier(world)
        torch.cuda.synchronize()
        gate_us = gate(stream, args.steps)
        ev0.record(stream)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                step(args.warmup + i)
        host_s = time.perf_counter() - t0
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms = max_over_ranks(ms_local, world, dev)
    value = world * T / (ms * 1e-3)
    achieved = nbytes / (ms_local * 1e-3) / 1e9

    # diagnostic pass: an event after every launch (which ends the PDL overlap
    # of consecutive launches, so each step reads a little slower than in the
    # timed region)
    n_diag = min(args.steps, 50)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_diag + 1)]
    gate(stream, n_diag)
    evs[0].record(stream)
    with torch.cuda.stream(stream):
        for i in range(n_diag):
            step(i)
            evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per_step = [evs[i].elapsed_time(evs[i + 1]) * 1e3 for i in range(n_diag)]

    # end to end through the C ABI with host buffers.  Headline form: the call
    # is given the pinned host inputs and outputs themselves, and the kernel
    # moves every byte across the host link (NVLink-C2C on Grace-Blackwell).
    # For comparison, the staged form copies the inputs to the device, calls,
    # and copies the outputs back (copy engines, one stream).
    h_parts = host_inp["partials"].pin_memory()
    h_res = host_inp["residual"].pin_memory()
    h_gamma = host_inp["gamma"].pin_memory()
    h_outs = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in sets[0][2].items()}
    d_parts, d_res, d_outs = sets[0]

    def e2e_step():
        pkg.ts_fused_reduce_norm(pattern, h_parts, h_res, h_gamma, EPS, launch_with_pdl=True, stream=stream,
                                 **h_outs)

    def staged_step():
        d_parts.copy_(h_parts, non_blocking=True)
        d_res.copy_(h_res, non_blocking=True)
        pkg.ts_fused_reduce_norm(pattern, d_parts, d_res, gamma, EPS, launch_with_pdl=True, stream=stream,
                                 **d_outs)
        for k, v in h_outs.items():
            v.copy_(d_outs[k], non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    with torch.cuda.stream(stream):
        e2e_ms = time_launches(e2e_step, e2e_steps, stream, warmup=2)
        staged_ms = time_launches(staged_step, e2e_steps, stream, warmup=2)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    staged_ms = max_over_ranks(staged_ms, world, dev)
    h2d = (h_parts.numel() + h_res.numel() + h_gamma.numel()) * 2
    d2h = sum(v.numel() * v.element_size() for v in h_outs.values())
    del h_parts, h_res, h_gamma, h_outs, sets, d_parts, d_res, d_outs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    rows = None
    if not args.no_rows:
        rows = measure_rows(dev, stream, peak, args.row_iters)
    call_cost = c_abi_call_cost() if rank == 0 and not args.no_rows else None

    cpu = cpu_all = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        rps, done, el = oracle_rows_per_second(host_inp, args.cpu_seconds, pattern, P)
        cpu = {"value": rps, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{done} rows of the R={R} T={T} H={H} pattern {pattern} (P={P}) workload "
                         f"(8-row batches, wrapping), {el:.1f} s of single-threaded C"}
        if args.cpu_all_cores:
            rps_all, cores = oracle_rows_per_second_all_cores(host_inp, args.cpu_seconds, pattern, P)
            cpu_all = {"value": rps_all, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                       "sample": f"one spawned process per core, each {args.cpu_seconds:.0f} s on its own rows "
                                 f"of the same workload"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": headline_config(world),
            "achieved_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": f"{peak_kind} HBM copy bandwidth",
                         "traffic": recorded_traffic("c3-p7")},
            "timed_region": {
                "gate_us": gate_us, "host_us_per_call": host_s / args.steps * 1e6,
                "per_step_us": [round(x, 2) for x in per_step],
                "per_step_median_us": st.median(per_step),
                "note": ("the timed launches sit behind a spin kernel of gate_us, so the region times the GPU "
                         "running them back to back; per_step_us is a separate pass with an event after every "
                         "launch (no PDL overlap between launches there)")},
            "e2e": {"value": T * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "mode": "pinned host inputs and outputs passed to the call; the kernel reads and writes "
                            "them across the host link (no staging copy)",
                    "staged": {"value": T * world / (staged_ms * 1e-3), "ms_per_step": staged_ms,
                               "mode": "cudaMemcpyAsync of the inputs to the device, the call, and of the "
                                       "outputs back, on one stream"}},
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "c_abi_host_us_per_call": call_cost,
            "gpu_launches": args.steps,
            "clocks": sampler.summary(),
            "kernel_source_hash": kernel_source_hash(),
            "rows": rows,
        }
        print(json.dumps(line), flush=True)


def check_world(gpus: int, env=None) -> str:
    """How to honour ``--gpus``: "run" (this process is one of the ranks, or
    N = 1) or "spawn" (start N ranks through torch.distributed.run).  Raises
    SystemExit when a torchrun world disagrees with --gpus."""
    env = os.environ if env is None else env
    if gpus < 1:
        raise SystemExit(f"--gpus must be >= 1 (got {gpus})")
    world = env.get("WORLD_SIZE")
    if world is None:
        return "spawn" if gpus > 1 else "run"
    if int(world) != gpus:
        raise SystemExit(f"--gpus {gpus} but WORLD_SIZE={world}: launch with --nproc-per-node {gpus}")
    return "run"


def spawn_command(argv: list, gpus: int, port: int) -> list:
    """torch.distributed.run command that starts ``gpus`` ranks of this script
    with the same arguments (one node, rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
            "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the other patterns/workloads")
    ap.add_argument("--row-iters", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-all-cores", dest="cpu_all_cores", action="store_false",
                    help="skip the all-cores oracle baseline")
    ap.add_argument("--profile-case", default=None,
                    help="only set up this named workload and launch it --launches times (for ncu)")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--sweep-t", action="store_true",
                    help="only print the per-call time of single cold fused calls against T")
    argv = sys.argv[1:] if argv is None else list(argv)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.sweep_t:
        sweep_t()
        return
    if args.profile_case:
        profile_case(args.profile_case, args.launches)
        return
    if check_world(args.gpus) == "spawn":
        import socket

        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        raise SystemExit(subprocess.call(spawn_command(argv, args.gpus, port)))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

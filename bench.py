"""Throughput of the fused reduce -> residual -> RMSNorm (+quant) path on GB300.

One step = one ``ts_fused_reduce_norm(kARResidualRMSNorm)`` call over the
R=8, T=4096, H=7168 bf16 workload (partials N(0, 0.5^2), residual N(0, 1),
gamma U(0.5, 1.5), seed 0), inputs resident in HBM, launched with the
pages' ``launch_with_pdl`` option (programmatic dependent launch: each call
still waits for the previous one to complete before touching memory).
Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``value`` is tokens (rows) per second over all ranks (each rank runs the
same per-GPU workload: weak scaling, no collective on the data path).  The
line also carries the roofline of the kernel (algorithmic bytes / CUDA-event
time against the measured HBM copy bandwidth), an end-to-end figure through
the C ABI with host buffers (the call given pinned host inputs and outputs,
which the kernel reads and writes across the host link; the staged-copy form
beside it), the CPU
oracle timed on a bounded sample of rows, the SM clocks sampled during the
timed region, and ``rows``: the other patterns and workloads timed the same
way (kAllReduce; FP8 per-tensor, FP8 1x128 blockwise, PartialOut on R=8,
T=8192; NVFP4 on R=4, T=16384, H=5120 in the three SF layouts; tensor-parallel
degrees 1, 2 and 4 on T=16384, H=5120; the reduce-scatter and all-gather forms;
the sharded MiniMax QK-norm and single-matrix norm on R=8, T=32768; and the R=2,
T=16 latency case).

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
WORKLOAD = ("kARResidualRMSNorm R=8 T=4096 H=7168: bf16 partials ~N(0,0.5^2), residual ~N(0,1), "
            "gamma ~U(0.5,1.5), eps 1e-6, seed 0")
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


KERNEL_SOURCES = ("ag_norm.cu", "device_util.cuh", "fused_rows.cu", "launch.h", "qk_norm.cu", "sf_layout.cuh")


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


def kernel_source_hash() -> str:
    """Hash of the device code (not the host-side argument checks), comments
    and layout excluded."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "reduce_residual_rmsnorm_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn in KERNEL_SOURCES:
            with open(os.path.join(csrc, fn), encoding="utf-8") as f:
                h.update(fn.encode() + b"\0" + _code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(key: str):
    """dram read+write bytes per launch from the committed ncu summary, if it was
    taken on the kernels as they are now (same source hash); else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    v = rec.get("captures", {}).get(kernel_source_hash(), {}).get("bytes_per_launch", {}).get(key)
    return None if v is None else int(v)


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

def oracle_rows_per_second(inp_host: dict, seconds: float, pattern: int = 1):
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
        oracle.fused_reduce_norm(pattern, parts, res, gamma, EPS, rows=rows)
        done += chunk
        row = (row + chunk) % T
        el = time.perf_counter() - start
        if el >= seconds:
            return done / el, done, el


def _oracle_worker(args):
    """One process of the all-cores baseline: memory-map the bf16 inputs the
    parent wrote, then run the oracle on this worker's rows for ``seconds``."""
    path, R, T, H, first, stride, seconds = args
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
        oracle.fused_reduce_norm(1, parts, res, gamma, EPS, rows=rows)
        done += 8
        row = (row + 8 * stride) % T
        el = time.perf_counter() - start
        if el >= seconds:
            return done, el


def oracle_rows_per_second_all_cores(inp_host: dict, seconds: float):
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
            futs = [ex.submit(_oracle_worker, (path, R, T, H, i, cores, seconds)) for i in range(cores)]
            res = [f.result(timeout=seconds + 300) for f in futs]
    return sum(done / el for done, el in res), cores


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

    shape = wl.WORKLOADS["C2"]
    inp = wl.fused_inputs(shape, seed=0)
    parts = [wl.bits(p) for p in inp["partials"]]
    res, gamma = wl.bits(inp["residual"]), wl.bits(inp["gamma"])
    t0 = time.perf_counter()
    oracle.fused_reduce_norm(1, parts, res, gamma, EPS, rows=np.arange(4))
    per_row = (time.perf_counter() - t0) / 4
    budget = 120.0  # seconds for warm-up + timed steps together
    rows_per_step = int(max(1, min(shape.T, budget / max(1, args.steps + args.warmup) / per_row)))
    step_rows = lambda i: (np.arange(rows_per_step) + i * rows_per_step) % shape.T  # noqa: E731
    for i in range(args.warmup):
        oracle.fused_reduce_norm(1, parts, res, gamma, EPS, rows=step_rows(i))
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.fused_reduce_norm(1, parts, res, gamma, EPS, rows=step_rows(args.warmup + i))
    el = time.perf_counter() - t0
    value = rows_per_step * args.steps / el
    sample = (f"{rows_per_step} of the {shape.T} rows per step (pattern 1, R=8, H=7168), "
              f"single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "pattern": 1, "R": 8, "T": 4096, "H": 7168},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def time_launches(fn, iters: int, stream, warmup: int = 3) -> float:
    """Average ms per call of ``fn`` (launching on ``stream``), CUDA events."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(iters):
        fn()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / iters


def roofline_entry(nbytes: int, ms: float, peak: float) -> dict:
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"us": ms * 1e3, "bytes": nbytes, "gbs": gbs, "frac": gbs / peak}


def _case_builders():
    """name -> builder(dev, stream) returning (call, algorithmic bytes per call, label).
    Builders allocate their inputs (drawn on the GPU) and outputs."""
    import torch

    import reduce_residual_rmsnorm_gb300 as pkg
    from reduce_residual_rmsnorm_gb300 import workloads as wl

    def c2(pattern, pdl=False):
        def build(dev, stream):
            shape = wl.WORKLOADS["C2"]
            inp = wl.fused_inputs(shape, seed=0, device=dev)
            T, H = shape.T, shape.H
            outs = pkg.new_outputs(pattern, T, H, dev)
            res = None if pattern == 0 else inp["residual"]
            gam = None if pattern == 0 else inp["gamma"]
            call = lambda: pkg.ts_fused_reduce_norm(pattern, inp["partials"], res, gam, EPS,  # noqa: E731
                                                    launch_with_pdl=pdl, stream=stream, **outs)
            return call, fused_bytes(pattern, 8, T, H)
        return build

    def c3(pattern, P=0):
        def build(dev, stream):
            shape = wl.WORKLOADS["C3"]
            inp = wl.fused_inputs(shape, seed=0, device=dev)
            T, H = shape.T, shape.H
            sf = None
            if pattern == 2:
                norm = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
                pkg.ts_fused_reduce_norm(1, inp["partials"], inp["residual"], inp["gamma"], EPS,
                                         residual_out=torch.empty_like(norm), norm_out=norm, stream=stream)
                sf = (448.0 / norm.float().abs().max()).reshape(1).to(torch.float32)
                del norm
            outs = pkg.new_outputs(pattern, T, H, dev, partial_cols=P)
            call = lambda: pkg.ts_fused_reduce_norm(pattern, inp["partials"], inp["residual"], inp["gamma"],  # noqa
                                                    EPS, sf, stream=stream, **outs)
            return call, fused_bytes(pattern, 8, T, H, P)
        return build

    def c4(layout):
        def build(dev, stream):
            shape = wl.WORKLOADS["C4"]
            inp = wl.fused_inputs(shape, seed=0, device=dev)
            T, H = shape.T, shape.H
            norm = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
            pkg.ts_fused_reduce_norm(1, inp["partials"], inp["residual"], inp["gamma"], EPS,
                                     residual_out=torch.empty_like(norm), norm_out=norm, stream=stream)
            g = (2688.0 / norm.float().abs().max()).reshape(1).to(torch.float32)
            del norm
            outs = pkg.new_outputs(3, T, H, dev, sf_layout=layout)
            call = lambda: pkg.ts_fused_reduce_norm(3, inp["partials"], inp["residual"], inp["gamma"], EPS,  # noqa
                                                    g, sf_layout=layout, stream=stream, **outs)
            return call, fused_bytes(3, 4, T, H, sf_layout=int(layout))
        return build

    def rs_add(rs_pattern, all_ranks=False):
        def build(dev, stream):
            shape = wl.WORKLOADS["C3"]
            inp = wl.fused_inputs(shape, seed=0, device=dev)
            R, T, H = shape.R, shape.T, shape.H
            gen = torch.Generator(device=dev)
            gen.manual_seed(1)
            add = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
            calls = []
            for rank in ([-1] if all_ranks else range(R)):
                start, count = pkg.rs_token_split(T, R, rank)
                form = 6 if rs_pattern == 7 else 1
                outs = pkg.new_outputs(form, count, H, dev)
                calls.append((rank, add[start:start + count], inp["residual"][start:start + count], outs))

            def call():
                for rank, a_in, res, outs in calls:
                    pkg.ts_reducescatter_fused_norm(rs_pattern, inp["partials"], rank, a_in, res, inp["gamma"],
                                                    EPS, launch_with_pdl=True, stream=stream, **outs)
            return call, rs_add_bytes(R, T, H, rs_pattern == 7) - (R - 1) * H * 2 * (1 if all_ranks else 0)
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
            outs = {"allgather_out": e(T, q + kv + rope)}
            if pattern == 1:
                outs.update(x_norm_out=e(T, q), y_norm_out=e(T, kv))
            elif pattern == 2:
                outs.update(y_norm_out=e(T, kv), quant_out=e(T, q, dt=torch.uint8),
                            scale_out=e(T, q // 128, dt=torch.float32))
            call = lambda: pkg.ts_allgather_fused_norm(pattern, slices, q, kv, rope, xg, yg, EPS, EPS,  # noqa
                                                       stream=stream, **outs)
            return call, ag_bytes(pattern, T, q, kv, rope)
        return build

    def c5(dev, stream):
        qs = wl.WORKLOADS["C5"]
        qi = wl.qk_inputs(qs, seed=0, device=dev)
        qo = torch.empty((qs.T, qs.R * qs.q_shard), dtype=torch.bfloat16, device=dev)
        ko = torch.empty((qs.T, qs.R * qs.k_shard), dtype=torch.bfloat16, device=dev)
        call = lambda: pkg.ts_qk_norm_sharded(qi["shards"], qs.q_shard, qs.k_shard, qi["q_weight"],  # noqa
                                              qi["k_weight"], EPS, qo, ko, stream=stream)
        return call, qk_bytes(qs.R, qs.T, qs.q_shard, qs.k_shard)

    def single(dev, stream):
        gen = torch.Generator(device=dev)
        gen.manual_seed(0)
        sh = torch.randn((8, 32768, 768), generator=gen, device=dev).to(torch.bfloat16)
        w = (torch.rand(8 * 768, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
        so = torch.empty((32768, 8 * 768), dtype=torch.bfloat16, device=dev)
        call = lambda: pkg.ts_rms_norm_sharded(sh, 768, w, EPS, so, stream=stream)  # noqa: E731
        return call, rms_sharded_bytes(8, 32768, 768)

    def c1(dev, stream):
        shape = wl.WORKLOADS["C1"]
        inp = wl.fused_inputs(shape, seed=0, device=dev)
        outs = pkg.new_outputs(1, 16, 4096, dev)
        def call(pdl=False):
            pkg.ts_fused_reduce_norm(1, inp["partials"], inp["residual"], inp["gamma"], EPS, stream=stream,
                                     launch_with_pdl=pdl, **outs)
        return call, fused_bytes(1, 2, 16, 4096)

    def tp(pattern, R):
        """Smaller tensor-parallel degrees on the R=4 T=16384 H=5120 shape."""
        def build(dev, stream):
            T, H = 16384, 5120
            inp = wl.fused_inputs(wl.FusedShape(R=R, T=T, H=H), seed=0, device=dev)
            g = None
            if pattern in (2, 3):
                norm = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
                pkg.ts_fused_reduce_norm(1, inp["partials"], inp["residual"], inp["gamma"], EPS,
                                         residual_out=torch.empty_like(norm), norm_out=norm, stream=stream)
                g = ((2688.0 if pattern == 3 else 448.0) / norm.float().abs().max()).reshape(1).to(torch.float32)
                del norm
            outs = pkg.new_outputs(pattern, T, H, dev)
            call = lambda: pkg.ts_fused_reduce_norm(pattern, inp["partials"], inp["residual"],  # noqa: E731
                                                    inp["gamma"], EPS, g, stream=stream, **outs)
            return call, fused_bytes(pattern, R, T, H)
        return build

    return {
        "c2-p1": ("kARResidualRMSNorm R=8 T=4096 H=7168 launch_with_pdl", c2(1, True)),
        "c2-p1-nopdl": ("kARResidualRMSNorm R=8 T=4096 H=7168 (plain launch)", c2(1)),
        "c2-p0": ("kAllReduce R=8 T=4096 H=7168", c2(0)),
        "c3-p2": ("kARResidualRMSNormFP8Quant R=8 T=8192 H=7168", c3(2)),
        "c3-p6": ("kARResidualRMSNormFP8BlockWiseQuant R=8 T=8192 H=7168", c3(6)),
        "c3-p7": ("kARResidualRMSNormPartialOutFP8BlockWiseQuant R=8 T=8192 H=7168 P=1024", c3(7, 1024)),
        "c3-p8": ("kARResidualRMSNormPartialOut R=8 T=8192 H=7168 P=1024", c3(8, 1024)),
        "c4-p3-linear": ("kARResidualRMSNormFP4Quant R=4 T=16384 H=5120 SF LINEAR", c4(2)),
        "c4-p3-swizzled": ("kARResidualRMSNormFP4Quant R=4 T=16384 H=5120 SF SWIZZLED_128x4", c4(0)),
        "c4-p3-swizzled8": ("kARResidualRMSNormFP4Quant R=4 T=16384 H=5120 SF SWIZZLED_8x4", c4(1)),
        "rs-add": ("kRSAddResidualRMSNorm R=8 T=8192 H=7168, all 8 rank slices (8 PDL calls)", rs_add(8)),
        "rs-add-all": ("kRSAddResidualRMSNorm R=8 T=8192 H=7168, rank -1 (one call)", rs_add(8, True)),
        "rs-add-fp8b": ("kRSAddResidualRMSNormFP8BlockWiseQuant R=8 T=8192 H=7168, all 8 rank slices (8 PDL calls)",
                        rs_add(7)),
        "ag-rms": ("kAllGatherfusedRMS R=8 T=65536 1536|512|64", ag(1)),
        "ag-rms-fp8b": ("kAllGatherfusedRMSFP8BlockWiseQuant R=8 T=65536 1536|512|64", ag(2)),
        "c5-qk": ("MiniMax QK-RMSNorm R=8 T=32768 Q=1024 K=128", c5),
        "single-768": ("single-matrix sharded RMSNorm R=8 T=32768 W=768", single),
        "tp1-p1": ("kARResidualRMSNorm R=1 T=16384 H=5120", tp(1, 1)),
        "tp2-p1": ("kARResidualRMSNorm R=2 T=16384 H=5120", tp(1, 2)),
        "tp2-p3": ("kARResidualRMSNormFP4Quant R=2 T=16384 H=5120 SF LINEAR", tp(3, 2)),
        "tp2-p6": ("kARResidualRMSNormFP8BlockWiseQuant R=2 T=16384 H=5120", tp(6, 2)),
        "tp4-p6": ("kARResidualRMSNormFP8BlockWiseQuant R=4 T=16384 H=5120", tp(6, 4)),
        "c1-p1": ("kARResidualRMSNorm R=2 T=16 H=4096 (latency)", c1),
    }


def measure_rows(dev, stream, peak: float, iters: int) -> dict:
    import torch

    rows = {}
    for key, (label, build) in _case_builders().items():
        if key == "c2-p1":
            continue  # the headline step, timed in run_ours
        with torch.cuda.stream(stream):
            call, nbytes = build(dev, stream)
            if key == "c1-p1":  # L2-resident latency case: stream launches and a CUDA graph
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
                rows[label] = {"us_stream_launch": ms_stream * 1e3, "us_in_cuda_graph": ms_graph * 1e3,
                               "us_in_cuda_graph_pdl": ms_pdl * 1e3, "bytes": nbytes}
            else:
                rows[label] = roofline_entry(nbytes, time_launches(call, iters, stream), peak)
        del call
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
        call, nbytes = build(dev, stream)
        torch.cuda.synchronize()
        for _ in range(launches):
            call()
    torch.cuda.synchronize()
    print(json.dumps({"case": key, "label": label, "launches": launches, "bytes_per_launch": nbytes}))


# (pattern, R, H) and T values of the per-call table: single calls with the inputs cold in L2
SWEEP_SHAPES = ((1, 8, 7168), (6, 8, 7168), (3, 4, 5120), (1, 2, 4096))
SWEEP_TOKENS = (1, 16, 64, 256, 1024, 4096, 16384)


def sweep_t(reps: int = 40) -> None:
    """Per-call time of single fused calls (launch_with_pdl) against T, with the
    inputs cold in L2: a CUDA graph of ``reps`` x (read a 256 MB buffer, call),
    minus a graph of ``reps`` reads alone.  One JSON line per (shape, T)."""
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
    acc = torch.zeros(1, dtype=torch.float32, device=dev)

    def read_flush():
        torch.sum(flush, dim=0, keepdim=True, out=acc)

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

    g_flush = graph_of(read_flush)
    print(json.dumps({"flush_us": per_call_ms(g_flush) * 1e3}), flush=True)
    for p, R, H in SWEEP_SHAPES:
        for T in SWEEP_TOKENS:
            inp = wl.fused_inputs(wl.FusedShape(R=R, T=T, H=H), seed=0, device=dev)
            outs = pkg.new_outputs(p, T, H, dev)
            sf = torch.tensor([100.0], device=dev) if p in (2, 3, 4, 5) else None

            def both():
                read_flush()
                pkg.ts_fused_reduce_norm(p, inp["partials"], inp["residual"], inp["gamma"], EPS, sf,
                                         stream=stream, launch_with_pdl=True, **outs)

            g = graph_of(both)
            ms = per_call_ms(g) - per_call_ms(g_flush)
            nb = fused_bytes(p, R, T, H)
            print(json.dumps({"pattern": p, "R": R, "T": T, "H": H, "us": ms * 1e3,
                              "frac": nb / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind}), flush=True)
            del g, inp, outs
            torch.cuda.synchronize()
            torch.cuda.empty_cache()


def run_ours(args):
    import numpy as np
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
    shape = wl.WORKLOADS["C2"]
    R, T, H = shape.R, shape.T, shape.H
    host_inp = wl.fused_inputs(shape, seed=0)
    parts = host_inp["partials"].to(dev)
    res = host_inp["residual"].to(dev)
    gamma = host_inp["gamma"].to(dev)
    res_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    norm_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    nbytes = fused_bytes(1, R, T, H)

    def step():
        pkg.ts_fused_reduce_norm(1, parts, res, gamma, EPS, residual_out=res_out, norm_out=norm_out,
                                 launch_with_pdl=True, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    with sampler:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                step()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms = max_over_ranks(ms_local, world, dev)
    value = world * T / (ms * 1e-3)
    achieved = nbytes / (ms_local * 1e-3) / 1e9

    # end to end through the C ABI with host buffers.  Headline form: the call
    # is given the pinned host inputs and outputs themselves, and the kernel
    # moves every byte across the host link (NVLink-C2C on Grace-Blackwell).
    # For comparison, the staged form copies the inputs to the device, calls,
    # and copies the outputs back (copy engines, one stream).
    h_parts = host_inp["partials"].pin_memory()
    h_res = host_inp["residual"].pin_memory()
    h_gamma = host_inp["gamma"].pin_memory()
    h_out_res = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    h_out_norm = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    d_parts = torch.empty_like(parts)
    d_res = torch.empty_like(res)

    def e2e_step():
        pkg.ts_fused_reduce_norm(1, h_parts, h_res, h_gamma, EPS, residual_out=h_out_res, norm_out=h_out_norm,
                                 launch_with_pdl=True, stream=stream)

    def staged_step():
        d_parts.copy_(h_parts, non_blocking=True)
        d_res.copy_(h_res, non_blocking=True)
        pkg.ts_fused_reduce_norm(1, d_parts, d_res, gamma, EPS, residual_out=res_out, norm_out=norm_out,
                                 launch_with_pdl=True, stream=stream)
        h_out_res.copy_(res_out, non_blocking=True)
        h_out_norm.copy_(norm_out, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    with torch.cuda.stream(stream):
        e2e_ms = time_launches(e2e_step, e2e_steps, stream, warmup=2)
        staged_ms = time_launches(staged_step, e2e_steps, stream, warmup=2)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    staged_ms = max_over_ranks(staged_ms, world, dev)
    h2d = (h_parts.numel() + h_res.numel() + h_gamma.numel()) * 2
    d2h = (h_out_res.numel() + h_out_norm.numel()) * 2
    del h_parts, h_res, h_gamma, h_out_res, h_out_norm, d_parts, d_res

    rows = None
    if not args.no_rows:
        rows = measure_rows(dev, stream, peak, args.row_iters)

    cpu = cpu_all = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        rps, done, el = oracle_rows_per_second(host_inp, args.cpu_seconds)
        cpu = {"value": rps, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{done} rows of the R=8 T=4096 H=7168 kARResidualRMSNorm workload "
                         f"(8-row batches, wrapping), {el:.1f} s of single-threaded C"}
        if args.cpu_all_cores:
            rps_all, cores = oracle_rows_per_second_all_cores(host_inp, args.cpu_seconds)
            cpu_all = {"value": rps_all, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                       "sample": f"one spawned process per core, each {args.cpu_seconds:.0f} s on its own rows "
                                 f"of the same workload"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "pattern": 1, "R": R, "T": T, "H": H,
                       "launch_with_pdl": True, "bytes_per_step": nbytes,
                       "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB per step > 129 MB); no flush",
                       "parallelism": f"replicas x{world} (rows are independent; no collective)"},
            "achieved_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": f"{peak_kind} HBM copy bandwidth",
                         "traffic": recorded_traffic("fused_rows_kernel pattern 1 R=8 T=4096 H=7168")},
            "e2e": {"value": T * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "mode": "pinned host inputs and outputs passed to the call; the kernel reads and writes "
                            "them across the host link (no staging copy)",
                    "staged": {"value": T * world / (staged_ms * 1e-3), "ms_per_step": staged_ms,
                               "mode": "cudaMemcpyAsync of the inputs to the device, the call, and of the "
                                       "outputs back, on one stream"}},
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "gpu_launches": args.steps,
            "clocks": sampler.summary(),
            "kernel_source_hash": kernel_source_hash(),
            "rows": rows,
        }
        print(json.dumps(line), flush=True)


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
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.sweep_t:
        sweep_t()
    elif args.profile_case:
        profile_case(args.profile_case, args.launches)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

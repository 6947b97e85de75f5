"""Host time of one call of each C-ABI entry point from a plain C99 caller
(tests/c_call_cost.c): every entry point is timed, and each call costs the
calling thread a few microseconds (argument checks, the launch configuration
from per-device cached properties, and the launch itself)."""
import json
import os
import subprocess

import pytest

from reduce_residual_rmsnorm_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

KEYS = ("fused_p1_R8_H7168", "fused_p6_R8_H7168", "fused_p3_R4_H5120_swizzled", "reducescatter_add_R8_H7168",
        "qk_R8", "rms_sharded_R8", "allgather_fp8_R8")


def test_c_abi_host_time_per_call(tmp_path):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = libbuild.build()
    cuda = os.path.dirname(os.path.dirname(libbuild.nvcc()))
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")) if os.path.isdir(d)]
    exe = tmp_path / "c_call_cost"
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(cuda, "include"),
                           os.path.join(ROOT, "tests", "c_call_cost.c"), "-o", str(exe), lib,
                           *[f"-L{d}" for d in libdirs], "-lcudart",
                           "-Wl,-rpath," + os.path.dirname(lib), *[f"-Wl,-rpath,{d}" for d in libdirs]])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    print(got)
    for k in KEYS:
        # a loose bound (shared hosts): a call that queried the driver or the
        # occupancy calculator every time, or synchronised, would still pass
        # this, so the figure itself is what is recorded, not judged here
        assert 0.0 < got[k] < 50.0, (k, got[k])

"""The header is a plain C ABI: a C99 program that includes it (strict
warnings) links against the library and gets the documented statuses back
(no GPU needed: every call returns before any launch), and, on a GPU, a C99
program computes through it on device and on pinned host buffers."""
import os
import subprocess

import pytest

from reduce_residual_rmsnorm_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c99_caller(tmp_path):
    lib = libbuild.build()
    exe = tmp_path / "abi_check"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_check.c"),
                           "-o", str(exe), lib, "-Wl,-rpath," + os.path.dirname(lib)])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


@pytest.mark.gpu
def test_c99_caller_on_the_gpu(tmp_path):
    """The same C99 ABI from a C program on a GPU: device buffers from the CUDA
    runtime's C API and pinned host buffers, values checked in closed form."""
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = libbuild.build()
    cuda = os.path.dirname(os.path.dirname(libbuild.nvcc()))
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")) if os.path.isdir(d)]
    exe = tmp_path / "c_gpu_check"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(cuda, "include"),
                           os.path.join(ROOT, "tests", "c_gpu_check.c"), "-o", str(exe), lib,
                           *[f"-L{d}" for d in libdirs], "-lcudart",
                           "-Wl,-rpath," + os.path.dirname(lib), *[f"-Wl,-rpath,{d}" for d in libdirs]])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr

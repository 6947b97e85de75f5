"""The header is a plain C ABI: a C99 program that includes it (strict
warnings) links against the library and gets the documented statuses back.
No GPU is needed: every call returns before any launch."""
import os
import subprocess

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

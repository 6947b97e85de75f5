"""The all-gather kernels find a gathered row's rank with a multiply-high in
place of a division (csrc/int_div.h, Granlund and Montgomery's method for
division by invariant integers).  The header compiles as plain C++; a host
program checks its quotients against the hardware division (no GPU needed)."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_multiply_high_division(tmp_path):
    exe = tmp_path / "int_div_check"
    subprocess.check_call(["g++", "-std=c++17", "-O2", "-Wall", "-Wextra", "-Werror",
                           "-I", os.path.join(ROOT, "reduce_residual_rmsnorm_gb300", "csrc"),
                           os.path.join(ROOT, "tests", "int_div_check.cpp"), "-o", str(exe)])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr

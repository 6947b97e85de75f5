"""Register and spill budget of the kernels (ptxas -v on a CPU build).

These kernels are HBM-bound and reach the roofline only with enough 16-byte loads in flight per SM: the fused row
kernel must fit two CTAs of up to 512 threads per SM (<= 64 registers)
wherever it holds at most 8 partials and 2 chunks per thread, which covers
every benchmarked workload.  No kernel may spill.
"""
import os
import re
import subprocess

import pytest

from reduce_residual_rmsnorm_gb300 import build as libbuild


@pytest.fixture(scope="module")
def resources(tmp_path_factory):
    out = tmp_path_factory.mktemp("ptxas")
    res = {}
    for src in libbuild.sources():
        if os.path.basename(src) == "api.cu":
            continue
        cmd = [libbuild.nvcc(), *libbuild.ARCH, *libbuild.NVCC_FLAGS, "-Xptxas", "-v", "-c", src, "-o",
               str(out / (os.path.basename(src) + ".o"))]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        name = None
        for line in r.stderr.splitlines():
            m = re.search(r"Compiling entry function '(\S+)'", line)
            if m:
                name = m.group(1)
                res[name] = {}
                continue
            if name is None:
                continue
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m:
                res[name]["spill"] = int(m.group(1)) + int(m.group(2))
            m = re.search(r"Used (\d+) registers", line)
            if m:
                res[name]["regs"] = int(m.group(1))
    return res


def test_no_kernel_spills(resources):
    spilled = {k: v for k, v in resources.items() if v.get("spill", 0)}
    assert not spilled, spilled


def test_fused_row_kernel_register_tiers(resources):
    """<= 8 partials, <= 2 chunks per thread: two 512-thread CTAs per SM (64
    registers), also where a thread issues both chunks' loads together; the
    paired instances (CTAs of up to 1024 threads) are among them and need the
    64 to be launchable at all."""
    # mangled template arguments: fused_rows_kernel<RB, V, Epilogue, ADD>
    checked = 0
    for name, v in resources.items():
        m = re.search(r"fused_rows_kernelILi(\d+)ELi(\d+)ELNS_8EpilogueE\dELb(\d)", name)
        if m and int(m.group(1)) <= 8 and int(m.group(2)) <= 2:
            assert v["regs"] <= 64, (name, v)
            checked += 1
    assert checked >= 20


def test_allgather_norm_kernel_fits_four_ctas_per_sm(resources):
    """Four 256-thread CTAs per SM (64 registers), except the segment form's
    FP8 instances of more than 4 chunks per lane with the gammas requested
    ahead, which the launcher runs only on calls of at most 6 rows per SM,
    at three CTAs per SM (80 registers)."""
    checked = three = 0
    for name, v in resources.items():
        if "ag_norm_kernel" in name or "ag_seg_kernel" in name:
            m = re.search(r"ag_seg_kernelILi(\d+)ELi2ELb1E", name)
            if m and int(m.group(1)) > 4:
                assert v["regs"] <= 80, (name, v)
                three += 1
            else:
                assert v["regs"] <= 64, (name, v)
            checked += 1
    assert checked >= 27 and three >= 1


def test_sharded_norm_kernels_keep_four_ctas_per_sm(resources):
    checked = 0
    for name, v in resources.items():
        m = re.search(r"qk_norm_kernelILi(\d+)ELi(\d+)E", name)
        if m and int(m.group(1)) <= 4:
            assert v["regs"] <= 64, (name, v)
            checked += 1
    assert checked >= 6

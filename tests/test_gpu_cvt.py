"""The GPU conversions of the library (cvt.rn.bf16x2, cvt.rn.satfinite.e4m3x2
and .e2m1x2, and the E4M3 decoder used for NVFP4 scale factors), driven
directly through a test-only probe kernel, equal the oracle's encoders on an
exhaustive sweep: every finite bf16 value at several scales, every rounding
midpoint of each format and its neighbours, zeros of both signs, subnormals,
values past saturation and a million random fp32 bit patterns.  The FP8 1x128
block quantiser's divide-free quotient gives the E4M3 code of the IEEE quotient
over its whole domain (every positive bf16 amax up to +inf, every bf16 n with
|n| <= amax), and the divide-free block scales amax / 448 and amax / 6 are the
IEEE quotients for every non-negative bf16 amax."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from reduce_residual_rmsnorm_gb300 import build as libbuild

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    out = tmp_path_factory.mktemp("cvt") / "libcvt_probe.so"
    subprocess.check_call([libbuild.nvcc(), *libbuild.ARCH, *libbuild.NVCC_FLAGS, "-shared", "-cudart", "static",
                           os.path.join(ROOT, "tests", "cvt_probe.cu"), "-o", str(out)])
    lib = ctypes.CDLL(str(out))
    lib.cvt_probe.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.cvt_probe.restype = ctypes.c_int
    lib.e4m3_values.argtypes = [ctypes.c_void_p]
    lib.e4m3_values.restype = ctypes.c_int
    lib.block_codes_probe.argtypes = [ctypes.c_void_p]
    lib.block_codes_probe.restype = ctypes.c_int
    lib.div_const_probe.argtypes = [ctypes.c_void_p]
    lib.div_const_probe.restype = ctypes.c_int
    return lib


def _run(lib, x):
    dev = torch.device("cuda:0")
    xt = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
    n = xt.numel()
    b = torch.empty(n, dtype=torch.int16, device=dev)
    e8 = torch.empty(n, dtype=torch.uint8, device=dev)
    e4 = torch.empty(n, dtype=torch.uint8, device=dev)
    assert lib.cvt_probe(xt.data_ptr(), n, b.data_ptr(), e8.data_ptr(), e4.data_ptr()) == 0
    torch.cuda.synchronize()
    return b.cpu().numpy().view(np.uint16), e8.cpu().numpy(), e4.cpu().numpy()


def _sweep():
    rng = np.random.default_rng(0)
    codes = np.arange(1 << 16, dtype=np.uint32)
    bf = (codes << 16).view(np.float32)
    bf = bf[np.isfinite(bf)]
    pos = np.sort(bf[bf > 0]).astype(np.float64)
    bf_mid = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    e4 = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    e4_mid = ((e4[:-1] + e4[1:]) / 2).astype(np.float32)
    e2 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float64)
    e2_mid = ((e2[:-1] + e2[1:]) / 2).astype(np.float32)
    mids = np.concatenate([bf_mid, e4_mid, e2_mid])
    near = np.concatenate([np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(np.inf))])
    rnd = rng.integers(0, 0x7F800000, 1_000_000, dtype=np.uint32).view(np.float32)
    with np.errstate(over="ignore"):  # scaled past fp32's range: +-inf, also swept
        scaled = np.concatenate([bf * np.float32(s) for s in (1.0, 3.0, 2.0 ** -8, 2.0 ** 8, 448.0 / 3.0)])
    special = np.array([0.0, 2.0 ** -149, 2.0 ** -126, 448.0, 464.0, 480.0, 1e30, np.inf, 6.0, 7.0, 1e-45],
                       np.float32)
    x = np.concatenate([bf, mids, near, rnd, scaled, special]).astype(np.float32)
    x = x[np.isfinite(x) | np.isinf(x)]
    return np.concatenate([x, -x]).astype(np.float32)


def test_conversions_match_the_oracle_encoders(probe):
    x = _sweep()
    b, e8, e4 = _run(probe, x)
    fin = np.isfinite(x)
    assert np.array_equal(b[fin], oracle.bf16_encode(x[fin]))
    assert np.array_equal(e8, oracle.e4m3_encode(x))
    assert np.array_equal(e4, oracle.e2m1_encode(x))


def test_e4m3_decoder_matches_the_oracle(probe):
    out = torch.empty(256, dtype=torch.float32, device="cuda:0")
    assert probe.e4m3_values(out.data_ptr()) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    fin = np.isfinite(want)  # 0x7F / 0xFF are the NaN codes
    assert np.array_equal(got[fin].view(np.uint32), want[fin].view(np.uint32))
    assert np.isnan(got[~fin]).all()


def test_block_quotient_codes_equal_the_ieee_divide_everywhere(probe):
    mism = torch.zeros(0x7F81, dtype=torch.int32, device="cuda:0")
    assert probe.block_codes_probe(mism.data_ptr()) == 0
    torch.cuda.synchronize()
    bad = mism.cpu().numpy()
    assert bad.sum() == 0, {hex(int(a)): int(bad[a]) for a in np.nonzero(bad)[0][:10]}


def test_block_scale_quotients_equal_the_ieee_divide_everywhere(probe):
    mism = torch.zeros(2, dtype=torch.int32, device="cuda:0")
    assert probe.div_const_probe(mism.data_ptr()) == 0
    torch.cuda.synchronize()
    assert mism.cpu().tolist() == [0, 0]

"""SWIZZLED_128x4 pinned to a consumer of the layout: an NVFP4 GEMM.

The pages only name SWIZZLED_128x4 (reading c14 defines the map), so the
oracle's map is checked here against the NVFP4 block-scaled matmul of the
CUDA libraries that PyTorch calls (`torch._scaled_mm` with float4_e2m1fn_x2
operands and float8_e4m3fn 1x16 block scales, which reads its scales in the
swizzled 128x4 layout).  A is random E2M1 codes with random per-16 block
scales placed by the oracle's map; B is the identity with every scale 1, so
C = dequant(A) exactly (one nonzero product per output, all values exact in
bf16).  The same A with its scales left in the plain row-major layout must
give a different C, which shows the check tells the layouts apart.  Where the
installed PyTorch or GPU has no NVFP4 matmul, the test is skipped.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

M = N = K = 128


def _pack(codes):
    """[rows, K] E2M1 codes -> [rows, K/2] bytes, even element in the low nibble."""
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def _run(dev, a_codes, sf_a_bytes, b_codes, sf_b_bytes):
    f4 = torch.float4_e2m1fn_x2
    a = torch.from_numpy(_pack(a_codes)).to(dev).view(f4)
    b = torch.from_numpy(_pack(b_codes)).to(dev).view(f4)
    sa = torch.from_numpy(sf_a_bytes).to(dev).view(torch.float8_e4m3fn)
    sb = torch.from_numpy(sf_b_bytes).to(dev).view(torch.float8_e4m3fn)
    c = torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    return c.float().cpu().numpy()


def test_swizzled_128x4_is_the_nvfp4_gemm_layout():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this PyTorch has no float4_e2m1fn_x2")
    dev = torch.device("cuda:0")
    oracle.load()
    rng = np.random.default_rng(5)
    a_codes = rng.integers(0, 16, (M, K)).astype(np.uint8)
    sf_a = rng.integers(0x28, 0x48, (M, K // 16)).astype(np.uint8)  # 2^-2 .. 2^1.9, positive
    b_codes = np.zeros((N, K), np.uint8)
    b_codes[np.arange(N), np.arange(K)] = 0x2  # E2M1 1.0
    sf_b = np.full((N, K // 16), 0x38, np.uint8)  # E4M3 1.0
    try:
        got = _run(dev, a_codes, oracle.sf_swizzle_128x4(sf_a).reshape(-1), b_codes,
                   oracle.sf_swizzle_128x4(sf_b).reshape(-1))
    except (RuntimeError, TypeError, NotImplementedError) as e:  # no NVFP4 matmul here
        pytest.skip(f"no NVFP4 scaled matmul available: {str(e).splitlines()[0]}")
    want = (oracle.e2m1_decode(a_codes).astype(np.float64) *
            np.repeat(oracle.e4m3_decode(sf_a).astype(np.float64), 16, axis=1))
    assert np.array_equal(got.astype(np.float64), want)
    plain = _run(dev, a_codes, sf_a.reshape(-1), b_codes, oracle.sf_swizzle_128x4(sf_b).reshape(-1))
    assert not np.array_equal(plain.astype(np.float64), want)

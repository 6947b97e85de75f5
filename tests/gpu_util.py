"""Helpers for the GPU parity tests: guarded output buffers and host copies."""
import numpy as np
import torch

GUARD = 256
FILL = 0xA5


class Guarded:
    """An output tensor inside a buffer with GUARD bytes of 0xA5 on both sides.

    The tensor itself also starts filled with 0xA5, so an element the kernel
    fails to write shows up as a mismatch, and a write outside the tensor
    shows up in ``intact()``."""

    def __init__(self, shape, dtype, device):
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((GUARD + nbytes + GUARD,), FILL, dtype=torch.uint8, device=device)
        self.nbytes = nbytes
        self.t = self.buf[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool((b[:GUARD] == FILL).all() and (b[GUARD + self.nbytes:] == FILL).all())


def guarded_outputs(pattern, T, H, device, partial_cols=0, layout=2, allreduce=True):
    """Guarded outputs of a pattern; ``layout`` is the NVFP4 SF layout code
    (0 SWIZZLED_128x4, 1 SWIZZLED_8x4, 2 LINEAR)."""
    p = int(pattern)
    bf = torch.bfloat16
    spec = {}
    if p == 0 or allreduce:
        spec["allreduce_out"] = ((T, H), bf)
    if p != 0:
        spec["residual_out"] = ((T, H), bf)
    if p in (1, 4, 5, 8):
        spec["norm_out"] = ((T, H), bf)
    if p in (7, 8):
        spec["partial_norm_out"] = ((T, partial_cols), bf)
    if p in (2, 4, 6, 7):
        spec["quant_out"] = ((T, H), torch.uint8)
    if p in (3, 5):
        spec["quant_out"] = ((T, H // 2), torch.uint8)
        if layout == 2:
            spec["scale_out"] = ((T, H // 16), torch.uint8)
        else:
            tile = 128 if layout == 0 else 8
            spec["scale_out"] = (((T + tile - 1) // tile * tile, (H // 16 + 3) // 4 * 4), torch.uint8)
    if p in (6, 7):
        spec["scale_out"] = ((T, H // 128), torch.float32)
    return {k: Guarded(s, d, device) for k, (s, d) in spec.items()}


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()

"""Device placement helpers for the GPU parity tests.

Places host arrays on the GPU inside a larger buffer so that tests can choose
the base-pointer offset (misalignment) and the row stride, and can check that
nothing outside the logical matrix was written (canaries).
"""
from __future__ import annotations

import numpy as np
import torch

CANARY_F32 = np.float32(-1234.5)
CANARY_U16 = np.uint16(0x7F81)  # a bf16 signalling-NaN pattern no kernel writes


class Placed:
    def __init__(self, buf, view, offset, rows, ld, cols, canary_bits):
        self.buf, self.t, self.offset = buf, view, offset
        self.rows, self.ld, self.cols = rows, ld, cols
        self.canary_bits = canary_bits

    def canaries_intact(self) -> bool:
        """True when every element outside the logical [rows, cols] block still
        holds the canary pattern."""
        raw = self.buf.view(torch.int16 if self.buf.element_size() == 2 else torch.int32)
        host = raw.cpu().numpy()
        mask = np.ones(host.shape, dtype=bool)
        for r in range(self.rows):
            s = self.offset + r * self.ld
            mask[s:s + self.cols] = False
        return bool((host[mask] == self.canary_bits).all())


def place(arr: np.ndarray, offset: int = 0, ld: int | None = None, pad: int = 40) -> Placed:
    """Copy a 2-D fp32 or bf16-bits (uint16) array to the GPU with a chosen
    element offset from a 512-byte aligned base and a chosen row stride."""
    rows, cols = arr.shape
    ld = cols if ld is None else ld
    n = offset + (rows - 1) * ld + cols + pad
    if arr.dtype == np.float32:
        canary = np.full(n, CANARY_F32, np.float32)
        bits = int(canary.view(np.int32)[0])
        tdtype = torch.float32
    elif arr.dtype == np.uint16:
        canary = np.full(n, CANARY_U16, np.uint16)
        bits = int(canary.view(np.int16)[0])
        tdtype = torch.bfloat16
    else:
        raise TypeError(arr.dtype)
    for r in range(rows):
        canary[offset + r * ld: offset + r * ld + cols] = arr[r]
    if tdtype == torch.float32:
        buf = torch.from_numpy(canary).cuda()
    else:
        buf = torch.from_numpy(canary.view(np.int16)).cuda().view(torch.bfloat16)
    view = buf.as_strided((rows, cols), (ld, 1), offset)
    return Placed(buf, view, offset, rows, ld, cols, bits)


def empty_like_placed(rows: int, cols: int, dtype, offset: int = 0, ld: int | None = None) -> Placed:
    z = np.zeros((rows, cols), np.float32 if dtype == torch.float32 else np.uint16)
    p = place(z, offset, ld)
    # overwrite the logical block with junk so a missing write is visible
    p.t.fill_(float("nan") if dtype == torch.float32 else float("nan"))
    return p


def bf16_to_f32_host(t: torch.Tensor) -> np.ndarray:
    bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

"""Device-side helpers for the GPU tests: upload, sentinel-filled outputs with canary
guard bands, and read-back."""
from __future__ import annotations

import numpy as np
import torch

from cases import SENTINEL_BF16, SENTINEL_F32

GUARD_ROWS = 2


def dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


class GuardedOut:
    """An output tensor of shape [rows, n] surrounded by GUARD_ROWS guard rows on each
    side, everything pre-filled with a NaN sentinel pattern."""

    def __init__(self, rows: int, n: int, out: str):
        self.rows, self.n, self.out = rows, n, out
        if out == "bf16":
            self.buf = torch.full((rows + 2 * GUARD_ROWS, n), SENTINEL_BF16, dtype=torch.int16, device="cuda")
            self.tensor = self.buf[GUARD_ROWS:GUARD_ROWS + rows].view(torch.bfloat16)
            self.sentinel = SENTINEL_BF16
        else:
            self.buf = torch.full((rows + 2 * GUARD_ROWS, n), SENTINEL_F32, dtype=torch.int32, device="cuda")
            self.tensor = self.buf[GUARD_ROWS:GUARD_ROWS + rows].view(torch.float32)
            self.sentinel = SENTINEL_F32

    def fill_from(self, values: np.ndarray):
        """Replace the inner rows with `values` (float32 only; used for D aliasing C)."""
        self.tensor.copy_(torch.from_numpy(values.astype(np.float32)))

    def host_bits(self) -> np.ndarray:
        b = self.buf.cpu().numpy()
        return b.view(np.uint16) if self.out == "bf16" else b.view(np.uint32)

    def check_guards(self):
        bits = self.host_bits()
        s = np.uint16(self.sentinel) if self.out == "bf16" else np.uint32(self.sentinel)
        assert np.all(bits[:GUARD_ROWS] == s) and np.all(bits[GUARD_ROWS + self.rows:] == s), \
            "write outside the output tensor"

    def inner_bits(self) -> np.ndarray:
        return self.host_bits()[GUARD_ROWS:GUARD_ROWS + self.rows]

    def values(self) -> np.ndarray:
        bits = self.inner_bits()
        with np.errstate(invalid="ignore"):     # untouched rows hold a NaN sentinel
            if self.out == "bf16":
                return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            return bits.view(np.float32).astype(np.float64)

    def is_sentinel(self) -> np.ndarray:
        s = np.uint16(self.sentinel) if self.out == "bf16" else np.uint32(self.sentinel)
        return np.all(self.inner_bits() == s, axis=1)

"""Helpers for the GPU parity tests: guarded device buffers, transfers to
numpy, and the comparison metrics.  No arithmetic of the method lives here."""
from __future__ import annotations

import numpy as np
import torch

PAD = 256  # guard entries before and after every caller buffer (512 B of bf16)
BF16_CANARY = 0x7FA5  # a NaN bit pattern nothing in a step writes
F32_CANARY = 0x7FC0FFEE


class Guarded:
    """A 1-D device buffer with canary regions on both sides.  ``t`` is the
    16-byte aligned view handed to the library; ``intact()`` checks that the
    canaries were not touched."""

    def __init__(self, n: int, dtype: torch.dtype, device="cuda"):
        self.n, self.dtype = n, dtype
        self.full = torch.empty(n + 2 * PAD, dtype=dtype, device=device)
        self._bits().fill_(self._canary())
        self.t = self.full[PAD:PAD + n]
        assert self.t.data_ptr() % 16 == 0

    def _bits(self):
        return self.full.view(torch.int16 if self.dtype == torch.bfloat16 else torch.int32)

    def _canary(self):
        return BF16_CANARY if self.dtype == torch.bfloat16 else F32_CANARY

    def intact(self) -> bool:
        b = self._bits()
        c = self._canary()
        return bool((b[:PAD] == c).all() and (b[PAD + self.n:] == c).all())


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def bits_equal(a: np.ndarray, b: np.ndarray) -> bool:
    """Bit-for-bit equality of float32 arrays (NaN patterns included)."""
    return np.array_equal(np.ascontiguousarray(a, np.float32).view(np.uint32),
                          np.ascontiguousarray(b, np.float32).view(np.uint32))


def rel_err(a: np.ndarray, ref: np.ndarray) -> float:
    """max_i |a_i - ref_i| / max(|ref_i|, rms(ref)): relative error with the
    denominator floored at the array's RMS, so that entries near a zero
    crossing (m after cancellation) are judged on the array's scale."""
    ref64 = ref.astype(np.float64)
    rms = float(np.sqrt(np.mean(ref64 ** 2))) if ref.size else 0.0
    den = np.maximum(np.abs(ref64), rms if rms > 0 else 1e-300)
    return float(np.max(np.abs(a.astype(np.float64) - ref64) / den)) if ref.size else 0.0


def bf16_ulp(a: np.ndarray, b: np.ndarray) -> int:
    def ordered(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return int(np.abs(ordered(a) - ordered(b)).max()) if a.size else 0

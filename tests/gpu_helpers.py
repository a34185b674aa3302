"""Shared helpers for the GPU parity tests: moving seeded operands to the
device in strided, guarded buffers and comparing against the oracle."""

import numpy as np
import torch

import gemm_inputs as gi

# bf16 / fp32 sentinels written around C; any change means an out-of-range write.
SENTINEL_BF16 = 0x7FBF  # a NaN pattern no rounding produces
SENTINEL_F32 = np.float32(-1.2345e38)


def bf16_to_dev(bits: np.ndarray, ld: int | None = None) -> torch.Tensor:
    """uint16 bf16 bits (rows x cols) -> CUDA bfloat16 view with row pitch ld."""
    rows, cols = bits.shape
    ld = ld or cols
    buf = torch.zeros((rows, ld), dtype=torch.int16, device="cuda")
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return buf.view(torch.bfloat16)[:, :cols]


def f32_to_dev(x: np.ndarray, ld: int | None = None) -> torch.Tensor:
    rows, cols = x.shape
    ld = ld or cols
    buf = torch.zeros((rows, ld), dtype=torch.float32, device="cuda")
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return buf[:, :cols]


def bf16_from_dev(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class GuardedC:
    """C (M x N, pitch ldc) inside a buffer with one spare row and spare
    columns, all pre-filled with a sentinel."""

    def __init__(self, M, N, ldc, dtype, init=None):
        self.M, self.N, self.ldc, self.dtype = M, N, ldc, dtype
        if dtype == "bf16":
            self.buf = torch.full((M + 1, ldc), SENTINEL_BF16, dtype=torch.int16, device="cuda")
            if init is not None:
                self.buf[:M, :N] = torch.from_numpy(np.ascontiguousarray(init).view(np.int16)).cuda()
            self.view = self.buf.view(torch.bfloat16)[:M, :N]
        else:
            self.buf = torch.full((M + 1, ldc), float(SENTINEL_F32), dtype=torch.float32,
                                  device="cuda")
            if init is not None:
                self.buf[:M, :N] = torch.from_numpy(np.ascontiguousarray(init)).cuda()
            self.view = self.buf[:M, :N]

    def result(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_from_dev(self.view)
        return self.view.cpu().numpy()

    def guards_intact(self) -> bool:
        b = self.buf.cpu().numpy()
        if self.dtype == "bf16":
            b = b.view(np.uint16)
            s = SENTINEL_BF16
            return bool((b[:self.M, self.N:] == s).all() and (b[self.M, :] == s).all())
        s = SENTINEL_F32
        return bool((b[:self.M, self.N:] == s).all() and (b[self.M, :] == s).all())


def widen(result: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return gi.bf16_bits_to_f32(result).astype(np.float64)
    return result.astype(np.float64)


def bf16_tolerance_violations(got_f64: np.ndarray, ref_f64: np.ndarray) -> int:
    """Elements breaking |C - C_ref| <= 2^-7 |C_ref| + 1e-2."""
    bad = np.abs(got_f64 - ref_f64) > (2.0**-7) * np.abs(ref_f64) + 1e-2
    bad |= ~np.isfinite(got_f64)
    return int(bad.sum())

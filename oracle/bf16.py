"""bfloat16 helpers for the oracle (test infrastructure only).

bfloat16 is the upper 16 bits of an IEEE binary32.  Rounding from binary32
to bfloat16 is round-to-nearest-even on the dropped 16 bits; NaNs stay NaN.
"""
from __future__ import annotations

import numpy as np


def round_f32_to_bf16_bits(x) -> np.ndarray:
    """Round binary32 values to bfloat16 (RNE) and return the uint16 bit patterns."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    # keep NaNs NaN (quiet, same sign)
    out = np.where(nan, ((bits >> np.uint64(16)).astype(np.uint16) | np.uint16(0x0040)), out)
    return out.astype(np.uint16)


def bits_to_f32(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to binary32 values (exact)."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def round_to_bf16(x) -> np.ndarray:
    """Round binary32 values to the nearest bfloat16 value, returned as binary32."""
    return bits_to_f32(round_f32_to_bf16_bits(x))


def ulp(x) -> np.ndarray:
    """One bfloat16 unit in the last place at the magnitude of ``x`` (float64).

    ulp(x) = 2^(max(floor(log2|x|), -126) - 7); at x = 0 it is the smallest
    bfloat16 subnormal 2^-133.
    """
    a = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126.0), -126.0)
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def torch_bf16_to_f64(t) -> np.ndarray:
    """A bf16 torch tensor (any device) as a float64 numpy array (exact)."""
    import torch

    return t.detach().to("cpu").to(torch.float32).numpy().astype(np.float64)


def torch_bf16_bits(t) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 torch tensor."""
    import torch

    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)

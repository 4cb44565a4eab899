"""Exact widening of stored inputs to float64 (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""
import numpy as np


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """bf16 bit patterns (uint16), fp32 or fp64 values -> float64, exactly."""
    if dtype == "f64":
        return np.asarray(a, dtype=np.float64)
    if dtype == "bf16":
        assert a.dtype == np.uint16
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def bf16_round_f64(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), as float64.

    Used only where a comparison needs the bf16 value a stored output would
    take; the rounding goes through fp32 first (fp64 -> fp32 -> bf16).
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    r = ((u + bias) >> 16).astype(np.uint32) << np.uint32(16)
    return r.view(np.float32).astype(np.float64)

"""Exact widening of stored inputs to float64 (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""
import numpy as np


def e4m3_to_f64(a: np.ndarray) -> np.ndarray:
    """FP8 E4M3 bit patterns (uint8) -> float64, exactly.

    The OCP 8-bit floating-point format E4M3 (the "FP8 KV cache data type" of the
    InfiniteHiP summary's throughput runs): 1 sign bit, 4 exponent bits with bias 7,
    3 mantissa bits; exponent 0 holds the subnormals m * 2^-9; there is no infinity and
    S.1111.111 is NaN, the only code that is not a number.
    """
    a = np.asarray(a)
    assert a.dtype == np.uint8
    u = a.astype(np.int64)
    s = np.where(u >> 7, -1.0, 1.0)
    e = (u >> 3) & 15
    m = u & 7
    v = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e - 10.0))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return s * v


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """bf16 bit patterns (uint16), FP8 E4M3 bit patterns (uint8), fp32 or fp64 values
    -> float64, exactly."""
    if dtype == "f64":
        return np.asarray(a, dtype=np.float64)
    if dtype == "e4m3":
        return e4m3_to_f64(a)
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

"""Seeded synthetic workloads for the sparse-attention hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no scoring, selection, softmax or index building).  Both
the fp64 oracle and the CUDA path consume exactly the arrays produced here.
"""
from .workloads import (  # noqa: F401
    DecodeCase,
    PrefillCase,
    f32_to_bf16_bits,
    f32_to_e4m3_bits,
    with_fp8_kv,
    decode_case,
    decode_steps,
    prefill_case,
    decode_tiny,
    decode_128k,
    decode_1m,
    decode_batch16,
    prefill_128k,
)

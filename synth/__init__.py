"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA-side tests.

This module only draws and rounds random numbers: it holds none of the
arithmetic of the method (no attention, no quantisation, no projection).
Both the float64 oracle and the CUDA library consume exactly the tensors
produced here, so "same seeded inputs" holds by construction.
"""

from .inputs import (  # noqa: F401
    Shapes,
    TINY,
    LAYER_1P3B,
    seed_rng,
    gaussian_bf16,
    gaussian_outliers_bf16,
    chunk_qkv,
    chunk_qkv_device,
    device_seed,
    recache_inputs,
    project_inputs,
    gains,
    bf16_to_f64,
)

"""Seeded synthetic inputs for the flash-attention backward.

This package only makes input data: counter-based random numbers, the
quantizers that turn f32 rows into raw F16 / q8_0 / q4_0 cache bytes, and
masks.  It holds none of the backward's arithmetic.  Both the CPU oracle and
the CUDA path consume exactly the arrays produced here.
"""
from .gen import (  # noqa: F401
    TYPE_F32, TYPE_F16, TYPE_Q8_0, TYPE_Q4_0, TYPE_NAMES,
    Problem, make_problem, from_config, config, CONFIGS, row_bytes,
    normal, uniform, quantize_rows, sample_indices,
)
from . import device  # noqa: F401,E402

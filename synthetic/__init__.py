"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark.

This package only draws random numbers in the shapes and value distributions of
the workloads.  It holds none of the NVFP4 arithmetic (no decoding, no
quantisation, no scale layout): both the CUDA path and the oracle consume what
it produces.
"""

from .generators import (  # noqa: F401
    E4M3_POS_NORMAL_2M4_2P4,
    E4M3_SUBNORMAL_BYTES,
    alpha_uniform,
    bf16_normal,
    gemm_square_inputs,
    packed_codes_uniform,
    rng_for,
    scales_uniform_normal,
    scales_with_zero_and_subnormal,
)

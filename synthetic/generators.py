"""Seeded generators for the NVFP4 workloads.

Every tensor is drawn from its own numpy ``Generator(PCG64)`` stream so that a
tensor of one size does not shift the draws of another.  Streams are derived
from ``(seed, name)``; the order of calls does not matter.

Distributions (their readings are listed in the design notes of the repository):

* packed E2M1 codes: every byte uniform over 0..255, i.e. both 4-bit codes of
  the byte independent and uniform over all 16 codes.
* block scales, square GEMM workloads: uniform over the 65 E4M3 encodings
  0x18..0x58, which are exactly the positive normal values in [2^-4, 2^4].
* block scales, large square workloads: 5 % of blocks zero, 5 % uniform over the
  seven E4M3 subnormal encodings 0x01..0x07, the rest as above.
* alpha: uniform over [0.25, 4] in float32.
* LLM / decode activations and weights: normal samples rounded to bfloat16
  (bit patterns returned as uint16).
"""

from __future__ import annotations

import hashlib

import numpy as np

# E4M3 encodings of the positive normal values 2^-4 .. 2^4 (exponent field 3..11).
E4M3_POS_NORMAL_2M4_2P4 = np.arange(0x18, 0x59, dtype=np.uint8)
# E4M3 subnormal encodings (exponent field 0, mantissa 1..7).
E4M3_SUBNORMAL_BYTES = np.arange(0x01, 0x08, dtype=np.uint8)


def rng_for(seed: int, name: str) -> np.random.Generator:
    """A PCG64 stream for tensor ``name`` under ``seed``."""
    h = hashlib.sha256(f"{int(seed)}:{name}".encode()).digest()
    return np.random.Generator(np.random.PCG64(int.from_bytes(h[:8], "little")))


def packed_codes_uniform(rows: int, K: int, seed: int, name: str) -> np.ndarray:
    """[rows, K/2] uint8; each nibble uniform over the 16 E2M1 codes."""
    assert K % 2 == 0
    return rng_for(seed, name).integers(0, 256, size=(rows, K // 2), dtype=np.uint8)


def scales_uniform_normal(rows: int, K: int, seed: int, name: str) -> np.ndarray:
    """[rows, K/16] uint8, uniform over the E4M3 encodings of 2^-4..2^4."""
    assert K % 16 == 0
    g = rng_for(seed, name)
    idx = g.integers(0, E4M3_POS_NORMAL_2M4_2P4.size, size=(rows, K // 16))
    return E4M3_POS_NORMAL_2M4_2P4[idx]


def scales_with_zero_and_subnormal(rows: int, K: int, seed: int, name: str,
                                   p_zero: float = 0.05, p_sub: float = 0.05) -> np.ndarray:
    """[rows, K/16] uint8: P(zero)=p_zero, P(subnormal)=p_sub, else normal 2^-4..2^4."""
    assert K % 16 == 0
    g = rng_for(seed, name)
    shape = (rows, K // 16)
    u = g.random(shape)
    normal = E4M3_POS_NORMAL_2M4_2P4[g.integers(0, E4M3_POS_NORMAL_2M4_2P4.size, size=shape)]
    sub = E4M3_SUBNORMAL_BYTES[g.integers(0, E4M3_SUBNORMAL_BYTES.size, size=shape)]
    out = np.where(u < p_zero, np.uint8(0), np.where(u < p_zero + p_sub, sub, normal))
    return out.astype(np.uint8)


def alpha_uniform(seed: int, name: str = "alpha", lo: float = 0.25, hi: float = 4.0) -> float:
    """A float32 value uniform over [lo, hi], returned as a Python float."""
    return float(np.float32(rng_for(seed, name).uniform(lo, hi)))


def bf16_normal(rows: int, cols: int, seed: int, name: str, std: float = 1.0) -> np.ndarray:
    """[rows, cols] uint16 bfloat16 bit patterns of N(0, std^2) samples.

    The float32 samples are rounded to bfloat16 by torch's CPU conversion, a
    library call; the result is only used as an input.
    """
    import torch

    x = rng_for(seed, name).standard_normal(size=(rows, cols), dtype=np.float32) * np.float32(std)
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def gemm_square_inputs(M: int, N: int, K: int, seed: int = 0, scales: str = "normal"):
    """Operands of the square W4A4 workloads: (A, SFA, B, SFB) with row-major scales.

    ``scales`` is "normal" (uniform over 2^-4..2^4) or "zero_sub" (5 % zero and
    5 % subnormal blocks mixed in).
    """
    A = packed_codes_uniform(M, K, seed, "A")
    B = packed_codes_uniform(N, K, seed, "B")
    if scales == "normal":
        SFA = scales_uniform_normal(M, K, seed, "SFA")
        SFB = scales_uniform_normal(N, K, seed, "SFB")
    elif scales == "zero_sub":
        SFA = scales_with_zero_and_subnormal(M, K, seed, "SFA")
        SFB = scales_with_zero_and_subnormal(N, K, seed, "SFB")
    else:
        raise ValueError(scales)
    return A, SFA, B, SFB

"""NVFP4 oracle: a plain, slow, obviously correct CPU statement of what the
NVFP4 block-scaled path computes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The library never calls it, and it shares no code, table or helper with
the CUDA path.

Sources (cited by page title and section):

* [P1] Colfax Research, "Optimizing an NVFP4 Blockscaled GEMM on RTX PRO 6000
  Blackwell GPU (SM120)".
* [P2] TileLang PR #3290, "[CUDA] Add an SM120 W4A16 NVFP4 GEMM example for
  decode-sized batches".

Number formats (E2M1 codes, one E4M3 scale per 16 K-elements, FP32 per-tensor
alpha): [P1] Version 2 (input footprint: 4 bits per element, 8 bits per 16
elements) and Version 5 (one scale broadcast to the 16 elements of a micro-block);
[P2] Design (two E2M1 codes per byte, one unsigned E4M3 scale per block, and a
weight scale that is per tensor or per output column).

Everything is computed in float64 (exact for the W4A4 workloads: each product is
an integer multiple of 2^-20, see ``gemm_exact_units``).  Where the pages fix
float32 arithmetic (quantisation, which decides integer codes) the oracle uses
IEEE float32 operations one at a time, never fused.

Pinned by tests/test_oracle_*.py; every function here has at least one pin that
is independent of the function itself (closed forms, brute force with exact
rationals, integer GEMMs, library decoders, hand-worked golden values).
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Decoding tables
# ---------------------------------------------------------------------------

#: Magnitudes of the E2M1 codes 0..7 (sign in bit 3): the 8 values the 4-bit
#: format represents, [P1] Version 2 / [P2] Design.
E2M1_MAGNITUDE = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_table() -> np.ndarray:
    """float64[16]: value of each 4-bit E2M1 code (bit 3 = sign, gives +-0)."""
    t = np.empty(16, dtype=np.float64)
    for c in range(16):
        mag = E2M1_MAGNITUDE[c & 7]
        t[c] = -mag if (c & 8) else mag
    return t


def e4m3_value(byte: int) -> float:
    """Value of one E4M3 byte (1 sign, 4 exponent bits bias 7, 3 mantissa bits).

    Normal (exponent field e in 1..15): (1 + m/8) * 2^(e-7).  Subnormal (e = 0):
    m * 2^-9.  0x7F and 0xFF are NaN; the format has no infinities.
    """
    s = -1.0 if (byte & 0x80) else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_table() -> np.ndarray:
    """float64[256]: value of each E4M3 byte."""
    return np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


_E2M1 = e2m1_table()
_E4M3 = e4m3_table()


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """[R, K/2] packed bytes -> [R, K] 4-bit codes; low nibble is the even k."""
    packed = np.asarray(packed, dtype=np.uint8)
    R, H = packed.shape
    out = np.empty((R, 2 * H), dtype=np.uint8)
    out[:, 0::2] = packed & 0x0F
    out[:, 1::2] = packed >> 4
    return out


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """[R, K] 4-bit codes -> [R, K/2] bytes (inverse of ``unpack_codes``)."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] & 0x0F) | ((codes[:, 1::2] & 0x0F) << 4)


def dequantize(packed: np.ndarray, sf_rowmajor: np.ndarray) -> np.ndarray:
    """float64 [R, K]: element value code * scale, scale = SF[r, k // 16].

    [P1] Version 5: one scale factor applies to all 16 elements of a micro-block.
    """
    codes = unpack_codes(packed)
    R, K = codes.shape
    sf = np.asarray(sf_rowmajor, dtype=np.uint8)
    assert sf.shape == (R, K // 16), (sf.shape, R, K)
    scale = np.repeat(_E4M3[sf], 16, axis=1)
    return _E2M1[codes] * scale


# ---------------------------------------------------------------------------
# W4A4 GEMM:  D[m,n] = alpha * sum_k (A[m,k] SFA[m,k/16]) (B[n,k] SFB[n,k/16])
# [P1] Version 1 (the GEMM) and Version 3 (alpha applied in FP32 to the
# accumulator before the conversion to the output type).
# ---------------------------------------------------------------------------


def gemm(A, SFA, B, SFB, alpha: float):
    """Full reference.  Returns (ref, abs_sum), both float64 [M, N].

    ref     = alpha * sum_k a_k b_k        (a, b the dequantised elements)
    abs_sum = sum_k |a_k b_k|              (for the tolerance bound)
    A is [M, K/2] and B is [N, K/2], both K-major; scales row-major.
    """
    a = dequantize(A, SFA)
    b = dequantize(B, SFB)
    ref = (a @ b.T) * float(alpha)
    abs_sum = np.abs(a) @ np.abs(b).T
    return ref, abs_sum


def gemm_at(A, SFA, B, SFB, alpha: float, rows, cols):
    """Reference at the sampled outputs (rows[i], cols[i]); float64 [n] each."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    a = dequantize(A[rows], SFA[rows])
    b = dequantize(B[cols], SFB[cols])
    prod = a * b
    return prod.sum(axis=1) * float(alpha), np.abs(prod).sum(axis=1)


def gemm_tile(A, SFA, B, SFB, alpha: float, r0: int, r1: int, c0: int, c1: int):
    """Reference of the output tile [r0:r1, c0:c1]."""
    return gemm(A[r0:r1], SFA[r0:r1], B[c0:c1], SFB[c0:c1], alpha)


def gemm_exact_units(A, SFA, B, SFB) -> np.ndarray:
    """int64 [M, N]: sum_k a_k b_k exactly, in units of 2^-20.

    Every E2M1 value is a multiple of 1/2 and every E4M3 value a multiple of
    2^-9, so each element is an integer times 2^-10 and each product an integer
    times 2^-20.  The element integers are at most 12 * 448 * 512 < 2^22, so for
    K <= 2^17 the sum fits in int64.  Scales must be finite.
    """
    ca = unpack_codes(A).astype(np.int64)
    cb = unpack_codes(B).astype(np.int64)
    code_int = np.array([round(2 * v) for v in _E2M1], dtype=np.int64)  # value * 2
    sf_int = np.array([0 if np.isnan(v) else round(abs(v) * 512) * (1 if v >= 0 else -1)
                       for v in _E4M3], dtype=np.int64)                  # value * 2^9
    ia = code_int[ca] * np.repeat(sf_int[np.asarray(SFA)], 16, axis=1)
    ib = code_int[cb] * np.repeat(sf_int[np.asarray(SFB)], 16, axis=1)
    return ia @ ib.T


def tolerance(ref, abs_sum, alpha: float):
    """Per-element acceptance bound: 2^-8 |ref| + 1e-6 |alpha| sum_k |a_k b_k|."""
    return np.abs(ref) * 2.0 ** -8 + 1e-6 * abs(float(alpha)) * abs_sum


# ---------------------------------------------------------------------------
# bfloat16 helpers (bit-level, round to nearest even)
# ---------------------------------------------------------------------------


def bf16_bits_to_f64(bits) -> np.ndarray:
    """uint16 bfloat16 bit patterns -> float64 values (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def f32_to_bf16_rne(x) -> np.ndarray:
    """float32 -> bfloat16 bits, round to nearest, ties to even; NaN stays NaN."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint32)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = np.where(nan, ((u >> 16) | 0x40).astype(np.uint32), r)
    return (r & 0xFFFF).astype(np.uint16)


# ---------------------------------------------------------------------------
# Quantisation (producer of the W4A4 operands of the LLM-linear workloads)
#
# The pages name the target format ([P2] Design: packed E2M1 + E4M3 block scale
# + global scale) but print no quantiser.  The reading implemented here is the
# usual two-level NVFP4 recipe:
#   g        = amax(|x|) / (6 * 448)                   (per tensor, FP32; 1 if amax = 0)
#   s_block  = E4M3_RNE_satfinite((amax_block / 6) / g)  (FP32 divisions)
#   code     = E2M1_RNE_sat(x / (dec(s_block) * g))       (FP32 mul, FP32 div)
#   a zero scale gives all-zero codes; no -0 code is emitted.
# ---------------------------------------------------------------------------

_E4M3_FINITE_POS = np.array([_E4M3[b] for b in range(0x7F)], dtype=np.float64)  # bytes 0..0x7E


def e4m3_encode_rne_satfinite(v) -> np.ndarray:
    """Non-negative float32 values -> E4M3 bytes, round to nearest even, clamp to 448.

    Written as "nearest entry of the table of all 127 non-negative finite E4M3
    values; on a tie take the even encoding", which is round-to-nearest-even on
    the 3-bit mantissa, including across the subnormal range.
    """
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    if np.any(v < 0) or np.any(np.isnan(v)):
        raise ValueError("scale must be non-negative and not NaN")
    T = _E4M3_FINITE_POS
    lo = np.clip(np.searchsorted(T, v, side="right") - 1, 0, T.size - 1)
    hi = np.minimum(lo + 1, T.size - 1)
    d_lo = v - T[lo]
    d_hi = T[hi] - v
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(v >= T[-1], T.size - 1, code)
    return code.astype(np.uint8)


_E2M1_POS = np.array(E2M1_MAGNITUDE, dtype=np.float64)


def e2m1_encode_rne_sat(v) -> np.ndarray:
    """float32 values -> 4-bit E2M1 codes, round to nearest even, clamp to +-6.

    Nearest of the 8 magnitudes; on a tie the even code (even mantissa bit).
    Values whose magnitude rounds to 0 give code 0 (never -0).  +-inf saturates.
    """
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    T = _E2M1_POS
    lo = np.clip(np.searchsorted(T, a, side="right") - 1, 0, T.size - 1)
    hi = np.minimum(lo + 1, T.size - 1)
    d_lo = a - T[lo]
    d_hi = T[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(take_hi, hi, lo)
    mag = np.where(a >= T[-1], T.size - 1, mag).astype(np.uint8)
    sign = ((v < 0) & (mag != 0)).astype(np.uint8) << 3
    return (mag | sign).astype(np.uint8)


def global_scale(x_bf16_bits) -> float:
    """Per-tensor FP32 scale g = amax / (6 * 448) (1.0 for an all-zero tensor)."""
    x = bf16_bits_to_f32(x_bf16_bits)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    if amax == 0:
        return 1.0
    return float(np.float32(amax) / np.float32(6.0 * 448.0))


def quantize(x_bf16_bits, g: float):
    """bf16 [R, K] (uint16 bits) -> (packed codes [R, K/2] uint8, scales [R, K/16] uint8)."""
    return quantize_f32(bf16_bits_to_f32(x_bf16_bits), g)


def quantize_f32(x, g: float):
    """The quantiser's steps on float32 input [R, K] (bf16 input converts exactly)."""
    x = np.asarray(x, dtype=np.float32)
    R, K = x.shape
    assert K % 16 == 0
    g32 = np.float32(g)
    blocks = x.reshape(R, K // 16, 16)
    amax = np.max(np.abs(blocks), axis=2)                            # exact
    s_f = (amax / np.float32(6.0)).astype(np.float32) / g32           # two RN divisions
    sbyte = e4m3_encode_rne_satfinite(s_f.astype(np.float32))
    sdec = _E4M3[sbyte].astype(np.float32)                            # exact
    denom = (sdec * g32).astype(np.float32)                           # RN multiply
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (blocks / denom[:, :, None]).astype(np.float32)           # RN division
    codes = e2m1_encode_rne_sat(v)
    codes = np.where((sbyte == 0)[:, :, None], np.uint8(0), codes)
    return pack_codes(codes.reshape(R, K)), sbyte


# ---------------------------------------------------------------------------
# Two-pass (value + residual) activation quantisation, [P2] follow-ups: the
# activations are quantised in two NVFP4 passes, a value pass and a pass over
# what it left out, and both run on the block-scaled FP4 MMA.  The pages give no
# formula; the plainest reading, used here:
#   q1 = quantize(x, g)
#   r  = x - dequant_f32(q1, g)      (float32: (code * scale) exact, * g RN, x - . RN)
#   q2 = quantize(r, g)              (same global scale, so one alpha = g * g_w)
#   D  = alpha * sum_k (dq1_k + dq2_k) * w_k
# ---------------------------------------------------------------------------


def residual_f32(x_bf16_bits, codes1, sf1, g: float) -> np.ndarray:
    """float32 [R, K]: x - (code * scale) * g, each step an IEEE float32 operation."""
    x = bf16_bits_to_f32(x_bf16_bits)
    R, K = x.shape
    vals = _E2M1[unpack_codes(codes1)].astype(np.float32)
    scl = np.repeat(_E4M3[np.asarray(sf1, dtype=np.uint8)].astype(np.float32), 16, axis=1)
    prod = (vals * scl).astype(np.float32)              # exact: at most 5 significant bits
    dq = (prod * np.float32(g)).astype(np.float32)       # RN multiply
    return (x - dq).astype(np.float32)                   # RN subtraction


def quantize_two_pass(x_bf16_bits, g: float):
    """bf16 [R, K] -> (codes1, sf1, codes2, sf2): the value pass and the residual pass."""
    codes1, sf1 = quantize(x_bf16_bits, g)
    codes2, sf2 = quantize_f32(residual_f32(x_bf16_bits, codes1, sf1, g), g)
    return codes1, sf1, codes2, sf2


def interleave_two_pass(codes1, sf1, codes2, sf2):
    """The library's two-pass operand: per 256-element K-block j, the value codes of
    the block then the residual codes of the same block, so a row holds 2K codes.

    Returns (codes [R, K] uint8, scales [R, 2K/16] uint8), row-major; K % 256 == 0.
    Value byte 128*j + t lands at byte 256*j + t, residual byte 128*j + t at
    256*j + 128 + t; value scale 16*j + u at 32*j + u, residual at 32*j + 16 + u.
    """
    c1, c2 = np.asarray(codes1, np.uint8), np.asarray(codes2, np.uint8)
    s1, s2 = np.asarray(sf1, np.uint8), np.asarray(sf2, np.uint8)
    R, half = c1.shape
    assert (2 * half) % 256 == 0
    nb = 2 * half // 256
    codes = np.stack([c1.reshape(R, nb, 128), c2.reshape(R, nb, 128)], axis=2).reshape(R, 2 * half)
    scales = np.stack([s1.reshape(R, nb, 16), s2.reshape(R, nb, 16)], axis=2).reshape(R, 4 * half // 16)
    return codes, scales


def gemm_two_pass(codes1, sf1, codes2, sf2, B, SFB, alpha: float):
    """(ref, abs_sum) float64 [M, N] of D = alpha * (dq1 + dq2) w^T.

    abs_sum = sum_k (|dq1_k| + |dq2_k|) |w_k|: both passes' products are summed.
    """
    a1 = dequantize(codes1, sf1)
    a2 = dequantize(codes2, sf2)
    b = dequantize(B, SFB)
    ref = ((a1 + a2) @ b.T) * float(alpha)
    abs_sum = (np.abs(a1) + np.abs(a2)) @ np.abs(b).T
    return ref, abs_sum


def gemm_two_pass_at(codes1, sf1, codes2, sf2, B, SFB, alpha: float, rows, cols):
    """gemm_two_pass at the sampled outputs (rows[i], cols[i]); float64 [n] each."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    a1 = dequantize(codes1[rows], sf1[rows])
    a2 = dequantize(codes2[rows], sf2[rows])
    b = dequantize(B[cols], SFB[cols])
    return ((a1 + a2) * b).sum(axis=1) * float(alpha), ((np.abs(a1) + np.abs(a2)) * np.abs(b)).sum(axis=1)


# ---------------------------------------------------------------------------
# Scale-factor layout: 128x4 atoms, [P1] Version 5.
# Within a 512-byte atom the scale of row m (0..127 in the band) and block b
# (0..3 in a 64-element K group) is at byte 16*(m mod 32) + 4*(m div 32 mod 4) + b;
# atoms run K-fastest inside a 128-row band.
# ---------------------------------------------------------------------------


def packed_scales_bytes(rows: int, K: int) -> int:
    """ceil(rows/128)*128 * ceil(K/64)*4."""
    return (-(-rows // 128)) * 128 * (-(-K // 64)) * 4


def pack_scales(sf_rowmajor) -> np.ndarray:
    """Row-major [R, K/16] scale bytes -> flat uint8 buffer in the 128x4 atom layout.

    Padding rows (up to a multiple of 128) and padding blocks (up to a multiple
    of 4) are zero.  The destination of every (r, c) is the closed form above.
    """
    sf = np.asarray(sf_rowmajor, dtype=np.uint8)
    R, C = sf.shape
    groups = -(-C // 4)
    out = np.zeros(packed_scales_bytes(R, 16 * C), dtype=np.uint8)
    r = np.arange(R, dtype=np.int64)[:, None]
    c = np.arange(C, dtype=np.int64)[None, :]
    band, m = r // 128, r % 128
    grp, b = c // 4, c % 4
    off = (band * groups + grp) * 512 + 16 * (m % 32) + 4 * (m // 32) + b
    out[off] = sf
    return out


# ---------------------------------------------------------------------------
# W4A16: y[m,n] = alpha * sum_k x[m,k] * W[n,k] * SW[n,k/16]    ([P2] Summary/Design)
# x is bf16, W is NVFP4; FP32 accumulate, BF16 out.  alpha is the weight's
# global scale.
# ---------------------------------------------------------------------------


def w4a16_linear(x_bf16_bits, W, SW, alpha: float):
    """Returns (ref, abs_sum), float64 [M, N]."""
    x = bf16_bits_to_f64(x_bf16_bits)
    w = dequantize(W, SW)
    ref = (x @ w.T) * float(alpha)
    abs_sum = np.abs(x) @ np.abs(w).T
    return ref, abs_sum


def w4a16_linear_colscale(x_bf16_bits, W, SW, alpha_col):
    """Per-column weight scale ([P2] Design: one weight scale per output column):
    y[m, n] = alpha_col[n] * sum_k x[m, k] * w[n, k].  Returns (ref, scaled_abs_sum),
    float64 [M, N], where scaled_abs_sum[m, n] = |alpha_col[n]| * sum_k |x w|, so
    that ``tolerance(ref, scaled_abs_sum, 1.0)`` is the per-element bound."""
    x = bf16_bits_to_f64(x_bf16_bits)
    w = dequantize(W, SW)
    a = np.asarray(alpha_col, dtype=np.float64).reshape(1, -1)
    ref = (x @ w.T) * a
    abs_sum = (np.abs(x) @ np.abs(w).T) * np.abs(a)
    return ref, abs_sum


def w4a16_linear_at(x_bf16_bits, W, SW, alpha: float, rows, cols):
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    x = bf16_bits_to_f64(np.asarray(x_bf16_bits)[rows])
    w = dequantize(W[cols], SW[cols])
    prod = x * w
    return prod.sum(axis=1) * float(alpha), np.abs(prod).sum(axis=1)


# ---------------------------------------------------------------------------
# W4A16 prepared-weight format ("Wprep").  [P2] Design, weight-layout paragraph: the
# weight is re-laid out once into fragment order, E2M1 codes placed so that
# shifts and masks give bfloat16 values fp4 * 2^-126, scales re-encoded as a
# byte b with bf16(0x7000 | b << 4) == scale * 2^119, zero scales zeroing their
# codes and negative scales flipping the code signs; the result has the size of
# the checkpoint tensors.  The exact bit order below is this library's own and
# is specified here independently of the CUDA code.
#
# Block (nt, kc): rows 16*nt .. 16*nt+15, K range 64*kc .. 64*kc+63, 576 bytes at
# offset (nt * (K/64) + kc) * 576.  For lane l in 0..31, g = l // 4, t = l % 4:
#   bytes [16 l, 16 l + 16): four little-endian 32-bit words w_j (j = 0..3),
#     word j covering k0 = 64 kc + 16 j, holding 8 codes:
#       a0 = (row g,   k0+2t),   a1 = (row g,   k0+2t+1),
#       a2 = (row g+8, k0+2t),   a3 = (row g+8, k0+2t+1),
#       a4 = (row g,   k0+2t+8), a5 = (row g,   k0+2t+9),
#       a6 = (row g+8, k0+2t+8), a7 = (row g+8, k0+2t+9)
#     bit positions of (code bit0, bit1, bit2, sign bit3):
#       a0: 6, 7, 8, 15     a1: 22, 23, 24, 31
#       a2: 28, 29, 30, 5   a3: 12, 13, 14, 21
#       a4: 25, 26, 27, 2   a5: 9, 10, 11, 18
#       a6: 4, 0, 1, 3      a7: 20, 16, 17, 19
#     With M = 0x81C081C0 (bits 6-8 and 15 of each bf16 half: mantissa MSB, the two
#     low exponent bits, sign) the four bf16x2 fragment registers of a word are
#       {a0, a1} = w & M,  {a2, a3} = rotl(w, 10) & M,  {a4, a5} = rotl(w, 13) & M,
#       {a6, a7} = ((w & 0x001B001B) * 0x1084 mod 2^32) & M
#     -- the product is the sum of the masked word shifted by 2, 7 and 12, three
#     copies with no common bit, so no carries and the sum is their union.  Eight
#     integer operations per word (one AND; rotate + AND twice; AND, multiply, AND).
#     No choice of plain shifts or rotations covers all 32 bits with four copies of
#     M (an exhaustive search finds none), which is why the fourth register takes
#     the multiply.
#   bytes [512 + 8 g, 512 + 8 g + 8) (shared by the four lanes with the same g):
#     byte 2j = enc(scale(row g, block 4 kc + j)),
#     byte 2j + 1 = enc(scale(row g + 8, block 4 kc + j)).
# ---------------------------------------------------------------------------

WPREP_BLOCK_BYTES = 576

_CODE_BITS = (
    (6, 7, 8, 15), (22, 23, 24, 31),
    (28, 29, 30, 5), (12, 13, 14, 21),
    (25, 26, 27, 2), (9, 10, 11, 18),
    (4, 0, 1, 3), (20, 16, 17, 19),
)
# (row offset, k offset) of a0..a7 relative to (g, k0 + 2t)
_CODE_POS = ((0, 0), (0, 1), (8, 0), (8, 1), (0, 8), (0, 9), (8, 8), (8, 9))


def w4a16_prepared_bytes(N: int, K: int) -> int:
    return N * K // 2 + N * K // 16


def scale_reencode(mag_byte: int) -> int:
    """Positive finite E4M3 byte (1..0x7E) -> byte b with bf16(0x7000 | b<<4) == scale * 2^119.

    A normal scale (1 + m/8) 2^(e-7) becomes b = ((e + 15) << 3) | m.  A subnormal
    scale m 2^-9 is first renormalised: with p = floor(log2 m) it equals
    (1 + f/8) 2^(p-9) where f = (m << (3-p)) & 7, so b = ((p + 13) << 3) | f.
    Zero maps to 0 (its codes are zeroed).
    """
    if mag_byte == 0:
        return 0
    e = mag_byte >> 3
    m = mag_byte & 7
    if e == 0:
        p = m.bit_length() - 1
        return ((p + 13) << 3) | ((m << (3 - p)) & 7)
    return ((e + 15) << 3) | m


def w4a16_prepare(W, SW) -> np.ndarray:
    """Codes [N, K/2] + row-major scales [N, K/16] -> flat uint8 Wprep (spec above)."""
    codes = unpack_codes(W).astype(np.uint32)
    sw = np.asarray(SW, dtype=np.uint8)
    N, K = codes.shape
    assert N % 16 == 0 and K % 64 == 0
    # Fold the scale's sign and zero into the codes ([P2] Design).
    neg_e = np.repeat((sw & 0x80) != 0, 16, axis=1)
    zero = (sw & 0x7F) == 0
    zero_e = np.repeat(zero, 16, axis=1)
    codes = np.where(neg_e, codes ^ 8, codes)
    codes = np.where(zero_e, 0, codes).astype(np.uint32)
    enc_table = np.array([scale_reencode(b) for b in range(0x80)], dtype=np.uint8)
    enc = np.where(zero, np.uint8(0), enc_table[sw & 0x7F]).astype(np.uint8)

    NT, KC = N // 16, K // 64
    Cb = codes.reshape(NT, 16, KC, 64)          # [nt, row in tile, kc, k in chunk]
    Eb = enc.reshape(NT, 16, KC, 4)             # [nt, row in tile, kc, block in chunk]
    lane = np.arange(32)
    g, t = lane // 4, lane % 4
    words = np.zeros((NT, KC, 32, 4), dtype=np.uint32)
    sbytes = np.zeros((NT, KC, 8, 8), dtype=np.uint8)   # [nt, kc, g, byte]
    g8 = np.arange(8)
    for j in range(4):
        for (dr, dk), bits in zip(_CODE_POS, _CODE_BITS):
            # advanced indices on axes 1 and 3 -> result [lane, nt, kc]
            c = Cb[:, g + dr, :, 16 * j + 2 * t + dk].transpose(1, 2, 0)
            for i, pos in enumerate(bits):
                words[:, :, :, j] |= ((c >> i) & 1) << np.uint32(pos)
        sbytes[:, :, :, 2 * j] = Eb[:, g8, :, j].transpose(1, 2, 0)
        sbytes[:, :, :, 2 * j + 1] = Eb[:, g8 + 8, :, j].transpose(1, 2, 0)
    out = np.empty((NT, KC, WPREP_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, :512] = words.astype("<u4").view(np.uint8).reshape(NT, KC, 512)
    out[:, :, 512:] = sbytes.reshape(NT, KC, 64)
    return out.reshape(-1)

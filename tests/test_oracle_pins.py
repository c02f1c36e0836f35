"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what it pins and where the fact comes from.  None of these
needs a GPU.
"""

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nvfp4_oracle as O
from synthetic import generators as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- decode tables

def _e2m1_from_bits(c):
    """E2M1 from its bit fields: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return -mag if s else mag


def test_e2m1_table_matches_bit_field_formula():
    t = O.e2m1_table()
    for c in range(16):
        assert Fraction(t[c]) == _e2m1_from_bits(c)
        assert np.signbit(t[c]) == bool(c & 8)


def test_e4m3_table_matches_torch_float8_decoder():
    # Library decoder (torch.float8_e4m3fn) over all 256 encodings, NaNs included.
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    t = O.e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(t))
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(t[~nan], ref[~nan])
    assert np.array_equal(np.signbit(t[~nan]), np.signbit(ref[~nan]))


def test_unpack_low_nibble_is_even_k():
    packed = np.array([[0x21, 0xF8]], dtype=np.uint8)
    assert O.unpack_codes(packed).tolist() == [[1, 2, 8, 15]]
    assert np.array_equal(O.pack_codes(O.unpack_codes(packed)), packed)


# ---------------------------------------------------------------- GEMM definition

def _frac_dequant(packed, sf):
    codes = O.unpack_codes(packed)
    R, K = codes.shape
    e4 = [Fraction(x) if not np.isnan(x) else None for x in
          torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()]
    return [[_e2m1_from_bits(int(codes[r, k])) * e4[int(sf[r, k // 16])] for k in range(K)]
            for r in range(R)]


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 16, 0), (3, 5, 64, 1), (8, 8, 128, 2), (7, 2, 64, 3)])
def test_gemm_equals_exact_rational_brute_force(M, N, K, seed):
    A = G.packed_codes_uniform(M, K, seed, "A")
    B = G.packed_codes_uniform(N, K, seed, "B")
    SFA = G.scales_with_zero_and_subnormal(M, K, seed, "SFA", 0.1, 0.2)
    SFB = G.scales_with_zero_and_subnormal(N, K, seed, "SFB", 0.1, 0.2)
    alpha = G.alpha_uniform(seed)
    ref, abs_sum = O.gemm(A, SFA, B, SFB, alpha)
    a = _frac_dequant(A, SFA)
    b = _frac_dequant(B, SFB)
    for m in range(M):
        for n in range(N):
            s = sum(a[m][k] * b[n][k] for k in range(K))
            sa = sum(abs(a[m][k] * b[n][k]) for k in range(K))
            assert Fraction(ref[m, n]) == s * Fraction(alpha)
            assert Fraction(abs_sum[m, n]) == sa


def test_single_block_dot_is_exact_in_float32():
    # One 16-element block: the code sum is a multiple of 1/4 with |.| <= 576 and
    # sfa*sfb has <= 8 significant bits, so the product is exact in FP32.
    g = np.random.default_rng(5)
    for _ in range(200):
        A = g.integers(0, 256, size=(1, 8), dtype=np.uint8)
        B = g.integers(0, 256, size=(1, 8), dtype=np.uint8)
        sa = g.integers(0, 0x7F, size=(1, 1), dtype=np.uint8)
        sb = g.integers(0, 0x7F, size=(1, 1), dtype=np.uint8)
        ref, _ = O.gemm(A, sa, B, sb, 1.0)
        assert float(np.float32(ref[0, 0])) == ref[0, 0]


def test_all_scales_one_is_integer_gemm_on_twice_the_codes():
    # With every scale = 1.0 (E4M3 0x38) the GEMM is an integer GEMM on 2*codes, /4.
    M, N, K = 16, 24, 512
    A = G.packed_codes_uniform(M, K, 7, "A")
    B = G.packed_codes_uniform(N, K, 7, "B")
    ones_a = np.full((M, K // 16), 0x38, dtype=np.uint8)
    ones_b = np.full((N, K // 16), 0x38, dtype=np.uint8)
    ref, _ = O.gemm(A, ones_a, B, ones_b, 1.0)
    two = np.array([int(2 * _e2m1_from_bits(c)) for c in range(16)], dtype=np.int64)
    ia = two[O.unpack_codes(A)]
    ib = two[O.unpack_codes(B)]
    exact = ia @ ib.T
    assert np.array_equal(ref * 4, exact.astype(np.float64))


def test_float64_gemm_equals_int64_gemm_on_square_workload_distribution():
    # Square workloads: scales in [2^-4, 2^4] -> |product| <= 2^33.2 units of 2^-20,
    # so float64 accumulation is exact over K <= 2^15.
    M, N, K = 64, 48, 2048
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=3, scales="zero_sub")
    ref, _ = O.gemm(A, SFA, B, SFB, 1.0)
    units = O.gemm_exact_units(A, SFA, B, SFB)
    assert np.array_equal(ref, units.astype(np.float64) * 2.0 ** -20)


def test_sampled_and_tile_references_agree_with_full():
    M, N, K = 40, 56, 256
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=4)
    ref, abs_sum = O.gemm(A, SFA, B, SFB, 1.75)
    rows = np.array([0, 5, 39, 17])
    cols = np.array([55, 0, 3, 31])
    r2, a2 = O.gemm_at(A, SFA, B, SFB, 1.75, rows, cols)
    assert np.array_equal(r2, ref[rows, cols])
    assert np.array_equal(a2, abs_sum[rows, cols])
    rt, at = O.gemm_tile(A, SFA, B, SFB, 1.75, 8, 24, 16, 40)
    assert np.array_equal(rt, ref[8:24, 16:40])


def test_tolerance_formula_scales_with_alpha():
    ref = np.array([256.0, -256.0, 0.0])
    abs_sum = np.array([1e6, 1e6, 1e6])
    tol = O.tolerance(ref, abs_sum, -2.0)
    assert np.allclose(tol, [1.0 + 2.0, 1.0 + 2.0, 2.0])


# ---------------------------------------------------------------- bf16 helpers

def test_bf16_rne_matches_torch():
    g = np.random.default_rng(11)
    x = g.standard_normal(1_000_000).astype(np.float32) * np.float32(1e3)
    # all tie patterns on a handful of exponents
    base = np.arange(0, 1 << 16, 97, dtype=np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f32_to_bf16_rne(x)
    nan = np.isnan(x)        # NaN payloads are a convention; both must stay NaN
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(O.bf16_bits_to_f64(got[nan])))
    assert np.array_equal(O.bf16_bits_to_f64(ref), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy(), equal_nan=True)


# ---------------------------------------------------------------- scale layout

def test_pack_scales_golden_offsets():
    for rows, K, r, c, off in _golden_rows("pack_scales_offsets.txt"):
        rows, K, r, c, off = int(rows), int(K), int(r), int(c), int(off)
        sf = np.zeros((rows, K // 16), dtype=np.uint8)
        sf[r, c] = 0xA5
        packed = O.pack_scales(sf)
        assert packed.size == O.packed_scales_bytes(rows, K)
        assert np.flatnonzero(packed).tolist() == [off], (rows, K, r, c)


@pytest.mark.parametrize("R,K", [(1, 64), (128, 64), (129, 320), (300, 1024), (256, 48)])
def test_pack_scales_is_bijection_with_zero_padding(R, K):
    C = K // 16
    ids = np.arange(R * C, dtype=np.int64)
    # Values 1..255 repeat, so check the permutation through two byte planes.
    lo = ((ids % 255) + 1).astype(np.uint8).reshape(R, C)
    hi = (((ids // 255) % 255) + 1).astype(np.uint8).reshape(R, C)
    plo, phi = O.pack_scales(lo), O.pack_scales(hi)
    assert plo.size == (-(-R // 128)) * 128 * (-(-K // 64)) * 4
    nz = np.flatnonzero(plo)
    assert nz.size == R * C and np.array_equal(np.flatnonzero(phi), nz)
    got = (phi[nz].astype(np.int64) - 1) * 255 + (plo[nz].astype(np.int64) - 1)
    assert np.array_equal(np.sort(got), ids)


def test_footprints_match_the_page():
    for S, mib in _golden_rows("footprints.txt"):
        S = int(S)
        codes = 2 * (S * S // 2)
        scales = 2 * (S * (S // 16))
        assert O.packed_scales_bytes(S, S) == S * (S // 16)
        assert (codes + scales) / 2 ** 20 == float(mib)


# ---------------------------------------------------------------- quantisation

def test_e2m1_rounding_golden():
    for v, code in _golden_rows("e2m1_rounding.txt"):
        got = int(O.e2m1_encode_rne_sat(np.array([float(v)], dtype=np.float32))[0])
        assert got == int(code, 16), v


def test_e2m1_encode_is_nearest_value_brute_force():
    g = np.random.default_rng(2)
    v = (g.standard_normal(20000) * 3).astype(np.float32)
    codes = O.e2m1_encode_rne_sat(v)
    vals = np.array([float(_e2m1_from_bits(c)) for c in range(16)])
    for x, c in zip(v.astype(np.float64), codes):
        err = abs(vals[c] - min(max(x, -6.0), 6.0))
        assert err <= np.min(np.abs(vals - min(max(x, -6.0), 6.0))) + 0.0


def test_e4m3_encode_matches_torch_rne_below_saturation():
    g = np.random.default_rng(3)
    v = np.concatenate([
        np.exp(g.uniform(np.log(1e-5), np.log(460.0), 200000)),
        O.e4m3_table()[:0x7F],                                     # exact values
        (O.e4m3_table()[:0x7E] + O.e4m3_table()[1:0x7F]) / 2,      # exact ties
    ]).astype(np.float32)
    v = v[v < 464.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode_rne_satfinite(v), ref)
    assert O.e4m3_encode_rne_satfinite(np.array([464.0, 1e30], dtype=np.float32)).tolist() == [0x7E, 0x7E]


def test_quantize_invariants():
    R, K = 64, 512
    x = G.bf16_normal(R, K, 0, "x")
    # a zero block and an all-negative tiny block
    x[0, :16] = 0
    x[1, 16:32] = 0x8001  # -tiny subnormal bf16
    g = O.global_scale(x)
    codes, sf = O.quantize(x, g)
    assert codes.shape == (R, K // 2) and sf.shape == (R, K // 16)
    dq = O.dequantize(codes, sf) * g
    xf = O.bf16_bits_to_f64(x)
    # every decoded value is bounded by 6 * scale * g
    sc = np.repeat(O.e4m3_table()[sf], 16, axis=1) * g
    assert np.all(np.abs(dq) <= 6 * sc + 0.0)
    assert np.all(O.unpack_codes(codes)[0, :16] == 0) and sf[0, 0] == 0
    assert np.all(O.unpack_codes(codes)[1, 16:32] == 0)
    assert not np.any(O.unpack_codes(codes) == 8)              # no -0 codes
    # the block's absmax element maps to code +-6 unless the scale was rounded
    # up (then it may map to the next lower magnitude 4)
    blocks = np.abs(xf).reshape(R, K // 16, 16)
    arg = blocks.argmax(axis=2)
    cmag = (O.unpack_codes(codes).reshape(R, K // 16, 16) & 7)
    top = np.take_along_axis(cmag, arg[:, :, None], 2)[:, :, 0]
    nz = sf != 0
    assert np.all((top[nz] == 7) | (top[nz] == 6))
    assert np.mean(top[nz] == 7) > 0.4
    # relative reconstruction error of an NVFP4 tensor from N(0,1) is ~10 %
    rel = np.linalg.norm(dq - xf) / np.linalg.norm(xf)
    assert 0.03 < rel < 0.2


def test_global_scale_reading():
    x = G.bf16_normal(4, 64, 0, "x")
    amax = np.max(np.abs(O.bf16_bits_to_f32(x)))
    assert O.global_scale(x) == float(np.float32(amax) / np.float32(2688.0))
    assert O.global_scale(np.zeros((2, 32), dtype=np.uint16)) == 1.0


def test_global_scale_golden_values():
    # Reading Q1: g = amax / (6 * 448), the largest E2M1 value times the largest
    # E4M3 scale, rounded once to float32; amax is taken over magnitudes.  Hand-worked
    # cases: 2688 = 6 * 448 gives exactly 1; a negative element of magnitude 5376 gives
    # exactly 2; amax = 1 and 0.75 give 1/2688 and 3/10752 rounded to nearest float32
    # (computed here from the exact rationals, not by a float division).
    cases = [
        ([2688.0, -1.0, 0.5], Fraction(1)),
        ([1.0, -5376.0, 3.0], Fraction(2)),
        ([1.0, -0.5, 0.25], _rn_f32(Fraction(1, 2688))),
        ([-0.75, 0.5], _rn_f32(Fraction(3, 4) / 2688)),
        ([float(255 * 2 ** 120), 1.0], _rn_f32(Fraction(255 * 2 ** 120, 2688))),  # the largest finite bf16
    ]
    for vals, want in cases:
        bits = _bf16_bits_of(vals)
        g = O.global_scale(bits.reshape(1, -1))
        assert Fraction(g) == want, (vals, g, float(want))
    assert _rn_f32(Fraction(1, 2688)) != Fraction(1, 2688)  # the rounding is not trivial


def test_float64_gemm_is_exact_where_its_bound_holds_on_llm_scales():
    # The LLM-shaped operands (quantised N(0,1) activations, N(0, 0.02) weights) carry
    # block scales up to 448, so a product can reach 2^57 units of 2^-20 and float64
    # accumulation is not exact in general.  Where an output's sum of |a_k b_k| stays
    # below 2^53 units, every partial sum is an integer number of units below 2^53 and
    # float64 must equal the exact int64 sum; the outputs outside the bound are
    # counted and must be within the float64 rounding bound K * 2^-53 * sum|a b|.
    for M, N, K in ((24, 40, 1024), (4, 8, 17408)):
        x = G.bf16_normal(M, K, 7, "x")
        w = G.bf16_normal(N, K, 7, "w", 0.02)
        A, SFA = O.quantize(x, O.global_scale(x))
        B, SFB = O.quantize(w, O.global_scale(w))
        ref, abs_sum = O.gemm(A, SFA, B, SFB, 1.0)
        units = O.gemm_exact_units(A, SFA, B, SFB)
        exact = units.astype(np.float64) * 2.0 ** -20
        in_bound = abs_sum * 2.0 ** 20 < 2.0 ** 53 * (1 - 2.0 ** -40)
        assert np.array_equal(ref[in_bound], exact[in_bound])
        out = ~in_bound
        assert np.all(np.abs(ref[out] - exact[out]) <= K * 2.0 ** -53 * abs_sum[out])
        print(f"K={K}: float64 exactness bound holds for {int(in_bound.sum())}/{in_bound.size} outputs")


# ---------------------------------------------------------------- W4A16

def test_w4a16_prepared_size_golden():
    for N, K, nbytes in _golden_rows("w4a16_prepared_size.txt"):
        assert O.w4a16_prepared_bytes(int(N), int(K)) == int(nbytes)
    W = G.packed_codes_uniform(128, 256, 0, "W")
    SW = G.scales_uniform_normal(128, 256, 0, "SW")
    assert O.w4a16_prepare(W, SW).size == 18432


def test_scale_reencode_identity_every_finite_e4m3():
    # bf16(0x7000 | b << 4) == scale * 2^119 for every positive finite E4M3 scale,
    # subnormals included (TileLang PR #3290, Design, "Weight layout").
    t = O.e4m3_table()
    for byte in range(1, 0x7F):
        b = O.scale_reencode(byte)
        assert 0 <= b < 256
        bits = np.array([0x7000 | (b << 4)], dtype=np.uint16)
        assert O.bf16_bits_to_f64(bits)[0] == t[byte] * 2.0 ** 119, hex(byte)


def _emulate_register_dequant(wprep, N, K):
    """Decode a Wprep buffer the way the W4A16 kernel's registers do (bf16 bit
    manipulation, then one bfloat16 multiply rounded to nearest even), and return
    float64 [N, K] weights times 2^-7 undone."""
    blocks = np.asarray(wprep, dtype=np.uint8).reshape(N // 16, K // 64, 576)
    out = np.zeros((N, K), dtype=np.float64)
    mask = 0x81C081C0
    for nt in range(N // 16):
        for kc in range(K // 64):
            blk = blocks[nt, kc]
            for lane in range(32):
                g, t = divmod(lane, 4)
                words = blk[16 * lane:16 * lane + 16].view("<u4")
                sb = blk[512 + 8 * g:512 + 8 * g + 8]
                for j in range(4):
                    w = int(words[j])
                    rotl = lambda v, n: ((v << n) | (v >> (32 - n))) & 0xFFFFFFFF
                    r0 = w & mask
                    r1 = rotl(w, 10) & mask
                    r2 = rotl(w, 13) & mask
                    r3 = (((w & 0x001B001B) * 0x1084) & 0xFFFFFFFF) & mask
                    regs = (r0, r1, r2, r3)
                    srow = (int(sb[2 * j]), int(sb[2 * j + 1]))          # rows g, g+8
                    # reg -> (row offset, k offset of the low half)
                    where = ((0, 0), (8, 0), (0, 8), (8, 8))
                    for reg, (dr, dk) in zip(regs, where):
                        s_bits = 0x7000 | (srow[dr // 8] << 4)
                        for half in range(2):
                            wb = (reg >> (16 * half)) & 0xFFFF
                            prod = O.bf16_bits_to_f32(np.array([wb], np.uint16))[0] * \
                                O.bf16_bits_to_f32(np.array([s_bits], np.uint16))[0]
                            # bf16 multiply: exact here, so rounding the f32 product is the bf16 result
                            pb = O.f32_to_bf16_rne(np.array([prod], np.float32))
                            out[16 * nt + g + dr, 64 * kc + 16 * j + 2 * t + dk + half] = \
                                O.bf16_bits_to_f64(pb)[0] * 2.0 ** 7
    return out


def test_wprep_register_dequant_every_scale_and_code():
    # Every finite E4M3 scale byte, both signs and zero, with every code.
    # (TileLang PR #3290, Tests: bit-exact emulation of the register dequant.)
    scales = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], dtype=np.uint8)
    n_rows = 16 * (-(-scales.size // 16))
    K = 64
    SW = np.zeros((n_rows, K // 16), dtype=np.uint8)
    SW[:scales.size, :] = scales[:, None]
    SW[:scales.size, 1] = scales[::-1][:, None][:, 0]
    codes = np.tile(np.arange(16, dtype=np.uint8), (n_rows, K // 16))
    codes = np.roll(codes, 3, axis=1)
    W = O.pack_codes(codes)
    wprep = O.w4a16_prepare(W, SW)
    got = _emulate_register_dequant(wprep, n_rows, K)
    want = O.dequantize(W, SW)
    assert np.array_equal(np.abs(got), np.abs(want))
    nzw = want != 0
    assert np.array_equal(np.sign(got[nzw]), np.sign(want[nzw]))


def test_w4a16_linear_equals_exact_rational_brute_force():
    M, N, K = 3, 16, 64
    x = G.bf16_normal(M, K, 1, "x")
    W = G.packed_codes_uniform(N, K, 1, "W")
    SW = G.scales_with_zero_and_subnormal(N, K, 1, "SW", 0.1, 0.2)
    ref, abs_sum = O.w4a16_linear(x, W, SW, 0.5)
    xf = [[Fraction(float(v)) for v in row] for row in O.bf16_bits_to_f64(x)]
    w = _frac_dequant(W, SW)
    for m in range(M):
        for n in range(N):
            s = sum(xf[m][k] * w[n][k] for k in range(K))
            # float64 rounding of the sum: relative error far below the tolerance
            assert abs(Fraction(ref[m, n]) - s * Fraction(1, 2)) <= Fraction(1, 2 ** 40) * (1 + abs(s))
            assert abs(Fraction(abs_sum[m, n]) - sum(abs(xf[m][k] * w[n][k]) for k in range(K))) \
                <= Fraction(1, 2 ** 40) * (1 + abs(s))


def test_w4a16_sampled_agrees_with_full():
    x = G.bf16_normal(5, 128, 2, "x")
    W = G.packed_codes_uniform(32, 128, 2, "W")
    SW = G.scales_uniform_normal(32, 128, 2, "SW")
    ref, abs_sum = O.w4a16_linear(x, W, SW, 2.0)
    r, a = O.w4a16_linear_at(x, W, SW, 2.0, [0, 4, 2], [31, 0, 7])
    assert np.allclose(r, ref[[0, 4, 2], [31, 0, 7]], rtol=1e-15, atol=0)


def test_w4a16_colscale_equals_exact_rational_brute_force():
    # Per-column weight scale: y[m, n] = alpha_n * sum_k x w, checked against exact
    # rationals with distinct alphas per column (negative, zero, non-power-of-two).
    M, N, K = 3, 16, 64
    x = G.bf16_normal(M, K, 7, "x")
    W = G.packed_codes_uniform(N, K, 7, "W")
    SW = G.scales_with_zero_and_subnormal(N, K, 7, "SW", 0.1, 0.2)
    alpha = np.array([0.375 * (n - 5) + (0.1 if n % 3 == 0 else 0.0) for n in range(N)], np.float32)
    alpha[4] = 0.0
    ref, sabs = O.w4a16_linear_colscale(x, W, SW, alpha)
    xf = [[Fraction(float(v)) for v in row] for row in O.bf16_bits_to_f64(x)]
    w = _frac_dequant(W, SW)
    for m in range(M):
        for n in range(N):
            a = Fraction(float(alpha[n]))
            s = sum(xf[m][k] * w[n][k] for k in range(K))
            sa = sum(abs(xf[m][k] * w[n][k]) for k in range(K))
            assert abs(Fraction(ref[m, n]) - a * s) <= Fraction(1, 2 ** 40) * (1 + abs(a * s))
            assert abs(Fraction(sabs[m, n]) - abs(a) * sa) <= Fraction(1, 2 ** 40) * (1 + abs(a) * sa)
    # A constant column scale is the global-scale case, whose own pin is above.
    r1, a1 = O.w4a16_linear_colscale(x, W, SW, np.full(N, 0.5, np.float32))
    r2, a2 = O.w4a16_linear(x, W, SW, 0.5)
    assert np.array_equal(r1, r2) and np.array_equal(a1 * 1.0, a2 * 0.5)


# ---------------------------------------------------------------- two-pass (value + residual)

def _bf16_bits_of(values):
    """Exactly representable values -> bfloat16 bit patterns (float32 bits >> 16)."""
    f = np.asarray(values, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value not exact in bfloat16"
    return (bits >> 16).astype(np.uint16)


def test_two_pass_hand_worked_block():
    # tests/golden/two_pass_block.txt: value grid at scale 1, residual grid at 2^-4.
    rows = _golden_rows("two_pass_block.txt")
    x = _bf16_bits_of([[float(r[1]) for r in rows]])
    code1 = [int(r[2], 16) for r in rows]
    code2 = [int(r[3], 16) for r in rows]
    c1, s1, c2, s2 = O.quantize_two_pass(x, 1.0)
    assert s1.tolist() == [[0x38]] and s2.tolist() == [[0x18]]
    assert O.unpack_codes(c1).tolist() == [code1]
    assert O.unpack_codes(c2).tolist() == [code2]
    # the two passes rebuild x exactly
    rebuilt = O.dequantize(c1, s1) + O.dequantize(c2, s2)
    assert np.array_equal(rebuilt, O.bf16_bits_to_f64(x))


def test_two_pass_of_a_representable_input_has_an_empty_residual():
    # x = code * scale with the code 6 (byte 7) in every block: the value pass
    # reproduces codes and scales, the residual is zero, the residual pass all zeros.
    rng = np.random.default_rng(11)
    R, K = 8, 64
    codes = rng.integers(0, 16, size=(R, K))
    codes[codes == 8] = 0                   # no negative zero in the input
    codes[:, ::16] = 7                      # a +6 in every block sets its amax
    sf = rng.integers(0x18, 0x59, size=(R, K // 16)).astype(np.uint8)
    x = O.dequantize(O.pack_codes(codes.astype(np.uint8)), sf)
    c1, s1, c2, s2 = O.quantize_two_pass(_bf16_bits_of(x), 1.0)
    assert np.array_equal(O.unpack_codes(c1), codes) and np.array_equal(s1, sf)
    assert not c2.any() and not s2.any()


def test_two_pass_error_is_within_the_residual_grid_and_far_below_one_pass():
    # Per element |x - g (dq1 + dq2)| <= dec(s2) g + 6 g 2^-10 + 2^-20 |x|: half of the
    # widest E2M1 gap (1 scale unit) covers every unsaturated element; a saturated one
    # misses by at most 6 g times the scale's rounding (0.375 units for normal scales,
    # 2^-10 absolute for subnormal ones); the float32 steps add a relative 2^-20.
    x = G.bf16_normal(64, 1024, 5, "x")
    g = O.global_scale(x)
    c1, s1, c2, s2 = O.quantize_two_pass(x, g)
    xf = O.bf16_bits_to_f64(x)
    err2 = np.abs(xf - (O.dequantize(c1, s1) + O.dequantize(c2, s2)) * g)
    dec2 = np.repeat(O.e4m3_table()[s2], 16, axis=1)
    assert np.all(err2 <= dec2 * g + 6 * g * 2.0 ** -10 + 2.0 ** -20 * np.abs(xf))
    err1 = np.abs(xf - O.dequantize(c1, s1) * g)
    assert np.sqrt((err2 ** 2).mean()) < np.sqrt((err1 ** 2).mean()) / 4


def test_interleave_two_pass_places_blocks_by_hand_offsets():
    R, K = 2, 512
    c1 = (np.arange(R * K // 2).reshape(R, K // 2) % 251).astype(np.uint8)
    c2 = (250 - c1).astype(np.uint8)
    s1 = (np.arange(R * K // 16).reshape(R, K // 16) % 97).astype(np.uint8)
    s2 = (s1 + 100).astype(np.uint8)
    A, S = O.interleave_two_pass(c1, s1, c2, s2)
    assert A.shape == (2, 512) and S.shape == (2, 64)
    assert A[0, 0] == c1[0, 0] and A[0, 127] == c1[0, 127]
    assert A[0, 128] == c2[0, 0] and A[0, 133] == c2[0, 5]
    assert A[0, 258] == c1[0, 130] and A[1, 511] == c2[1, 255]
    assert S[0, 15] == s1[0, 15] and S[0, 16] == s2[0, 0]
    assert S[0, 33] == s1[0, 17] and S[1, 63] == s2[1, 31]


def test_gemm_two_pass_equals_exact_rational_brute_force():
    M, N, K = 2, 3, 256
    x = G.bf16_normal(M, K, 3, "x")
    c1, s1, c2, s2 = O.quantize_two_pass(x, O.global_scale(x))
    B = G.packed_codes_uniform(N, K, 3, "B")
    SFB = G.scales_uniform_normal(N, K, 3, "SFB")
    ref, abs_sum = O.gemm_two_pass(c1, s1, c2, s2, B, SFB, 0.75)
    a1, a2, w = _frac_dequant(c1, s1), _frac_dequant(c2, s2), _frac_dequant(B, SFB)
    for m in range(M):
        for n in range(N):
            s = sum((a1[m][k] + a2[m][k]) * w[n][k] for k in range(K)) * Fraction(3, 4)
            sa = sum((abs(a1[m][k]) + abs(a2[m][k])) * abs(w[n][k]) for k in range(K))
            assert Fraction(ref[m, n]) == s          # every term is a multiple of 2^-20
            assert Fraction(abs_sum[m, n]) == sa


def test_gemm_two_pass_is_a_plain_gemm_over_the_interleaved_operand():
    # The layout the library's kernels run: 2K interleaved activation codes against
    # the weight with each of its 256-element K-blocks used twice.
    M, N, K = 5, 7, 512
    x = G.bf16_normal(M, K, 4, "x")
    c1, s1, c2, s2 = O.quantize_two_pass(x, O.global_scale(x))
    B = G.packed_codes_uniform(N, K, 4, "B")
    SFB = G.scales_uniform_normal(N, K, 4, "SFB")
    A2, S2 = O.interleave_two_pass(c1, s1, c2, s2)
    Bd, Sd = O.interleave_two_pass(B, SFB, B, SFB)
    r1, a1 = O.gemm_two_pass(c1, s1, c2, s2, B, SFB, 1.25)
    r2, a2 = O.gemm(A2, S2, Bd, Sd, 1.25)
    assert np.array_equal(r1, r2) and np.array_equal(a1, a2)
    r3, _ = O.gemm_two_pass_at(c1, s1, c2, s2, B, SFB, 1.25, [4, 0], [6, 2])
    assert np.array_equal(r3, r1[[4, 0], [6, 2]])


# ---------------------------------------------------------------- quantiser, step by step in exact arithmetic

def _rn_f32(q):
    """Round a Fraction to the nearest float32 value (ties to even), as a Fraction:
    spacing 2^(e-23) in the binade [2^e, 2^(e+1)), 2^-149 below 2^-126."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    spacing = Fraction(2) ** (max(e, -126) - 23)
    n = a / spacing
    k = n.numerator // n.denominator
    rem = n - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    return sign * k * spacing


def _nearest_even(v, values):
    """Index of the nearest of the non-negative `values` to |v| (ties to the even index),
    saturating at the largest."""
    a = abs(v)
    if a >= values[-1]:
        return len(values) - 1
    best = min(range(len(values)), key=lambda i: (abs(values[i] - a), i % 2))
    return best


def _e4m3_values():
    return [Fraction(float(v)) for v in torch.arange(0x7F, dtype=torch.int32).to(torch.uint8)
            .view(torch.float8_e4m3fn).double().numpy()]            # bytes 0x00..0x7E, ascending


def _assert_quantize_matches_exact_steps(x, g, f32=False):
    # Q2/Q3 applied with exact rationals and an explicit float32 rounding after each
    # IEEE operation, the scale and the codes chosen by brute force over the formats'
    # values: an implementation of the same reading that shares nothing with the
    # oracle's numpy float32 arithmetic.
    e4 = _e4m3_values()
    e2 = [Fraction(m) for m in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    codes, sf = O.quantize_f32(x, g) if f32 else O.quantize(x, g)
    cu = O.unpack_codes(codes)
    gf = Fraction(float(np.float32(g)))
    for b in range(x.shape[0]):
        xs = [Fraction(float(v)) for v in (x[b].astype(np.float64) if f32 else O.bf16_bits_to_f64(x[b]))]
        amax = max(abs(v) for v in xs)
        s = _rn_f32(_rn_f32(amax / 6) / gf)
        sbyte = _nearest_even(s, e4)
        assert sf[b, 0] == sbyte, (b, g)
        for k in range(16):
            if sbyte == 0:
                want = 0
            else:
                denom = _rn_f32(e4[sbyte] * gf)
                v = _rn_f32(xs[k] / denom)
                mag = _nearest_even(v, e2)
                want = 0 if mag == 0 else mag | (8 if v < 0 else 0)
            assert cu[b, k] == want, (b, k, g)


def test_quantize_equals_exact_rational_steps():
    rng = np.random.default_rng(12)
    blocks = [G.bf16_normal(1, 16, s, "x")[0] for s in range(40)]
    blocks += [O.f32_to_bf16_rne((rng.standard_normal(16) * 10.0 ** rng.uniform(-8, 4)).astype(np.float32))
               for _ in range(40)]
    # grid points and midpoints of E2M1 at scale 1 (ties at g = 1)
    blocks.append(O.f32_to_bf16_rne(np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25,
                                              -1.75, -2.5, -3.5, -5, 0], np.float32)))
    x = np.stack(blocks)
    for g in (1.0, O.global_scale(x), 0.0123456789, 3.7e-3):
        _assert_quantize_matches_exact_steps(x, g)


def test_quantize_scale_order_at_e4m3_midpoints():
    # Global scales g for which (amax / 6) / g, each division rounded, is exactly a
    # midpoint between two E4M3 values while amax / (6 g) falls on the other side of
    # it: the scale byte then depends on the order of the two divisions, so these
    # blocks separate the stated order from a one-division shortcut.  (amax = 6.375,
    # amax / 6 = 1.0625 exactly; the scales are searched over float32 neighbours.)
    e4 = np.array([float(v) for v in _e4m3_values()])
    found = []
    for b in range(0x30, 0x58):
        mid = (e4[b] + e4[b + 1]) / 2
        g0 = np.float32(1.0625 / mid)
        g = (g0 + np.arange(-3000, 3000, dtype=np.float32) * np.spacing(g0)).astype(np.float32)
        s = (np.float32(1.0625) / g).astype(np.float32)
        sw = (np.float32(6.375) / (np.float32(6.0) * g).astype(np.float32)).astype(np.float32)
        ok = (s.astype(np.float64) == mid) & (np.sign(sw.astype(np.float64) - mid) != 0)
        if ok.any():
            found.append(float(g[np.flatnonzero(ok)[0]]))
    assert len(found) >= 4
    rng = np.random.default_rng(13)
    for g in found:
        vals = np.concatenate([[6.375], rng.uniform(-6, 6, 15)]).astype(np.float32)
        _assert_quantize_matches_exact_steps(O.f32_to_bf16_rne(vals)[None, :], g)


def test_quantize_f32_rounds_the_quotient_in_float32():
    # Float32 inputs (the residual of the two-pass quantiser) can put x / denom within
    # half an ulp of an E2M1 midpoint without reaching it, so the float32 rounding of
    # the denominator and of the quotient decide codes.  The blocks hold, besides their
    # amax (6 times the denominator), the seventeen float32 neighbours of
    # midpoint x denominator for every E2M1 midpoint, under several global scales.
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    e4 = np.array([float(v) for v in _e4m3_values()])
    n_ties = 0
    for g in (0.7, 0.0123456789, 1.1, 3.3e-3, 0.3):
        g32 = np.float32(g)
        s = np.float32(np.float32(np.float32(6.0) / np.float32(6.0)) / g32)
        sbyte = int(O.e4m3_encode_rne_satfinite(np.array([s], np.float32))[0])
        d = np.float32(np.float32(e4[sbyte]) * g32)
        xs = []
        for m in mids:
            base = np.float32(m * float(d))
            for k in range(-8, 9):
                x = np.float32(base + np.float32(k) * np.spacing(base))
                q = Fraction(float(x)) / Fraction(float(d))
                n_ties += int(q != m and _rn_f32(q) == m)
                xs.append(x)
        xs = np.array(xs, np.float32)
        blocks = []
        for c in range(0, len(xs), 15):
            chunk = xs[c:c + 15]
            blk = np.zeros(16, np.float32)
            blk[0] = np.float32(6.0 * float(d))
            blk[1:1 + len(chunk)] = chunk
            blocks.append(blk)
        _assert_quantize_matches_exact_steps(np.stack(blocks), g, f32=True)
    assert n_ties >= 10  # quotients that round onto a midpoint without equalling it


def test_residual_equals_exact_rational_steps():
    # r = RN(x - RN(value * scale * g)), value * scale exact: checked element by element
    # with exact rationals and the hand-written float32 rounding, on N(0,1) data whose
    # global scale is not a power of two (so RN(value * scale * g) does round).
    x = G.bf16_normal(4, 256, 31, "x")
    g = O.global_scale(x)
    codes, sf = O.quantize(x, g)
    r = O.residual_f32(x, codes, sf, g)
    gf = Fraction(float(np.float32(g)))
    e4 = _e4m3_values()
    cu = O.unpack_codes(codes)
    xf = O.bf16_bits_to_f64(x)
    for i in range(x.shape[0]):
        for k in range(x.shape[1]):
            val = _e2m1_from_bits(int(cu[i, k]))
            want = _rn_f32(Fraction(float(xf[i, k])) - _rn_f32(val * e4[int(sf[i, k // 16])] * gf))
            assert Fraction(float(r[i, k])) == want, (i, k)

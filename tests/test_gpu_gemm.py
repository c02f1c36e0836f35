"""GPU parity of the NVFP4 block-scaled GEMM against the oracle.

Tolerance per BF16 output element: |D - ref| <= 2^-8 |ref| + 1e-6 |alpha| sum_k |a_k b_k|,
ref the exact (float64) alpha * sum_k a_k b_k.  Full comparison where M*N*K <= 2^34,
otherwise seeded random samples plus the four corner 128 x 128 tiles.
"""

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_gb300 as nv
from oracle import nvfp4_oracle as O
from synthetic import generators as G
from gpu_util import assert_within, corner_tiles, dev, dev_bf16, host_bits, host_f64, sample_points

pytestmark = pytest.mark.gpu

try:
    _NCFG = len(nv.gemm_configs())
except ImportError:  # library not built on this host; the tests are skipped anyway
    _NCFG = 2
CONFIGS = [0] + list(range(1, 1 + _NCFG))


def run_gemm(A, SFA, B, SFB, alpha, M, N, K, config=0):
    sfa = nv.pack_scales(dev(SFA), K)
    sfb = nv.pack_scales(dev(SFB), K)
    D = nv.gemm(dev(A), sfa, dev(B), sfb, alpha, M, N, K, config=config)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    return D


def check_full(A, SFA, B, SFB, alpha, D, what):
    ref, abs_sum = O.gemm(A, SFA, B, SFB, alpha)
    return assert_within(host_f64(D), ref, abs_sum, alpha, what)


def check_sampled(A, SFA, B, SFB, alpha, D, M, N, n_samples, what):
    rows, cols = sample_points(M, N, n_samples)
    Dh = host_f64(D[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()])
    ref, abs_sum = O.gemm_at(A, SFA, B, SFB, alpha, rows, cols)
    assert_within(Dh, ref, abs_sum, alpha, what + " samples")
    for r0, r1, c0, c1 in corner_tiles(M, N):
        ref, abs_sum = O.gemm_tile(A, SFA, B, SFB, alpha, r0, r1, c0, c1)
        assert_within(host_f64(D[r0:r1, c0:c1]), ref, abs_sum, alpha, f"{what} tile {(r0, c0)}")


@pytest.mark.parametrize("config", CONFIGS)
def test_gemm_256_cube(config):
    M = N = K = 256
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=0)
    D = run_gemm(A, SFA, B, SFB, 1.0, M, N, K, config)
    check_full(A, SFA, B, SFB, 1.0, D, f"256^3 config {config}")


@pytest.mark.parametrize("config", CONFIGS)
def test_gemm_all_scales_one_is_bit_exact(config):
    # All scales 1.0: the sum is an integer GEMM on 2*codes divided by 4; partial
    # sums stay below 2^24 quarter units, so FP32 accumulation is exact in any
    # order and D must be the round-to-nearest-even BF16 of the exact value.
    M, N, K = 256, 256, 1024
    A = G.packed_codes_uniform(M, K, 1, "A")
    B = G.packed_codes_uniform(N, K, 1, "B")
    S1 = np.full((M, K // 16), 0x38, np.uint8)
    S2 = np.full((N, K // 16), 0x38, np.uint8)
    D = run_gemm(A, S1, B, S2, 1.0, M, N, K, config)
    exact = O.gemm_exact_units(A, S1, B, S2).astype(np.float64) * 2.0 ** -20
    want = O.f32_to_bf16_rne(exact.astype(np.float32))
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
    got = host_bits(D)
    assert np.array_equal(got, want), f"{int((got != want).sum())} elements differ"


@pytest.mark.parametrize("config", CONFIGS)
def test_gemm_single_block_products_are_exact(config):
    # K = 64 with only one 16-block scale non-zero per row: every output is one
    # block dot product times sfa*sfb, exact in FP32, so D is its BF16 rounding.
    M, N, K = 128, 256, 64
    A = G.packed_codes_uniform(M, K, 2, "A")
    B = G.packed_codes_uniform(N, K, 2, "B")
    SFA = np.zeros((M, 4), np.uint8)
    SFB = np.zeros((N, 4), np.uint8)
    rng = np.random.default_rng(9)
    blk = 2
    SFA[:, blk] = rng.integers(0x01, 0x7F, M)
    SFB[:, blk] = rng.integers(0x01, 0x7F, N)
    D = run_gemm(A, SFA, B, SFB, 1.0, M, N, K, config)
    ref, _ = O.gemm(A, SFA, B, SFB, 1.0)
    assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)
    want = O.f32_to_bf16_rne(ref.astype(np.float32))
    assert np.array_equal(host_bits(D), want)


@pytest.mark.parametrize("config", CONFIGS)
def test_gemm_distinct_scales_per_row_and_block(config):
    # One-hot-like structure: scales differ per (row, block), so any mix-up of
    # the scale-factor layout (rows, 32-row groups, blocks, bands) shows.
    M, N, K = 256, 256, 512
    A = G.packed_codes_uniform(M, K, 4, "A")
    B = G.packed_codes_uniform(N, K, 4, "B")
    r = np.arange(M)[:, None]
    c = np.arange(K // 16)[None, :]
    SFA = (0x18 + (r * 7 + c * 3) % 65).astype(np.uint8)
    SFB = (0x18 + (r * 5 + c * 11) % 65).astype(np.uint8)
    D = run_gemm(A, SFA, B, SFB, 0.75, M, N, K, config)
    check_full(A, SFA, B, SFB, 0.75, D, f"distinct scales config {config}")


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("M,N,K", [(200, 136, 320), (1, 8, 64), (129, 264, 576), (384, 520, 1088)])
def test_gemm_ragged_shapes(config, M, N, K):
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=M + N + K, scales="zero_sub")
    alpha = G.alpha_uniform(M)
    D = run_gemm(A, SFA, B, SFB, alpha, M, N, K, config)
    check_full(A, SFA, B, SFB, alpha, D, f"{M}x{N}x{K} config {config}")


def test_gemm_2048_full():
    S = 2048
    A, SFA, B, SFB = G.gemm_square_inputs(S, S, S, seed=0)
    alpha = G.alpha_uniform(0)
    D = run_gemm(A, SFA, B, SFB, alpha, S, S, S)
    check_full(A, SFA, B, SFB, alpha, D, "2048^3")


@pytest.mark.parametrize("S", [4096, 8192])
def test_gemm_square_sampled(S):
    A, SFA, B, SFB = G.gemm_square_inputs(S, S, S, seed=0)
    alpha = G.alpha_uniform(0)
    D = run_gemm(A, SFA, B, SFB, alpha, S, S, S)
    check_sampled(A, SFA, B, SFB, alpha, D, S, S, 512, f"{S}^3")


@pytest.mark.parametrize("S", [16384])
def test_gemm_large_square_zero_and_subnormal_scales(S):
    A, SFA, B, SFB = G.gemm_square_inputs(S, S, S, seed=0, scales="zero_sub")
    alpha = G.alpha_uniform(0)
    D = run_gemm(A, SFA, B, SFB, alpha, S, S, S)
    check_sampled(A, SFA, B, SFB, alpha, D, S, S, 1024, f"{S}^3 zero/subnormal scales")


def test_gemm_repeat_is_bit_identical():
    M, N, K = 1024, 1024, 2048
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=5)
    sfa, sfb = nv.pack_scales(dev(SFA), K), nv.pack_scales(dev(SFB), K)
    a, b = dev(A), dev(B)
    D1 = nv.gemm(a, sfa, b, sfb, 1.5, M, N, K)
    D2 = nv.gemm(a, sfa, b, sfb, 1.5, M, N, K)
    torch.cuda.synchronize()
    assert torch.equal(D1.view(torch.int16), D2.view(torch.int16))


@pytest.mark.parametrize("M", [128, 1024, 8192])
@pytest.mark.parametrize("N,K", [(5120, 5120), (17408, 5120), (5120, 17408), (6144, 5120)])
def test_gemm_llm_linear(M, N, K):
    # Activations N(0,1) and weights N(0,0.02) in BF16, quantised (byte-exact
    # against the oracle) with per-tensor scales; alpha = g_x * g_w.
    x = G.bf16_normal(M, K, 11, "x")
    w = G.bf16_normal(N, K, 11, "w", 0.02)
    gx, gw = O.global_scale(x), O.global_scale(w)
    alpha = float(np.float32(gx) * np.float32(gw))
    A, SFA = nv.quantize(dev_bf16(x), gx)
    B, SFB = nv.quantize(dev_bf16(w), gw)
    Ah, SFAh = O.quantize(x, gx)
    Bh, SFBh = O.quantize(w, gw)
    assert np.array_equal(SFA.cpu().numpy(), SFAh) and np.array_equal(A.cpu().numpy(), Ah)
    assert np.array_equal(SFB.cpu().numpy(), SFBh) and np.array_equal(B.cpu().numpy(), Bh)
    D = nv.gemm(A, nv.pack_scales(SFA, K), B, nv.pack_scales(SFB, K), alpha, M, N, K)
    torch.cuda.synchronize()
    if M * N * K <= 2 ** 34:
        check_full(Ah, SFAh, Bh, SFBh, alpha, D, f"llm {M}x{N}x{K}")
    else:
        check_sampled(Ah, SFAh, Bh, SFBh, alpha, D, M, N, 1024, f"llm {M}x{N}x{K}")

"""GPU parity of the W4A16 path: prepare is byte-exact against the oracle's
packer, linear is within the tolerance of the exact float64 reference and
bit-identical on repeat calls."""

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_gb300 as nv
from oracle import nvfp4_oracle as O
from synthetic import generators as G
from gpu_util import assert_within, corner_tiles, dev, dev_bf16, host_f64, sample_points

pytestmark = pytest.mark.gpu


def quantized_weight(N, K, seed):
    w = G.bf16_normal(N, K, seed, "w", 0.02)
    g = O.global_scale(w)
    W, SW = O.quantize(w, g)
    return W, SW, g


@pytest.mark.parametrize("N,K", [(16, 64), (256, 512), (5120, 5120)])
def test_prepare_byte_exact(N, K):
    W = G.packed_codes_uniform(N, K, 3, "W")
    SW = G.scales_with_zero_and_subnormal(N, K, 3, "SW", 0.1, 0.1)
    # negative scales too (sign folded into the codes)
    SW = np.where(np.random.default_rng(1).random(SW.shape) < 0.2, SW | 0x80, SW).astype(np.uint8)
    got = nv.w4a16_prepare(dev(W), dev(SW)).cpu().numpy()
    assert np.array_equal(got, O.w4a16_prepare(W, SW))


@pytest.mark.parametrize("M", [1, 2, 8, 9, 17, 32, 33, 64, 72, 144])
def test_linear_small_full(M):
    N, K = 256, 512
    x = G.bf16_normal(M, K, M, "x")
    W = G.packed_codes_uniform(N, K, M, "W")
    SW = G.scales_with_zero_and_subnormal(N, K, M, "SW", 0.05, 0.05)
    SW = np.where(np.random.default_rng(M).random(SW.shape) < 0.1, SW | 0x80, SW).astype(np.uint8)
    alpha = 0.375
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    y = nv.w4a16_linear(dev_bf16(x), wp, alpha, N)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    ref, abs_sum = O.w4a16_linear(x, W, SW, alpha)
    assert_within(host_f64(y), ref, abs_sum, alpha, f"w4a16 M={M}")


@pytest.mark.parametrize("M,N,K", [(40, 384, 768), (24, 256, 4096), (200, 128, 1280), (300, 256, 512)])
def test_linear_tensor_core_edges(M, N, K):
    # Ragged K (last weight chunk partly outside the tensor), many K chunks for few
    # rows (the K split across a cluster with its fixed-order reduction), and token
    # counts above one 256-token tile.
    x = G.bf16_normal(M, K, M + K, "x")
    W = G.packed_codes_uniform(N, K, M + K, "W")
    SW = G.scales_with_zero_and_subnormal(N, K, M + K, "SW", 0.05, 0.05)
    alpha = 1.25
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    y = nv.w4a16_linear(dev_bf16(x), wp, alpha, N)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    ref, abs_sum = O.w4a16_linear(x, W, SW, alpha)
    assert_within(host_f64(y), ref, abs_sum, alpha, f"w4a16 {M}x{N}x{K}")


@pytest.mark.parametrize("N,K", [(5120, 5120), (17408, 5120), (5120, 17408)])
@pytest.mark.parametrize("M", [1, 8, 32, 72, 144, 1024])
def test_linear_decode_shapes(M, N, K):
    x = G.bf16_normal(M, K, 21, "x")
    W, SW, g = quantized_weight(N, K, 21)
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    y = nv.w4a16_linear(dev_bf16(x), wp, g, N)
    torch.cuda.synchronize()
    if M * N * K <= 2 ** 34:
        ref, abs_sum = O.w4a16_linear(x, W, SW, g)
        assert_within(host_f64(y), ref, abs_sum, g, f"w4a16 {M}x{N}x{K}")
    else:
        rows, cols = sample_points(M, N, 1024)
        ref, abs_sum = O.w4a16_linear_at(x, W, SW, g, rows, cols)
        got = host_f64(y[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()])
        assert_within(got, ref, abs_sum, g, f"w4a16 {M}x{N}x{K} samples")
        for r0, r1, c0, c1 in corner_tiles(M, N):
            ref, abs_sum = O.w4a16_linear(x[r0:r1], W[c0:c1], SW[c0:c1], g)
            assert_within(host_f64(y[r0:r1, c0:c1]), ref, abs_sum, g, f"w4a16 tile {(r0, c0)}")


@pytest.mark.parametrize("M", [1, 32, 144])
def test_linear_repeat_is_bit_identical(M):
    N, K = 5120, 5120
    x = dev_bf16(G.bf16_normal(M, K, 2, "x"))
    W, SW, g = quantized_weight(N, K, 2)
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    y1 = nv.w4a16_linear(x, wp, g, N)
    y2 = nv.w4a16_linear(x, wp, g, N)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))

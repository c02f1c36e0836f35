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


def _chain_inputs(M, seed):
    # Two layers: x [M x 5120] -> W1 (N=1024, K=5120) -> y1 [M x 1024] -> W2 (N=5120, K=1024).
    x = dev_bf16(G.bf16_normal(M, 5120, seed, "x"))
    W1, SW1, g1 = quantized_weight(1024, 5120, seed)
    W2, SW2, g2 = quantized_weight(5120, 1024, seed + 1)
    return x, (nv.w4a16_prepare(dev(W1), dev(SW1)), g1), (nv.w4a16_prepare(dev(W2), dev(SW2)), g2)


@pytest.mark.parametrize("M", [1, 20, 144])
def test_linear_chain_waits_for_the_previous_call(M):
    # Each call may start before the previous kernel in the stream has finished
    # (programmatic dependent launch) and must wait for it before reading x: the
    # second layer reads the first layer's output.  Back-to-back calls must give
    # the same bits as calls separated by a device synchronisation, every time.
    x, (w1, g1), (w2, g2) = _chain_inputs(M, 31)
    y1 = torch.empty((M, 1024), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((M, 5120), dtype=torch.bfloat16, device="cuda")
    nv.w4a16_linear(x, w1, g1, 1024, out=y1)
    torch.cuda.synchronize()
    nv.w4a16_linear(y1, w2, g2, 5120, out=y2)
    torch.cuda.synchronize()
    want1, want2 = y1.clone(), y2.clone()
    for _ in range(20):
        y1.zero_()
        y2.zero_()
        nv.w4a16_linear(x, w1, g1, 1024, out=y1)
        nv.w4a16_linear(y1, w2, g2, 5120, out=y2)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(y1.view(torch.int16), want1.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), want2.view(torch.int16))


def test_linear_back_to_back_writes_keep_the_last():
    # Two calls writing the same y: the result is the second call's.
    N, K = 5120, 5120
    W, SW, g = quantized_weight(N, K, 4)
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    xa = dev_bf16(G.bf16_normal(1, K, 5, "xa"))
    xb = dev_bf16(G.bf16_normal(1, K, 6, "xb"))
    want = nv.w4a16_linear(xb, wp, g, N)
    torch.cuda.synchronize()
    y = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
    for _ in range(20):
        nv.w4a16_linear(xa, wp, g, N, out=y)
        nv.w4a16_linear(xb, wp, g, N, out=y)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("M", [1, 144])
def test_linear_graph_replay_matches_eager(M):
    # The calls allocate nothing and keep no per-call device state, so a captured
    # chain replays to the same bits as eager execution.
    x, (w1, g1), (w2, g2) = _chain_inputs(M, 41)
    e1 = nv.w4a16_linear(x, w1, g1, 1024)
    e2 = nv.w4a16_linear(e1, w2, g2, 5120)
    torch.cuda.synchronize()
    y1 = torch.empty_like(e1)
    y2 = torch.empty_like(e2)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            nv.w4a16_linear(x, w1, g1, 1024, out=y1, stream=s)
            nv.w4a16_linear(y1, w2, g2, 5120, out=y2, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        y1.zero_()
        y2.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(y1.view(torch.int16), e1.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), e2.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (17, 384, 1024), (32, 256, 4096), (72, 256, 512),
                                   (40, 384, 768), (300, 256, 1280)])
def test_linear_colscale(M, N, K):
    # One FP32 scale per output column (negative, zero and non-power-of-two values),
    # through the decode kernel (M <= 32, cluster K split) and the tensor-core path
    # (M > 32, with and without its cluster reduction).
    x = G.bf16_normal(M, K, M + 3, "x")
    W = G.packed_codes_uniform(N, K, M + 3, "W")
    SW = G.scales_with_zero_and_subnormal(N, K, M + 3, "SW", 0.05, 0.05)
    SW = np.where(np.random.default_rng(M).random(SW.shape) < 0.1, SW | 0x80, SW).astype(np.uint8)
    alpha = np.random.default_rng(N + M).uniform(-4.0, 4.0, N).astype(np.float32)
    alpha[::17] = 0.0
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    y = nv.w4a16_linear_colscale(dev_bf16(x), wp, dev(alpha), N)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    ref, sabs = O.w4a16_linear_colscale(x, W, SW, alpha)
    assert_within(host_f64(y), ref, sabs, 1.0, f"w4a16 colscale {M}x{N}x{K}")


def test_linear_colscale_rejects_bad_scale_pointer():
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device="cuda")
    wp = torch.zeros(nv.w4a16_prepared_bytes(128, 256), dtype=torch.uint8, device="cuda")
    y = torch.empty((1, 128), dtype=torch.bfloat16, device="cuda")
    lib = nv.load_library()
    st = lib.nvfp4_w4a16_linear_colscale(x.data_ptr(), wp.data_ptr(), None, y.data_ptr(), 1, 128, 256,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == -1
    a = torch.ones(129, dtype=torch.float32, device="cuda")
    st = lib.nvfp4_w4a16_linear_colscale(x.data_ptr(), wp.data_ptr(), a.data_ptr() + 4, y.data_ptr(), 1, 128, 256,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == -3


def test_linear_more_than_1024_tokens():
    # TileLang PR #3290 runs M > 1024 as 1024-row chunks; here token tiles of at most 256 cover
    # any M in one launch.
    M, N, K = 1300, 256, 512
    x = G.bf16_normal(M, K, 8, "x")
    W = G.packed_codes_uniform(N, K, 8, "W")
    SW = G.scales_uniform_normal(N, K, 8, "SW")
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    y = nv.w4a16_linear(dev_bf16(x), wp, 0.75, N)
    torch.cuda.synchronize()
    ref, abs_sum = O.w4a16_linear(x, W, SW, 0.75)
    assert_within(host_f64(y), ref, abs_sum, 0.75, "w4a16 M=1300")


@pytest.mark.parametrize("M", [1, 32, 144])
def test_weights_prepared_by_the_kernel_just_before(M):
    # The linear call streams its prepared weights before it waits for the previous
    # kernel in the stream; w4a16_prepare signals its dependents only by completing,
    # so a weight prepared immediately before the call (nothing in between) is read
    # complete.  Every repetition must give the bits of the first, checked against
    # the oracle.
    N, K = 5120, 5120
    W, SW, g = quantized_weight(N, K, 41)
    x = G.bf16_normal(M, K, 41, "x")
    xd, Wd, SWd = dev_bf16(x), dev(W), dev(SW)
    wp = torch.empty(nv.w4a16_prepared_bytes(N, K), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    want = None
    for it in range(8):
        wp.zero_()
        y.zero_()
        nv.w4a16_prepare(Wd, SWd, out=wp)
        nv.w4a16_linear(xd, wp, g, N, out=y)
        torch.cuda.synchronize()
        if want is None:
            want = y.clone()
            rows, cols = sample_points(M, N, 512)
            ref, abs_sum = O.w4a16_linear_at(x, W, SW, g, rows, cols)
            assert_within(host_f64(y[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]),
                          ref, abs_sum, g, "prepared just before")
        assert torch.equal(y.view(torch.int16), want.view(torch.int16)), f"iteration {it}"
    assert nv.device_error() == 0

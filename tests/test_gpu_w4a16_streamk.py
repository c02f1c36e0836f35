"""GPU parity of nvfp4_w4a16_linear_streamk, the W4A16 linear with the work split
evenly over the SMs (TileLang PR #3290, Design: the persistent stream-K kernel with a
deterministic fix-up of split tiles).  Outputs are within the tolerance of the exact
float64 reference; repeats and graph replays are bit-identical, and every call leaves
the workspace tickets at zero."""

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_gb300 as nv
from oracle import nvfp4_oracle as O
from synthetic import generators as G
from gpu_util import assert_within, corner_tiles, dev, dev_bf16, host_f64, sample_points

pytestmark = pytest.mark.gpu


def _ws():
    return torch.zeros(nv.w4a16_streamk_workspace_bytes(), dtype=torch.uint8, device="cuda")


def _tickets_zero(ws):
    # the tickets (up to 2 per SM) follow the partial slots: 2 x SMs x 32 KB
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    off = 2 * sms * 32 * 256 * 4
    return bool((ws[off:off + 8 * sms] == 0).all())


def _weights(N, K, seed, signed=True):
    W = G.packed_codes_uniform(N, K, seed, "W")
    SW = G.scales_with_zero_and_subnormal(N, K, seed, "SW", 0.05, 0.05)
    if signed:
        SW = np.where(np.random.default_rng(seed).random(SW.shape) < 0.1, SW | 0x80, SW).astype(np.uint8)
    return W, SW


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16, 17, 32])
def test_split_groups_full(M):
    # N = 384: a full 256-row group and a half one (rows past N read as zero);
    # K = 1280: 20 blocks per group, 40 units over one block per SM, so every group is
    # summed from about 20 parts through the workspace.
    N, K = 384, 1280
    x = G.bf16_normal(M, K, M, "x")
    W, SW = _weights(N, K, M)
    alpha = 0.625
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    ws = _ws()
    y = nv.w4a16_linear_streamk(dev_bf16(x), wp, alpha, N, ws)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert _tickets_zero(ws)
    ref, abs_sum = O.w4a16_linear(x, W, SW, alpha)
    assert_within(host_f64(y), ref, abs_sum, alpha, f"stream-K w4a16 M={M}")


@pytest.mark.parametrize("M", [2, 32])
def test_whole_groups_and_ragged_parts(M):
    # K = 256 (4 blocks per group) and 320 groups: each block's share (about 8.4
    # units) holds whole groups, written straight to y, and split ones at its ends.
    N, K = 256 * 320, 256
    x = G.bf16_normal(M, K, 40 + M, "x")
    W, SW = _weights(N, K, 40 + M)
    alpha = 1.5
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    ws = _ws()
    y = nv.w4a16_linear_streamk(dev_bf16(x), wp, alpha, N, ws)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    ref, abs_sum = O.w4a16_linear(x, W, SW, alpha)
    assert_within(host_f64(y), ref, abs_sum, alpha, f"stream-K whole groups M={M}")


@pytest.mark.parametrize("N,K", [(5120, 5120), (17408, 5120), (5120, 17408)])
@pytest.mark.parametrize("M", [1, 8, 32])
def test_decode_shapes(M, N, K):
    x = G.bf16_normal(M, K, 21, "x")
    w = G.bf16_normal(N, K, 21, "w", 0.02)
    g = O.global_scale(w)
    W, SW = O.quantize(w, g)
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    ws = _ws()
    y = nv.w4a16_linear_streamk(dev_bf16(x), wp, g, N, ws)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    rows, cols = sample_points(M, N, 1024)
    ref, abs_sum = O.w4a16_linear_at(x, W, SW, g, rows, cols)
    got = host_f64(y[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()])
    assert_within(got, ref, abs_sum, g, f"stream-K {M}x{N}x{K} samples")
    for r0, r1, c0, c1 in corner_tiles(M, N):
        ref, abs_sum = O.w4a16_linear(x[r0:r1], W[c0:c1], SW[c0:c1], g)
        assert_within(host_f64(y[r0:r1, c0:c1]), ref, abs_sum, g, f"stream-K tile {(r0, c0)}")


def test_colscale():
    M, N, K = 5, 640, 2304
    x = G.bf16_normal(M, K, 7, "x")
    W, SW = _weights(N, K, 7)
    acol = (np.random.default_rng(7).random(N) * 2 - 0.5).astype(np.float32)
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    ws = _ws()
    y = nv.w4a16_linear_streamk(dev_bf16(x), wp, 0.0, N, ws, alpha_col=dev(acol))
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    ref, sabs = O.w4a16_linear_colscale(x, W, SW, acol)
    assert_within(host_f64(y), ref, sabs, 1.0, "stream-K colscale")


@pytest.mark.parametrize("M", [1, 17, 32])
def test_repeat_and_graph_replay_are_bit_identical(M):
    N, K = 5120, 5120
    x = dev_bf16(G.bf16_normal(M, K, 2, "x"))
    W, SW = _weights(N, K, 2, signed=False)
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    ws = _ws()
    y1 = nv.w4a16_linear_streamk(x, wp, 0.5, N, ws)
    y2 = nv.w4a16_linear_streamk(x, wp, 0.5, N, ws)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    y = torch.empty_like(y1)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                nv.w4a16_linear_streamk(x, wp, 0.5, N, ws, out=y, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(4):
        y.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert _tickets_zero(ws)
    assert torch.equal(y.view(torch.int16), y1.view(torch.int16))


def test_chain_waits_for_the_previous_call():
    # The second layer reads the first layer's output; calls may start before the
    # previous kernel in the stream ends (programmatic dependent launch).
    M = 4
    x = dev_bf16(G.bf16_normal(M, 5120, 31, "x"))
    W1, SW1 = _weights(1024, 5120, 31, signed=False)
    W2, SW2 = _weights(5120, 1024, 32, signed=False)
    w1 = nv.w4a16_prepare(dev(W1), dev(SW1))
    w2 = nv.w4a16_prepare(dev(W2), dev(SW2))
    ws = _ws()
    y1 = torch.empty((M, 1024), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((M, 5120), dtype=torch.bfloat16, device="cuda")
    nv.w4a16_linear_streamk(x, w1, 0.01, 1024, ws, out=y1)
    torch.cuda.synchronize()
    nv.w4a16_linear_streamk(y1, w2, 0.02, 5120, ws, out=y2)
    torch.cuda.synchronize()
    want1, want2 = y1.clone(), y2.clone()
    for _ in range(20):
        y1.zero_()
        y2.zero_()
        nv.w4a16_linear_streamk(x, w1, 0.01, 1024, ws, out=y1)
        nv.w4a16_linear_streamk(y1, w2, 0.02, 5120, ws, out=y2)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(y1.view(torch.int16), want1.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), want2.view(torch.int16))


def _tc_tickets_zero(ws):
    # the tensor-core tickets (one per SM) follow the decode region and the 2 x SMs
    # tensor-core partial slots of 128 x 256 floats
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    off = (2 * sms * 32 * 256 * 4 + sms * 8 + 256) + 2 * sms * 128 * 256 * 4
    return bool((ws[off:off + 4 * sms] == 0).all())


@pytest.mark.parametrize("M,N,K", [
    (33, 256, 512),      # up to 256 tokens: the cluster-split tensor-core kernel
    (72, 384, 1280),
    (144, 1024, 2304),
    (256, 640, 4096),
    (300, 512, 1024),    # stream-K: two token tiles of 160 (150 valid each), 16 x 8 units
    (1024, 256, 2048),   # stream-K: four token tiles, 256 units
    (520, 1152, 768),    # stream-K: three token tiles of 176 (168 valid in the last), ragged shares
    (2048, 640, 4096),   # stream-K: eight token tiles, 2560 units on the SMs
])
def test_tensor_core_streamk(M, N, K):
    x = G.bf16_normal(M, K, 50 + M, "x")
    W, SW = _weights(N, K, 50 + M)
    alpha = 0.375
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    ws = _ws()
    y = nv.w4a16_linear_streamk(dev_bf16(x), wp, alpha, N, ws)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert _tc_tickets_zero(ws) and _tickets_zero(ws)
    ref, abs_sum = O.w4a16_linear(x, W, SW, alpha)
    assert_within(host_f64(y), ref, abs_sum, alpha, f"tensor-core stream-K {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(72, 17408, 5120), (144, 5120, 17408), (1024, 5120, 5120)])
def test_tensor_core_streamk_layer_shapes(M, N, K):
    x = G.bf16_normal(M, K, 22, "x")
    w = G.bf16_normal(N, K, 22, "w", 0.02)
    g = O.global_scale(w)
    W, SW = O.quantize(w, g)
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    ws = _ws()
    y = nv.w4a16_linear_streamk(dev_bf16(x), wp, g, N, ws)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert _tc_tickets_zero(ws)
    rows, cols = sample_points(M, N, 1024)
    ref, abs_sum = O.w4a16_linear_at(x, W, SW, g, rows, cols)
    got = host_f64(y[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()])
    assert_within(got, ref, abs_sum, g, f"tensor-core stream-K {M}x{N}x{K} samples")
    for r0, r1, c0, c1 in corner_tiles(M, N):
        ref, abs_sum = O.w4a16_linear(x[r0:r1], W[c0:c1], SW[c0:c1], g)
        assert_within(host_f64(y[r0:r1, c0:c1]), ref, abs_sum, g, f"tensor-core stream-K tile {(r0, c0)}")


def test_tensor_core_streamk_colscale_and_repeats():
    M, N, K = 600, 640, 2304  # three token tiles of 208 x 5 groups: the stream-K kernel
    x = G.bf16_normal(M, K, 8, "x")
    W, SW = _weights(N, K, 8)
    acol = (np.random.default_rng(8).random(N) * 2 - 0.5).astype(np.float32)
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    ws = _ws()
    xd = dev_bf16(x)
    ac = dev(acol)
    y1 = nv.w4a16_linear_streamk(xd, wp, 0.0, N, ws, alpha_col=ac)
    y2 = nv.w4a16_linear_streamk(xd, wp, 0.0, N, ws, alpha_col=ac)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    ref, sabs = O.w4a16_linear_colscale(x, W, SW, acol)
    assert_within(host_f64(y1), ref, sabs, 1.0, "tensor-core stream-K colscale")
    # graph replay of three calls: the same bits, tickets back at zero
    y = torch.empty_like(y1)
    gr = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(gr, stream=s):
            for _ in range(3):
                nv.w4a16_linear_streamk(xd, wp, 0.0, N, ws, alpha_col=ac, out=y, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        y.zero_()
        gr.replay()
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert _tc_tickets_zero(ws)
    assert torch.equal(y.view(torch.int16), y1.view(torch.int16))


def test_workspace_checks():
    N, K = 256, 512
    x = dev_bf16(G.bf16_normal(1, K, 3, "x"))
    W, SW = _weights(N, K, 3)
    wp = nv.w4a16_prepare(dev(W), dev(SW))
    small = torch.zeros(nv.w4a16_streamk_workspace_bytes() - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.w4a16_linear_streamk(x, wp, 1.0, N, small)
    assert e.value.status == -1
    with pytest.raises(nv.NVFP4Error) as e:
        nv.w4a16_linear_streamk(x, wp, float("inf"), N, _ws())
    assert e.value.status == -1

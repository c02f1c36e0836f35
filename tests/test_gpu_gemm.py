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


@pytest.mark.parametrize("S", [16384, 32768])
def test_gemm_large_square_zero_and_subnormal_scales(S):
    A, SFA, B, SFB = G.gemm_square_inputs(S, S, S, seed=0, scales="zero_sub")
    alpha = G.alpha_uniform(0)
    D = run_gemm(A, SFA, B, SFB, alpha, S, S, S)
    check_sampled(A, SFA, B, SFB, alpha, D, S, S, 1024, f"{S}^3 zero/subnormal scales")


@pytest.mark.parametrize("config", [4, 5])
@pytest.mark.parametrize("M,N,K", [(128, 256, 4096), (200, 136, 2048), (128, 520, 1344), (384, 264, 17408)])
def test_gemm_split_k_over_a_cluster(config, M, N, K):
    # Few tiles and long K: the K blocks are split over clusters of 2..8 CTAs
    # (uneven ranges when the block count is not a multiple; a ragged last block
    # when K % 256 != 0) and reduced in rank order through distributed shared memory.
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=K + N, scales="zero_sub")
    alpha = G.alpha_uniform(K)
    D = run_gemm(A, SFA, B, SFB, alpha, M, N, K, config)
    check_full(A, SFA, B, SFB, alpha, D, f"split-K {M}x{N}x{K} config {config}")
    D2 = run_gemm(A, SFA, B, SFB, alpha, M, N, K, config)
    assert torch.equal(D.view(torch.int16), D2.view(torch.int16))


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


def _llm_operands(M, N, K, seed):
    x = G.bf16_normal(M, K, seed, "x")
    w = G.bf16_normal(N, K, seed, "w", 0.02)
    return dev_bf16(x), dev_bf16(w), O.global_scale(x), O.global_scale(w)


@pytest.mark.parametrize("M,N,K", [(128, 5120, 5120), (512, 1024, 2048), (96, 768, 1024)])
def test_quantize_pack_gemm_chain_back_to_back(M, N, K):
    # quantize -> pack -> GEMM -> W4A16 (reading D as its activations), issued
    # back to back: every kernel may start before its predecessor ends (programmatic
    # launch) and must wait for it before reading what it wrote.  The chain must give
    # the bits of the same calls separated by device synchronisations, every time.
    x, w, gx, gw = _llm_operands(M, N, K, 17)
    B, SFB = nv.quantize(w, gw)
    sfb = nv.pack_scales(SFB, K)
    W2 = G.packed_codes_uniform(256, N, 3, "W2")
    S2 = G.scales_uniform_normal(256, N, 3, "S2")
    wp2 = nv.w4a16_prepare(dev(W2), dev(S2))
    A = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    SFA = torch.empty((M, K // 16), dtype=torch.uint8, device="cuda")
    sfa = torch.empty(nv.packed_scales_bytes(M, K), dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, 256), dtype=torch.bfloat16, device="cuda")
    alpha = float(np.float32(gx) * np.float32(gw))

    def chain(sync):
        s = torch.cuda.synchronize if sync else (lambda: None)
        nv.quantize(x, gx, A, SFA)
        s()
        nv.pack_scales(SFA, K, sfa)
        s()
        nv.gemm(A, sfa, B, sfb, alpha, M, N, K, out=D)
        s()
        nv.w4a16_linear(D, wp2, 0.5, 256, out=y)
        s()

    chain(True)
    torch.cuda.synchronize()
    want_d, want_y = D.clone(), y.clone()
    Ah, SFAh = O.quantize(G.bf16_normal(M, K, 17, "x"), gx)
    assert np.array_equal(A.cpu().numpy(), Ah) and np.array_equal(SFA.cpu().numpy(), SFAh)
    for _ in range(10):
        for t in (A, SFA, sfa, D, y):
            t.zero_()
        chain(False)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(D.view(torch.int16), want_d.view(torch.int16))
    assert torch.equal(y.view(torch.int16), want_y.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(128, 2048, 4096), (1024, 1024, 1024)])
def test_gemm_back_to_back_writes_keep_the_last(M, N, K):
    A1, SFA1, B, SFB = G.gemm_square_inputs(M, N, K, seed=6)
    A2, SFA2, _, _ = G.gemm_square_inputs(M, N, K, seed=7)
    sfa1, sfa2 = nv.pack_scales(dev(SFA1), K), nv.pack_scales(dev(SFA2), K)
    a1, a2, b, sfb = dev(A1), dev(A2), dev(B), nv.pack_scales(dev(SFB), K)
    want = nv.gemm(a2, sfa2, b, sfb, 1.0, M, N, K)
    torch.cuda.synchronize()
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for _ in range(10):
        nv.gemm(a1, sfa1, b, sfb, 1.0, M, N, K, out=D)
        nv.gemm(a2, sfa2, b, sfb, 1.0, M, N, K, out=D)
    torch.cuda.synchronize()
    assert torch.equal(D.view(torch.int16), want.view(torch.int16))


def _streamk_workspace():
    return torch.zeros(nv.gemm_streamk_workspace_bytes(), dtype=torch.uint8, device="cuda")


def _partials_written(ws):
    # the flag words take the first KB; the FP32 partial tiles follow
    return bool(ws[1024:].any())


@pytest.mark.parametrize("M,N,K", [(2304, 2304, 8192), (2200, 2104, 8192), (2304, 4864, 8192)])
def test_gemm_streamk_full(M, N, K):
    # 81 / 81 / 171 tiles of 256 x 256 on about 76 CTA pairs, 32 K-blocks each: the last
    # waves' (tile, K-block) units are split over the pairs, and tiles shared by two pairs
    # are finished from a partial in the workspace (ragged edges in the second shape).
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=M + K, scales="zero_sub")
    alpha = G.alpha_uniform(K)
    ws = _streamk_workspace()
    sfa, sfb, a, b = nv.pack_scales(dev(SFA), K), nv.pack_scales(dev(SFB), K), dev(A), dev(B)
    D = nv.gemm_streamk(a, sfa, b, sfb, alpha, M, N, K, ws)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert _partials_written(ws), "the stream-K schedule did not run"
    check_full(A, SFA, B, SFB, alpha, D, f"stream-K {M}x{N}x{K}")
    # the workspace is ready for the next call: same bits again, flags back to zero
    for _ in range(3):
        D2 = nv.gemm_streamk(a, sfa, b, sfb, alpha, M, N, K, ws)
    torch.cuda.synchronize()
    assert torch.equal(D.view(torch.int16), D2.view(torch.int16))
    flags = ws[:1024].view(torch.int32)
    assert int(flags.abs().sum()) == 0


def test_gemm_streamk_all_scales_one_is_bit_exact():
    M, N, K = 2304, 2304, 8192
    A = G.packed_codes_uniform(M, K, 1, "A")
    B = G.packed_codes_uniform(N, K, 1, "B")
    S1 = np.full((M, K // 16), 0x38, np.uint8)
    S2 = np.full((N, K // 16), 0x38, np.uint8)
    ws = _streamk_workspace()
    D = nv.gemm_streamk(dev(A), nv.pack_scales(dev(S1), K), dev(B), nv.pack_scales(dev(S2), K), 1.0, M, N, K, ws)
    torch.cuda.synchronize()
    assert _partials_written(ws)
    # all scales 1: every product is a multiple of 1/4 and every partial sum stays below
    # 36 K < 2^19, so the oracle's float64 sum (and its float32 rounding) is exact
    exact, _ = O.gemm(A, S1, B, S2, 1.0)
    assert np.array_equal(host_bits(D), O.f32_to_bf16_rne(exact.astype(np.float32)))


def test_gemm_streamk_llm_layer_and_graph_replay():
    # 1024 tokens x (5120, 5120): 80 tiles for ~76 pairs, the case stream-K is for.
    M, N, K = 1024, 5120, 5120
    x = G.bf16_normal(M, K, 13, "x")
    w = G.bf16_normal(N, K, 13, "w", 0.02)
    gx, gw = O.global_scale(x), O.global_scale(w)
    alpha = float(np.float32(gx) * np.float32(gw))
    A, sfa = nv.quantize_packed(dev_bf16(x), gx)
    B, sfb = nv.quantize_packed(dev_bf16(w), gw)
    ws = _streamk_workspace()
    D = nv.gemm_streamk(A, sfa, B, sfb, alpha, M, N, K, ws)
    torch.cuda.synchronize()
    Ah, SFAh = O.quantize(x, gx)
    Bh, SFBh = O.quantize(w, gw)
    check_sampled(Ah, SFAh, Bh, SFBh, alpha, D, M, N, 1024, "stream-K llm 1024x5120x5120")
    out = torch.empty_like(D)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            nv.gemm_streamk(A, sfa, B, sfb, alpha, M, N, K, ws, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(out.view(torch.int16), D.view(torch.int16))


def test_gemm_streamk_declined_runs_data_parallel():
    # 81 tiles but only 4 K-blocks each: the fix-up would cost more than the second wave
    # it saves, so the call runs the data-parallel pair kernel: nvfp4_gemm's bits, and
    # the workspace's partial tiles stay untouched.
    M, N, K = 2304, 2304, 1024
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=21)
    a, b, sfa, sfb = dev(A), dev(B), nv.pack_scales(dev(SFA), K), nv.pack_scales(dev(SFB), K)
    ws = _streamk_workspace()
    D = nv.gemm_streamk(a, sfa, b, sfb, 0.5, M, N, K, ws)
    want = nv.gemm(a, sfa, b, sfb, 0.5, M, N, K)
    torch.cuda.synchronize()
    assert not _partials_written(ws)
    assert torch.equal(D.view(torch.int16), want.view(torch.int16))


def test_gemm_streamk_rejects_bad_workspace():
    M = N = K = 512
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=3)
    a, b, sfa, sfb = dev(A), dev(B), nv.pack_scales(dev(SFA), K), nv.pack_scales(dev(SFB), K)
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.gemm_streamk(a, sfa, b, sfb, 1.0, M, N, K, small)
    assert e.value.status == -1


@pytest.mark.parametrize("M,N,K,config", [(1024, 2048, 4096, 3), (128, 5120, 5120, 0), (512, 1024, 2048, 1)])
def test_weights_written_by_the_kernel_just_before(M, N, K, config):
    # The GEMM reads its weight operand (B, SFB) before it waits for the previous
    # kernel in the stream.  The library's producers signal their dependents only by
    # completing, so weights they write immediately before the GEMM -- with nothing
    # in between -- must be complete when the GEMM reads them.  Two producers:
    # quantize_packed (codes and packed scales) and pack_scales (packed scales only).
    x, w, gx, gw = _llm_operands(M, N, K, 23)
    alpha = float(np.float32(gx) * np.float32(gw))
    A, SFA = nv.quantize_packed(x, gx)
    B = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    SFB = torch.empty(nv.packed_scales_bytes(N, K), dtype=torch.uint8, device="cuda")
    B_rm, SFB_rm = nv.quantize(w, gw)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    wh = G.bf16_normal(N, K, 23, "w", 0.02)
    Bh, SFBh = O.quantize(wh, gw)
    Ah, SFAh = O.quantize(G.bf16_normal(M, K, 23, "x"), gx)
    want = None
    for it in range(8):
        B.zero_()
        SFB.zero_()
        D.zero_()
        if it % 2 == 0:
            nv.quantize_packed(w, gw, B, SFB)
        else:
            B.copy_(B_rm)
            nv.pack_scales(SFB_rm, K, SFB)
        nv.gemm(A, SFA, B, SFB, alpha, M, N, K, out=D, config=config)
        torch.cuda.synchronize()
        if want is None:
            want = D.clone()
            check_sampled(Ah, SFAh, Bh, SFBh, alpha, D, M, N, 512, f"weights just written {M}x{N}x{K}")
        assert torch.equal(D.view(torch.int16), want.view(torch.int16)), f"iteration {it}"
    assert nv.device_error() == 0


def _config_index(tag):
    return 1 + next(i for i, n in enumerate(nv.gemm_configs()) if tag in n)


def test_clc_schedule_matches_static_pairs():
    # 12 x 12 = 144 tiles of 256 x 256 for ~76 co-resident CTA pairs: the first clusters
    # cancel pending ones and take their tiles (Colfax Research's SM120 NVFP4 GEMM
    # article, Appendix: cluster launch control).
    # Each tile is computed the same way under either schedule: identical bits.
    M = N = 3072
    K = 512
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=5)
    D_static = run_gemm(A, SFA, B, SFB, 0.5, M, N, K, config=_config_index("2cta_256x256_k256x4 ("))
    D_clc = run_gemm(A, SFA, B, SFB, 0.5, M, N, K, config=_config_index("clc"))
    assert torch.equal(D_static.view(torch.int16), D_clc.view(torch.int16))
    check_sampled(A, SFA, B, SFB, 0.5, D_clc, M, N, 512, "CLC 3072x3072x512")

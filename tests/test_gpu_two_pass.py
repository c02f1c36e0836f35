"""GPU parity of the two-pass (value + residual) W4A4 path against the oracle:
nvfp4_quantize_two_pass byte-exact, nvfp4_gemm_two_pass within the GEMM tolerance
(|D - ref| <= 2^-8 |ref| + 1e-6 |alpha| sum_k (|dq1_k| + |dq2_k|) |b_k|)."""

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_gb300 as nv
from oracle import nvfp4_oracle as O
from synthetic import generators as G
from gpu_util import assert_within, corner_tiles, dev, dev_bf16, host_f64, sample_points

pytestmark = pytest.mark.gpu


def _oracle_operand(x, g):
    c1, s1, c2, s2 = O.quantize_two_pass(x, g)
    A2, S2 = O.interleave_two_pass(c1, s1, c2, s2)
    return (c1, s1, c2, s2), A2, O.pack_scales(S2)


@pytest.mark.parametrize("R,K,std", [(1, 256, 1.0), (130, 512, 1.0), (300, 1280, 0.02), (128, 5120, 1.0),
                                     (1024, 5120, 1.0)])
def test_quantize_two_pass_byte_exact(R, K, std):
    x = G.bf16_normal(R, K, 17, "x", std)
    g = O.global_scale(x)
    codes2, sf2 = nv.quantize_two_pass(dev_bf16(x), g)
    torch.cuda.synchronize()
    _, A2, SP2 = _oracle_operand(x, g)
    assert np.array_equal(codes2.cpu().numpy(), A2)
    assert np.array_equal(sf2.cpu().numpy(), SP2)


def test_quantize_two_pass_edge_blocks():
    # Zero rows, blocks whose residual is exactly zero, tiny values whose scales
    # underflow, values that saturate the scale, and a global scale of 1.
    R, K = 3, 512
    x = np.zeros((R, K), np.float32)
    x[1, :16] = [6.0, 4.375, 2.8125, 2.125, 1.59375, 0.9375, 0.53125, 0.0,
                 -6.0, -4.25, -2.8125, -2.125, -1.5, -0.9375, -0.53125, 0.0]
    x[1, 16:32] = 3.0                       # representable: empty residual
    x[1, 32:48] = 1e-4                      # scales underflow to zero
    x[1, 48:64] = 3.0e5                     # scale saturates at 448
    rng = np.random.default_rng(2)
    x[2] = rng.standard_normal(K).astype(np.float32)
    bits = O.f32_to_bf16_rne(x)
    codes2, sf2 = nv.quantize_two_pass(dev_bf16(bits), 1.0)
    torch.cuda.synchronize()
    _, A2, SP2 = _oracle_operand(bits, 1.0)
    assert np.array_equal(codes2.cpu().numpy(), A2)
    assert np.array_equal(sf2.cpu().numpy(), SP2)


def _two_pass_case(M, N, K, seed):
    x = G.bf16_normal(M, K, seed, "x")
    gx = O.global_scale(x)
    B = G.packed_codes_uniform(N, K, seed, "B")
    SFB = G.scales_with_zero_and_subnormal(N, K, seed, "SFB", 0.05, 0.05)
    ops, A2, SP2 = _oracle_operand(x, gx)
    alpha = float(np.float32(gx) * np.float32(0.75))
    return x, gx, ops, A2, SP2, B, SFB, alpha


# The shapes reach every kernel family through the automatic choice over 2K:
# split-K clusters, CTA pairs (also with ragged M and N), 128 x 128 and 128 x 256 tiles.
@pytest.mark.parametrize("M,N,K", [(128, 512, 512), (1024, 2560, 512), (1000, 2600, 768),
                                   (10240, 128, 256), (128, 20480, 256)])
def test_gemm_two_pass_full(M, N, K):
    x, gx, ops, A2, SP2, B, SFB, alpha = _two_pass_case(M, N, K, M + N + K)
    D = nv.gemm_two_pass(dev(A2), dev(SP2), dev(B), nv.pack_scales(dev(SFB), K), alpha, M, N, K)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    ref, abs_sum = O.gemm_two_pass(*ops, B, SFB, alpha)
    assert_within(host_f64(D), ref, abs_sum, alpha, f"two-pass {M}x{N}x{K} "
                  f"({nv.gemm_config_name(nv.gemm_choose_config(M, N, 2 * K))})")


def test_gemm_two_pass_equals_plain_gemm_on_the_duplicated_weight():
    # Same kernels, same order of summation: the two-pass call is bit for bit
    # nvfp4_gemm over 2K with every 256-element K-block of the weight stored twice.
    M, N, K = 1024, 5120, 1024
    x, gx, ops, A2, SP2, B, SFB, alpha = _two_pass_case(M, N, K, 9)
    Bd, Sd = O.interleave_two_pass(B, SFB, B, SFB)
    a2, sp2 = dev(A2), dev(SP2)
    D2 = nv.gemm_two_pass(a2, sp2, dev(B), nv.pack_scales(dev(SFB), K), alpha, M, N, K)
    Dd = nv.gemm(a2, sp2, dev(Bd), nv.pack_scales(dev(Sd), 2 * K), alpha, M, N, 2 * K)
    torch.cuda.synchronize()
    assert torch.equal(D2.view(torch.int16), Dd.view(torch.int16))


def test_two_pass_llm_layer_chain_and_accuracy():
    # 1024 tokens x (5120, 5120): x quantised on the GPU in two passes, then the GEMM;
    # sampled against the oracle, and closer to the BF16 product than one pass.
    M, N, K = 1024, 5120, 5120
    x = G.bf16_normal(M, K, 23, "x")
    w = G.bf16_normal(N, K, 23, "w", 0.02)
    gx, gw = O.global_scale(x), O.global_scale(w)
    alpha = float(np.float32(gx) * np.float32(gw))
    xd = dev_bf16(x)
    A2, SP2 = nv.quantize_two_pass(xd, gx)
    A1, SP1 = nv.quantize_packed(xd, gx)
    B, SFBp = nv.quantize_packed(dev_bf16(w), gw)
    D2 = nv.gemm_two_pass(A2, SP2, B, SFBp, alpha, M, N, K)
    D1 = nv.gemm(A1, SP1, B, SFBp, alpha, M, N, K)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    c1, s1, c2, s2 = O.quantize_two_pass(x, gx)
    Bh, SFBh = O.quantize(w, gw)
    rows, cols = sample_points(M, N, 1024)
    Dh = host_f64(D2[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()])
    ref, abs_sum = O.gemm_two_pass_at(c1, s1, c2, s2, Bh, SFBh, alpha, rows, cols)
    assert_within(Dh, ref, abs_sum, alpha, "two-pass llm samples")
    for r0, r1, q0, q1 in corner_tiles(M, N):
        ref, abs_sum = O.gemm_two_pass(c1[r0:r1], s1[r0:r1], c2[r0:r1], s2[r0:r1], Bh[q0:q1], SFBh[q0:q1], alpha)
        assert_within(host_f64(D2[r0:r1, q0:q1]), ref, abs_sum, alpha, f"two-pass llm tile {(r0, q0)}")
    # against x times the dequantised weight (the activation's own quantisation error)
    xf = O.bf16_bits_to_f64(x[rows])
    wf = O.dequantize(Bh[cols], SFBh[cols]) * gw
    exact = (xf * wf).sum(axis=1)
    e1 = np.abs(host_f64(D1[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]) - exact)
    e2 = np.abs(Dh - exact)
    assert e2.mean() < e1.mean() / 4


def test_two_pass_rejects_k_not_multiple_of_256():
    x = dev_bf16(G.bf16_normal(4, 320, 1, "x"))
    with pytest.raises(nv.NVFP4Error) as e:
        nv.quantize_two_pass(x, 1.0)
    assert e.value.status == -2
    a = torch.zeros((128, 320), dtype=torch.uint8, device="cuda")
    s = torch.zeros(nv.packed_scales_bytes(128, 640), dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.gemm_two_pass(a, s, a, s, 1.0, 128, 128, 320)
    assert e.value.status == -2

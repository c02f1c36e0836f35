"""GPU parity of the operand producers: quantize and pack_scales are byte-exact
against the oracle."""

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_gb300 as nv
from oracle import nvfp4_oracle as O
from synthetic import generators as G
from gpu_util import dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("R,K", [(1, 64), (1, 16), (129, 320), (300, 1024), (256, 48), (8192, 5120)])
def test_pack_scales_byte_exact(R, K):
    sf = G.scales_with_zero_and_subnormal(R, K, 5, "sf", 0.05, 0.05)
    got = nv.pack_scales(dev(sf), K).cpu().numpy()
    want = O.pack_scales(sf)
    assert got.shape == want.shape
    assert np.array_equal(got, want)


def test_pack_scales_many_bands_and_unaligned_source():
    # More (band, 32-atom) tiles than resident thread blocks (the grid-stride path),
    # then a source one byte off a word boundary (the byte-load path).
    R, K = 128 * 1300, 64
    sf = G.scales_with_zero_and_subnormal(R, K, 6, "sf", 0.05, 0.05)
    assert np.array_equal(nv.pack_scales(dev(sf), K).cpu().numpy(), O.pack_scales(sf))
    R, K = 300, 1024
    sf = G.scales_with_zero_and_subnormal(R, K, 8, "sf", 0.05, 0.05)
    raw = dev(np.concatenate([np.zeros(1, np.uint8), sf.ravel()]))
    shifted = raw[1:].view(R, K // 16)
    assert shifted.data_ptr() % 4 != 0
    assert np.array_equal(nv.pack_scales(shifted, K).cpu().numpy(), O.pack_scales(sf))


@pytest.mark.parametrize("R,K,std", [(64, 512, 1.0), (300, 5120, 1.0), (128, 5120, 0.02), (8192, 5120, 1.0)])
def test_quantize_byte_exact(R, K, std):
    x = G.bf16_normal(R, K, 7, "x", std)
    g = O.global_scale(x)
    codes, sf = nv.quantize(dev_bf16(x), g)
    wc, ws = O.quantize(x, g)
    assert np.array_equal(sf.cpu().numpy(), ws)
    assert np.array_equal(codes.cpu().numpy(), wc)


def test_quantize_rounding_ties_and_edge_values():
    # Block 0: amax 6, g = 1 -> scale 1.0, so the elements hit every E2M1 tie exactly.
    # Block 1: scale tie 1.0625 (between 1.0 and 1.125) -> even encoding 0x38.
    # Block 2: scale tie 1.1875 (between 1.125 and 1.25) -> even encoding 0x3A.
    # Block 3: all zero.  Block 4: tiny values whose scale underflows to 0.
    # Block 5: values that saturate the scale (448) and the codes (6).
    vals = np.zeros((1, 6 * 16), dtype=np.float32)
    vals[0, 0:16] = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75,
                     -2.5, -3.5, -5.0, 0.1]
    vals[0, 16] = 6.375
    vals[0, 17:32] = np.linspace(-6, 6, 15)
    vals[0, 32] = 7.125
    vals[0, 33:48] = np.linspace(-7, 7, 15)
    vals[0, 64:80] = 1e-6
    vals[0, 80:96] = 3e4
    x = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    g = 1.0
    codes, sf = nv.quantize(dev_bf16(x), g)
    wc, ws = O.quantize(x, g)
    assert ws[0, :3].tolist() == [0x38, 0x38, 0x3A]
    assert ws[0, 3] == 0 and ws[0, 4] == 0 and ws[0, 5] == 0x7E
    assert np.array_equal(sf.cpu().numpy(), ws)
    assert np.array_equal(codes.cpu().numpy(), wc)


def test_quantize_then_pack_feeds_gemm_layout():
    x = G.bf16_normal(256, 512, 3, "x")
    g = O.global_scale(x)
    _, sf = nv.quantize(dev_bf16(x), g)
    packed = nv.pack_scales(sf, 512).cpu().numpy()
    assert np.array_equal(packed, O.pack_scales(O.quantize(x, g)[1]))


@pytest.mark.parametrize("R,K,std", [(1, 16, 1.0), (129, 320, 1.0), (300, 5120, 0.02), (256, 48, 1.0),
                                     (8192, 5120, 1.0)])
def test_quantize_packed_byte_exact(R, K, std):
    # Fused quantize + pack: codes as nvfp4_quantize, scales byte for byte the oracle's
    # pack of the oracle's row-major scales, zero padding included (ragged rows and
    # a ragged last atom).
    x = G.bf16_normal(R, K, 9, "x", std)
    g = O.global_scale(x)
    sf_packed = torch.full((nv.packed_scales_bytes(R, K),), 0xAB, dtype=torch.uint8, device="cuda")
    codes, sfp = nv.quantize_packed(dev_bf16(x), g, sf_packed=sf_packed)
    wc, ws = O.quantize(x, g)
    assert np.array_equal(codes.cpu().numpy(), wc)
    assert np.array_equal(sfp.cpu().numpy(), O.pack_scales(ws))


def test_quantize_packed_then_gemm():
    # The W4A4 prefill chain without a separate pack: quantize_packed on both operands,
    # then the GEMM, within the tolerance of the oracle on the oracle's own operands.
    M, N, K = 200, 384, 1024
    x = G.bf16_normal(M, K, 12, "x")
    w = G.bf16_normal(N, K, 12, "w", 0.02)
    gx, gw = O.global_scale(x), O.global_scale(w)
    A, sfa = nv.quantize_packed(dev_bf16(x), gx)
    B, sfb = nv.quantize_packed(dev_bf16(w), gw)
    alpha = float(np.float32(gx) * np.float32(gw))
    D = nv.gemm(A, sfa, B, sfb, alpha, M, N, K)
    torch.cuda.synchronize()
    Ah, SFAh = O.quantize(x, gx)
    Bh, SFBh = O.quantize(w, gw)
    ref, abs_sum = O.gemm(Ah, SFAh, Bh, SFBh, alpha)
    from gpu_util import assert_within, host_f64
    assert_within(host_f64(D), ref, abs_sum, alpha, "quantize_packed -> gemm")


@pytest.mark.parametrize("packed", [False, True])
def test_quantize_tiny_global_scale_byte_exact(packed):
    # g = 1e-37 and values ~1e-39 (bfloat16 subnormals): the block scales are E4M3
    # subnormals, scale * g is a float32 subnormal whose reciprocal overflows, and the
    # quantiser divides element by element.  The codes are mostly non-zero.
    R, K = 64, 512
    x = O.f32_to_bf16_rne((np.random.default_rng(4).standard_normal((R, K)) * 1e-39).astype(np.float32))
    g = 1e-37
    wc, ws = O.quantize(x, g)
    denom = (O.e4m3_table()[ws].astype(np.float32) * np.float32(g)).astype(np.float32)
    with np.errstate(over="ignore", divide="ignore"):
        assert np.isinf(np.float32(1) / denom[ws > 0]).all()  # the path under test is reached
    assert (O.unpack_codes(wc) != 0).mean() > 0.5
    if packed:
        codes, sfp = nv.quantize_packed(dev_bf16(x), g)
        assert np.array_equal(sfp.cpu().numpy(), O.pack_scales(ws))
    else:
        codes, sf = nv.quantize(dev_bf16(x), g)
        assert np.array_equal(sf.cpu().numpy(), ws)
    assert np.array_equal(codes.cpu().numpy(), wc)

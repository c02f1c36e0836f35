"""The Python binding refuses device buffers shorter than the sizes an entry point
reads or writes (the C ABI cannot see buffer sizes), before anything is launched."""

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_gb300 as nv

pytestmark = pytest.mark.gpu


def _u8(n):
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def test_gemm_entry_points_reject_short_buffers():
    M, N, K = 256, 256, 512
    A, B = _u8(M * K // 2), _u8(N * K // 2)
    SFA, SFB = _u8(nv.packed_scales_bytes(M, K)), _u8(nv.packed_scales_bytes(N, K))
    ws = _u8(nv.gemm_streamk_workspace_bytes())
    short = {"A": (_u8(M * K // 2 - 16), SFA, B, SFB), "SFA": (A, _u8(16), B, SFB),
             "B": (A, SFA, _u8(N * K // 2 - 16), SFB), "SFB": (A, SFA, B, _u8(16))}
    for name, (a, sa, b, sb) in short.items():
        with pytest.raises(ValueError, match=name):
            nv.gemm(a, sa, b, sb, 1.0, M, N, K)
        with pytest.raises(ValueError, match=name):
            nv.gemm_streamk(a, sa, b, sb, 1.0, M, N, K, ws)
        with pytest.raises(ValueError, match=name):
            nv.gemm_streamk_noalloc(a, sa, b, sb, 1.0, M, N, K)
    small_out = torch.empty((M, N - 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="out"):
        nv.gemm(A, SFA, B, SFB, 1.0, M, N, K, out=small_out)
    # two-pass: the activation operand holds 2K codes per row
    with pytest.raises(ValueError, match="A"):
        nv.gemm_two_pass(A, _u8(nv.packed_scales_bytes(M, 2 * K)), B, SFB, 1.0, M, N, K)
    torch.cuda.synchronize()
    assert nv.device_error() == 0


def test_producers_and_w4a16_reject_short_buffers():
    rows, K = 128, 512
    x = torch.zeros((rows, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="codes"):
        nv.quantize(x, 1.0, codes=_u8(rows * K // 2 - 8))
    with pytest.raises(ValueError, match="sf"):
        nv.quantize(x, 1.0, sf=_u8(rows * K // 16 - 1))
    with pytest.raises(ValueError, match="codes"):
        nv.quantize_packed(x, 1.0, codes=_u8(16))
    N = 256
    W, SW = _u8(N * K // 2).view(N, K // 2), _u8(N * K // 16).view(N, K // 16)
    with pytest.raises(ValueError, match="out"):
        nv.w4a16_prepare(W, SW, out=_u8(64))
    wp = nv.w4a16_prepare(W, SW)
    xs = torch.zeros((4, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="Wprep"):
        nv.w4a16_linear(xs, wp[:-16], 1.0, N)
    with pytest.raises(ValueError, match="out"):
        nv.w4a16_linear(xs, wp, 1.0, N, out=torch.empty((4, N - 8), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert nv.device_error() == 0

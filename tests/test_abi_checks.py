"""Host-side argument checks of the C ABI, exercised without a GPU.

Every entry point checks its arguments on the host and returns INVALID_ARG (-1),
UNSUPPORTED_SHAPE (-2) or MISALIGNED (-3) before it touches the device.  Each call
below carries at least one invalid argument, so none can reach a launch on any
machine; the pointers are stand-in addresses that are never dereferenced."""

import ctypes

import pytest

import nvfp4_block_scaled_gb300 as nv
from nvfp4_block_scaled_gb300 import build as nvbuild

INVALID, SHAPE, MISALIGNED = -1, -2, -3
P = 0x10000000      # a 16-byte-aligned stand-in address
ODD = P + 1         # misaligned by one byte
P4 = P + 4          # 4-byte but not 8-byte aligned
NAN, INF = float("nan"), float("inf")


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return nv.load_library()


def _gemm(lib, A=P, SFA=P, B=P, SFB=P, alpha=1.0, D=P, M=256, N=256, K=256):
    return lib.nvfp4_gemm(A, SFA, B, SFB, ctypes.c_float(alpha), D, M, N, K, None)


@pytest.mark.parametrize("kwargs,want", [
    (dict(A=None), INVALID), (dict(SFB=None), INVALID), (dict(D=None), INVALID),
    (dict(M=0), INVALID), (dict(N=4), INVALID), (dict(K=32), INVALID), (dict(M=-5), INVALID),
    (dict(M=1 << 31), INVALID),
    (dict(N=12), SHAPE), (dict(K=96), SHAPE),
    (dict(alpha=NAN), INVALID), (dict(alpha=INF), INVALID), (dict(alpha=-INF), INVALID),
    (dict(A=ODD), MISALIGNED), (dict(SFA=P4), MISALIGNED), (dict(D=ODD), MISALIGNED),
])
def test_gemm_argument_checks(lib, kwargs, want):
    assert _gemm(lib, **kwargs) == want


def test_gemm_variants_argument_checks(lib):
    f = ctypes.c_float(1.0)
    # an unknown configuration
    assert lib.nvfp4_gemm_config(P, P, P, P, f, P, 256, 256, 256, 99, None) == INVALID
    assert lib.nvfp4_gemm_config(P, P, P, P, f, P, 256, 256, 256, -1, None) == INVALID
    # stream-K: a missing or misaligned workspace
    assert lib.nvfp4_gemm_streamk(P, P, P, P, f, P, 256, 256, 256, None, 1 << 30, None) == INVALID
    assert lib.nvfp4_gemm_streamk(P, P, P, P, f, P, 256, 256, 256, ODD, 1 << 30, None) == MISALIGNED
    assert lib.nvfp4_gemm_streamk(P, P, P, P, f, P, 0, 256, 256, P, 1 << 30, None) == INVALID
    # two-pass: the weight's K must be a multiple of 256
    assert lib.nvfp4_gemm_two_pass(P, P, P, P, f, P, 256, 256, 320, None) == SHAPE
    assert lib.nvfp4_gemm_two_pass(None, P, P, P, f, P, 256, 256, 512, None) == INVALID


@pytest.mark.parametrize("fn", ["nvfp4_quantize", "nvfp4_quantize_packed", "nvfp4_quantize_two_pass"])
def test_quantizer_argument_checks(lib, fn):
    q = getattr(lib, fn)
    K = 512
    assert q(None, 4, K, ctypes.c_float(1.0), P, P, None) == INVALID
    assert q(P, 0, K, ctypes.c_float(1.0), P, P, None) == INVALID
    assert q(P, 4, 8, ctypes.c_float(1.0), P, P, None) == INVALID          # K < 16
    assert q(P, 4, 24, ctypes.c_float(1.0), P, P, None) == SHAPE           # K % 16
    for g in (0.0, -1.0, INF, NAN):
        assert q(P, 4, K, ctypes.c_float(g), P, P, None) == INVALID, g
    assert q(ODD, 4, K, ctypes.c_float(1.0), P, P, None) == MISALIGNED
    assert q(P, 4, K, ctypes.c_float(1.0), P4, P, None) == MISALIGNED      # codes need 8 bytes
    if fn != "nvfp4_quantize":
        assert q(P, 4, K, ctypes.c_float(1.0), P, ODD, None) == MISALIGNED  # packed scales: 16 bytes
    if fn == "nvfp4_quantize_two_pass":
        assert q(P, 4, 320, ctypes.c_float(1.0), P, P, None) == SHAPE       # K % 256


def test_pack_and_prepare_argument_checks(lib):
    assert lib.nvfp4_pack_scales(None, 4, 64, P, None) == INVALID
    assert lib.nvfp4_pack_scales(P, 4, 24, P, None) == SHAPE
    assert lib.nvfp4_pack_scales(P, 4, 64, ODD, None) == MISALIGNED
    assert lib.nvfp4_w4a16_prepare(P, P, 8, 256, P, None) == INVALID        # N < 16
    assert lib.nvfp4_w4a16_prepare(P, P, 24, 256, P, None) == SHAPE         # N % 16
    assert lib.nvfp4_w4a16_prepare(P, P, 128, 96, P, None) == SHAPE         # K % 64
    assert lib.nvfp4_w4a16_prepare(P, P, 128, 256, ODD, None) == MISALIGNED


def test_w4a16_argument_checks(lib):
    f = ctypes.c_float(0.5)
    lin = lib.nvfp4_w4a16_linear
    assert lin(None, P, f, P, 1, 256, 512, None) == INVALID
    assert lin(P, P, f, P, 0, 256, 512, None) == INVALID
    assert lin(P, P, f, P, 1, 192, 512, None) == SHAPE                      # N % 128
    assert lin(P, P, f, P, 1, 256, 320, None) == SHAPE                      # K % 256
    assert lin(ODD, P, f, P, 1, 256, 512, None) == MISALIGNED
    assert lin(P, P, ctypes.c_float(NAN), P, 1, 256, 512, None) == INVALID
    col = lib.nvfp4_w4a16_linear_colscale
    assert col(P, P, None, P, 1, 256, 512, None) == INVALID
    assert col(P, P, P4, P, 1, 256, 512, None) == MISALIGNED
    assert col(P, P, P, P, 1, 256, 320, None) == SHAPE


def test_w4a16_streamk_argument_checks(lib):
    f = ctypes.c_float(0.5)
    sk = lib.nvfp4_w4a16_linear_streamk
    assert sk(None, P, f, None, P, 1, 256, 512, P, 1 << 30, None) == INVALID
    assert sk(P, P, f, None, P, 1, 192, 512, P, 1 << 30, None) == SHAPE   # N % 128
    assert sk(P, P, f, None, P, 1, 256, 320, P, 1 << 30, None) == SHAPE   # K % 256
    assert sk(P, P, ctypes.c_float(NAN), None, P, 1, 256, 512, P, 1 << 30, None) == INVALID
    assert sk(P, P, f, P4, P, 1, 256, 512, P, 1 << 30, None) == MISALIGNED  # alpha_col
    assert sk(P, P, f, None, P, 1, 256, 512, None, 1 << 30, None) == INVALID  # workspace
    assert sk(P, P, f, None, P, 1, 256, 512, ODD, 1 << 30, None) == MISALIGNED


def test_mma_ceiling_argument_checks(lib):
    assert lib.nvfp4_mma_ceiling(3, 64, None, None, None) == INVALID
    assert lib.nvfp4_mma_ceiling(0, 6, None, None, None) == INVALID
    assert lib.nvfp4_mma_ceiling(0, 0, None, None, None) == INVALID


def test_size_helpers_reject_invalid_shapes(lib):
    assert nv.packed_scales_bytes(0, 64) == 0 and nv.packed_scales_bytes(4, -16) == 0
    assert nv.w4a16_prepared_bytes(0, 256) == 0 and nv.w4a16_prepared_bytes(128, 100) == 0

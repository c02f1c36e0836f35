"""Host-side checks of the C-ABI library: it builds, loads and exports every
symbol include/nvfp4.h declares; host-side helpers that need no GPU."""

import ctypes
import os
import re

import pytest

import nvfp4_block_scaled_gb300 as nv
from nvfp4_block_scaled_gb300 import build as nvbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return nv.load_library()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_binding_symbols():
    assert _header_functions() == sorted(nv.ABI_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings_and_version(lib):
    assert nv.status_string(0) == "NVFP4_OK"
    assert nv.status_string(-3) == "NVFP4_ERR_MISALIGNED"
    assert nv.status_string(-6) == "NVFP4_ERR_TIMEOUT"
    assert nv.status_string(12345) == "NVFP4_ERR_UNKNOWN"
    assert nv.version() == 10000


def test_size_helpers_match_closed_forms(lib):
    from oracle import nvfp4_oracle as O

    for rows, K in [(1, 16), (128, 64), (129, 320), (8192, 8192), (32768, 32768)]:
        assert nv.packed_scales_bytes(rows, K) == O.packed_scales_bytes(rows, K)
    assert nv.packed_scales_bytes(0, 64) == 0
    assert nv.packed_scales_bytes(4, 20) == 0
    for N, K in [(5120, 5120), (17408, 5120), (128, 256)]:
        assert nv.w4a16_prepared_bytes(N, K) == O.w4a16_prepared_bytes(N, K)
    assert nv.w4a16_prepared_bytes(100, 256) == 0


def test_gemm_config_names(lib):
    names = nv.gemm_configs()
    assert len(names) >= 2 and all(isinstance(n, str) for n in names)
    assert nv.gemm_config_name(0) is None


def test_bad_arguments_are_rejected_before_any_device_work(lib):
    L = nv.load_library()
    # Null pointers and non-positive sizes are rejected by the host checks,
    # which run before the device is queried, so no GPU is needed here.
    assert L.nvfp4_gemm(None, None, None, None, 1.0, None, 128, 128, 128, None) == -1
    assert L.nvfp4_gemm(16, 16, 16, 16, 1.0, 16, 0, 128, 128, None) == -1
    assert L.nvfp4_gemm(16, 16, 16, 16, 1.0, 16, 128, 128, 96, None) == -2     # K % 64
    assert L.nvfp4_gemm(16, 16, 16, 16, 1.0, 16, 128, 132, 128, None) == -2    # N % 8
    assert L.nvfp4_gemm(17, 16, 16, 16, 1.0, 16, 128, 128, 128, None) == -3    # misaligned A
    assert L.nvfp4_gemm(16, 16, 16, 16, float("nan"), 16, 128, 128, 128, None) == -1
    assert L.nvfp4_quantize(16, 4, 24, 1.0, 16, 16, None) == -2                # K % 16
    assert L.nvfp4_quantize(16, 4, 32, 0.0, 16, 16, None) == -1                # scale <= 0
    assert L.nvfp4_quantize(16, 4, 32, float("inf"), 16, 16, None) == -1
    assert L.nvfp4_pack_scales(16, 4, 32, 8, None) == -3                       # out misaligned
    assert L.nvfp4_w4a16_prepare(16, 16, 24, 64, 16, None) == -2               # N % 16
    assert L.nvfp4_w4a16_linear(16, 16, 1.0, 16, 1, 192, 256, None) == -2      # N % 128
    assert L.nvfp4_w4a16_linear(16, 16, 1.0, 16, 1, 128, 320, None) == -2      # K % 256
    assert L.nvfp4_w4a16_linear(16, 16, 1.0, 16, 0, 128, 256, None) == -1
    assert L.nvfp4_gemm_config(16, 16, 16, 16, 1.0, 16, 128, 128, 128, 99, None) == -1


def test_package_has_no_cpu_path():
    # The library never imports the oracle, and the oracle never imports the library.
    pkg = os.path.join(ROOT, "nvfp4_block_scaled_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                for bad in ("import oracle", "from oracle", "nvfp4_oracle"):
                    assert bad not in src, (f, bad)
    for dirpath, _, files in os.walk(os.path.join(ROOT, "oracle")):
        for f in files:
            if f.endswith(".py"):
                assert "nvfp4_block_scaled_gb300" not in open(os.path.join(dirpath, f)).read(), f

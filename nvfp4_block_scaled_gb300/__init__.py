"""Python binding of the GB300 NVFP4 block-scaled library (include/nvfp4.h).

Argument marshalling only: every computation runs in the CUDA kernels of
``_build/libnvfp4_gb300.so``.  The functions take torch CUDA tensors (torch is
used for device memory and streams), pass their data pointers and the current
CUDA stream to the C ABI, and raise ``NVFP4Error`` on a non-OK status.  There is
no CPU fallback: if the shared library has not been built, the first call raises.

Entry points (same names as the C ABI, without the ``nvfp4_`` prefix):
  quantize, quantize_packed, quantize_two_pass, packed_scales_bytes, pack_scales,
  gemm, gemm_streamk, gemm_streamk_workspace_bytes, gemm_streamk_noalloc,
  gemm_two_pass, gemm_config_name, gemm_choose_config, w4a16_prepared_bytes,
  w4a16_prepare, w4a16_linear, w4a16_linear_colscale, w4a16_streamk_workspace_bytes,
  w4a16_linear_streamk, mma_ceiling, device_error.

Every entry point checks that each tensor it is given holds at least the bytes the
call reads or writes (the C ABI takes raw pointers and cannot), and raises
``ValueError`` before anything is launched otherwise.
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libnvfp4_gb300.so")

#: Every symbol include/nvfp4.h declares.
ABI_SYMBOLS = (
    "nvfp4_status_string", "nvfp4_version", "nvfp4_quantize", "nvfp4_quantize_packed",
    "nvfp4_quantize_two_pass", "nvfp4_gemm_two_pass", "nvfp4_packed_scales_bytes",
    "nvfp4_pack_scales", "nvfp4_gemm", "nvfp4_gemm_config", "nvfp4_gemm_streamk",
    "nvfp4_gemm_streamk_workspace_bytes", "nvfp4_gemm_streamk_noalloc", "nvfp4_gemm_config_name",
    "nvfp4_gemm_choose_config", "nvfp4_w4a16_prepared_bytes", "nvfp4_w4a16_prepare",
    "nvfp4_w4a16_linear", "nvfp4_w4a16_linear_colscale", "nvfp4_w4a16_streamk_workspace_bytes",
    "nvfp4_w4a16_linear_streamk", "nvfp4_mma_ceiling", "nvfp4_device_error",
    "nvfp4_test_streamk_fault",
)

NVFP4_OK = 0


class NVFP4Error(RuntimeError):
    def __init__(self, fn: str, status: int, name: str):
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status
        self.status_name = name


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) and return the shared library; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"NVFP4 CUDA library not found at {path}; build it with "
            "`python -m nvfp4_block_scaled_gb300.build` (there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    c_i64, c_p, c_f, c_i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    sig = {
        "nvfp4_status_string": (ctypes.c_char_p, [c_i]),
        "nvfp4_version": (c_i, []),
        "nvfp4_quantize": (c_i, [c_p, c_i64, c_i64, c_f, c_p, c_p, c_p]),
        "nvfp4_quantize_packed": (c_i, [c_p, c_i64, c_i64, c_f, c_p, c_p, c_p]),
        "nvfp4_quantize_two_pass": (c_i, [c_p, c_i64, c_i64, c_f, c_p, c_p, c_p]),
        "nvfp4_gemm_two_pass": (c_i, [c_p, c_p, c_p, c_p, c_f, c_p, c_i64, c_i64, c_i64, c_p]),
        "nvfp4_packed_scales_bytes": (ctypes.c_size_t, [c_i64, c_i64]),
        "nvfp4_pack_scales": (c_i, [c_p, c_i64, c_i64, c_p, c_p]),
        "nvfp4_gemm": (c_i, [c_p, c_p, c_p, c_p, c_f, c_p, c_i64, c_i64, c_i64, c_p]),
        "nvfp4_gemm_config": (c_i, [c_p, c_p, c_p, c_p, c_f, c_p, c_i64, c_i64, c_i64, c_i, c_p]),
        "nvfp4_gemm_streamk": (c_i, [c_p, c_p, c_p, c_p, c_f, c_p, c_i64, c_i64, c_i64, c_p, ctypes.c_size_t, c_p]),
        "nvfp4_gemm_streamk_workspace_bytes": (ctypes.c_size_t, []),
        "nvfp4_gemm_streamk_noalloc": (c_i, [c_p, c_p, c_p, c_p, c_f, c_p, c_i64, c_i64, c_i64, c_i, c_p]),
        "nvfp4_gemm_config_name": (ctypes.c_char_p, [c_i]),
        "nvfp4_gemm_choose_config": (c_i, [c_i64, c_i64, c_i64]),
        "nvfp4_w4a16_prepared_bytes": (ctypes.c_size_t, [c_i64, c_i64]),
        "nvfp4_w4a16_prepare": (c_i, [c_p, c_p, c_i64, c_i64, c_p, c_p]),
        "nvfp4_w4a16_linear": (c_i, [c_p, c_p, c_f, c_p, c_i64, c_i64, c_i64, c_p]),
        "nvfp4_w4a16_linear_colscale": (c_i, [c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_p]),
        "nvfp4_w4a16_streamk_workspace_bytes": (ctypes.c_size_t, []),
        "nvfp4_mma_ceiling": (c_i, [c_i, c_i, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), c_p]),
        "nvfp4_w4a16_linear_streamk": (c_i, [c_p, c_p, c_f, c_p, c_p, c_i64, c_i64, c_i64, c_p, ctypes.c_size_t,
                                             c_p]),
        "nvfp4_device_error": (c_i, [c_p, c_i]),
        "nvfp4_test_streamk_fault": (c_i, [c_i, ctypes.c_uint64]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().nvfp4_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != NVFP4_OK:
        raise NVFP4Error(fn, status, status_string(status))


def _stream(stream=None) -> int:
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int:
    return int(t.data_ptr())


def _cuda(t, name, dtype=None):
    import torch

    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _need(t, name, nbytes):
    """Raise unless tensor t holds at least nbytes bytes.  The C ABI takes raw pointers
    and cannot see buffer sizes, so this is where a short buffer is caught before a
    kernel reads or writes past it.  Skipped when the size is not positive (invalid
    shapes are reported by the library's own argument checks)."""
    have = t.numel() * t.element_size()
    if nbytes > 0 and have < nbytes:
        raise ValueError(f"{name} holds {have} bytes, needs {nbytes}")


def _gemm_buffers(A, SFA, B, SFB, out, M, N, K, a_k):
    """Size checks shared by the GEMM entry points; a_k is the activation's K in codes
    (K, or 2K for the two-pass operand)."""
    M, N, K, a_k = int(M), int(N), int(K), int(a_k)
    _need(A, "A", M * a_k // 2)
    _need(SFA, "SFA", packed_scales_bytes(M, a_k) if M > 0 and a_k > 0 else 0)
    _need(B, "B", N * K // 2)
    _need(SFB, "SFB", packed_scales_bytes(N, K) if N > 0 and K > 0 else 0)
    _need(out, "out", 2 * M * N)


# ---------------------------------------------------------------- entry points

def version() -> int:
    return int(load_library().nvfp4_version())


def packed_scales_bytes(rows: int, K: int) -> int:
    return int(load_library().nvfp4_packed_scales_bytes(int(rows), int(K)))


def w4a16_prepared_bytes(N: int, K: int) -> int:
    return int(load_library().nvfp4_w4a16_prepared_bytes(int(N), int(K)))


def quantize(x, global_scale: float, codes=None, sf=None, stream=None):
    """bf16 [rows, K] -> (codes uint8 [rows, K/2], row-major scales uint8 [rows, K/16])."""
    import torch

    _cuda(x, "x", torch.bfloat16)
    rows, K = x.shape
    if codes is None:
        codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty((rows, K // 16), dtype=torch.uint8, device=x.device)
    _cuda(codes, "codes", torch.uint8)
    _cuda(sf, "sf", torch.uint8)
    _need(codes, "codes", rows * K // 2)
    _need(sf, "sf", rows * (K // 16))
    _check("nvfp4_quantize", load_library().nvfp4_quantize(
        _ptr(x), rows, K, float(global_scale), _ptr(codes), _ptr(sf), _stream(stream)))
    return codes, sf


def quantize_packed(x, global_scale: float, codes=None, sf_packed=None, stream=None):
    """bf16 [rows, K] -> (codes uint8 [rows, K/2], packed scales uint8 [packed_scales_bytes])."""
    import torch

    _cuda(x, "x", torch.bfloat16)
    rows, K = x.shape
    n = packed_scales_bytes(rows, K)
    if codes is None:
        codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=x.device)
    if sf_packed is None:
        sf_packed = torch.empty((n,), dtype=torch.uint8, device=x.device)
    _cuda(codes, "codes", torch.uint8)
    _cuda(sf_packed, "sf_packed", torch.uint8)
    if sf_packed.numel() < n:
        raise ValueError(f"sf_packed holds {sf_packed.numel()} bytes, needs {n}")
    _need(codes, "codes", rows * K // 2)
    _check("nvfp4_quantize_packed", load_library().nvfp4_quantize_packed(
        _ptr(x), rows, K, float(global_scale), _ptr(codes), _ptr(sf_packed), _stream(stream)))
    return codes, sf_packed


def quantize_two_pass(x, global_scale: float, codes2=None, sf2_packed=None, stream=None):
    """bf16 [rows, K] -> (codes2 uint8 [rows, K] (value and residual K-blocks of 256
    interleaved), packed scales uint8 [packed_scales_bytes(rows, 2K)])."""
    import torch

    _cuda(x, "x", torch.bfloat16)
    rows, K = x.shape
    n = packed_scales_bytes(rows, 2 * K)
    if codes2 is None:
        codes2 = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
    if sf2_packed is None:
        sf2_packed = torch.empty((n,), dtype=torch.uint8, device=x.device)
    _cuda(codes2, "codes2", torch.uint8)
    _cuda(sf2_packed, "sf2_packed", torch.uint8)
    if codes2.numel() < rows * K:
        raise ValueError(f"codes2 holds {codes2.numel()} bytes, needs {rows * K}")
    if sf2_packed.numel() < n:
        raise ValueError(f"sf2_packed holds {sf2_packed.numel()} bytes, needs {n}")
    _check("nvfp4_quantize_two_pass", load_library().nvfp4_quantize_two_pass(
        _ptr(x), rows, K, float(global_scale), _ptr(codes2), _ptr(sf2_packed), _stream(stream)))
    return codes2, sf2_packed


def pack_scales(sf, K: int | None = None, out=None, stream=None):
    """Row-major scales [rows, K/16] -> packed 128x4-atom buffer (uint8, flat)."""
    import torch

    _cuda(sf, "sf", torch.uint8)
    rows, C = sf.shape
    K = 16 * C if K is None else int(K)
    n = packed_scales_bytes(rows, K)
    if out is None:
        out = torch.empty((n,), dtype=torch.uint8, device=sf.device)
    _cuda(out, "out", torch.uint8)
    if out.numel() < n:
        raise ValueError(f"out holds {out.numel()} bytes, needs {n}")
    _check("nvfp4_pack_scales", load_library().nvfp4_pack_scales(_ptr(sf), rows, K, _ptr(out), _stream(stream)))
    return out


def gemm(A, SFA, B, SFB, alpha: float, M: int, N: int, K: int, out=None, config: int = 0, stream=None):
    """D = bf16(alpha * (A*SFA)(B*SFB)^T); A [M, K/2], B [N, K/2] packed codes, SFA/SFB packed."""
    import torch

    for t, nm in ((A, "A"), (SFA, "SFA"), (B, "B"), (SFB, "SFB")):
        _cuda(t, nm, torch.uint8)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _cuda(out, "out", torch.bfloat16)
    _gemm_buffers(A, SFA, B, SFB, out, M, N, K, K)
    lib = load_library()
    _check("nvfp4_gemm", lib.nvfp4_gemm_config(
        _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), float(alpha), _ptr(out), int(M), int(N), int(K),
        int(config), _stream(stream)))
    return out


def gemm_streamk_workspace_bytes() -> int:
    return int(load_library().nvfp4_gemm_streamk_workspace_bytes())


def gemm_streamk(A, SFA, B, SFB, alpha: float, M: int, N: int, K: int, workspace, out=None, stream=None):
    """nvfp4_gemm with the stream-K schedule; workspace: zero-filled uint8 CUDA tensor of at
    least gemm_streamk_workspace_bytes() bytes, reusable across calls on one stream."""
    import torch

    for t, nm in ((A, "A"), (SFA, "SFA"), (B, "B"), (SFB, "SFB"), (workspace, "workspace")):
        _cuda(t, nm, torch.uint8)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _cuda(out, "out", torch.bfloat16)
    _gemm_buffers(A, SFA, B, SFB, out, M, N, K, K)
    _check("nvfp4_gemm_streamk", load_library().nvfp4_gemm_streamk(
        _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), float(alpha), _ptr(out), int(M), int(N), int(K),
        _ptr(workspace), int(workspace.numel()), _stream(stream)))
    return out


def gemm_streamk_noalloc(A, SFA, B, SFB, alpha: float, M: int, N: int, K: int, out=None, stream=None,
                         reset_scratch: bool = False):
    """gemm_streamk with the library's static per-device workspace (no buffer passed, nothing
    allocated); calls overlapping on the GPU share that workspace and race."""
    import torch

    for t, nm in ((A, "A"), (SFA, "SFA"), (B, "B"), (SFB, "SFB")):
        _cuda(t, nm, torch.uint8)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _cuda(out, "out", torch.bfloat16)
    _gemm_buffers(A, SFA, B, SFB, out, M, N, K, K)
    _check("nvfp4_gemm_streamk_noalloc", load_library().nvfp4_gemm_streamk_noalloc(
        _ptr(A), _ptr(SFA), _ptr(B), _ptr(SFB), float(alpha), _ptr(out), int(M), int(N), int(K),
        1 if reset_scratch else 0, _stream(stream)))
    return out


def gemm_two_pass(A2, SFA2, B, SFB, alpha: float, M: int, N: int, K: int, out=None, stream=None):
    """D = bf16(alpha (dq1 + dq2) w^T) for a two-pass activation from quantize_two_pass;
    K is the weight's K (A2 holds 2K codes per row)."""
    import torch

    for t, nm in ((A2, "A2"), (SFA2, "SFA2"), (B, "B"), (SFB, "SFB")):
        _cuda(t, nm, torch.uint8)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A2.device)
    _cuda(out, "out", torch.bfloat16)
    _gemm_buffers(A2, SFA2, B, SFB, out, M, N, K, 2 * int(K))
    _check("nvfp4_gemm_two_pass", load_library().nvfp4_gemm_two_pass(
        _ptr(A2), _ptr(SFA2), _ptr(B), _ptr(SFB), float(alpha), _ptr(out), int(M), int(N), int(K),
        _stream(stream)))
    return out


def gemm_config_name(config: int):
    r = load_library().nvfp4_gemm_config_name(int(config))
    return None if r is None else r.decode()


def gemm_configs():
    names, i = [], 1
    while (n := gemm_config_name(i)) is not None:
        names.append(n)
        i += 1
    return names


def gemm_choose_config(M: int, N: int, K: int) -> int:
    r = int(load_library().nvfp4_gemm_choose_config(int(M), int(N), int(K)))
    if r < 0:
        _check("nvfp4_gemm_choose_config", r)
    return r


def w4a16_prepare(W, SW, out=None, stream=None):
    """NVFP4 weight (codes [N, K/2], row-major scales [N, K/16]) -> prepared bytes."""
    import torch

    _cuda(W, "W", torch.uint8)
    _cuda(SW, "SW", torch.uint8)
    N, half = W.shape
    K = 2 * half
    n = w4a16_prepared_bytes(N, K)
    if out is None:
        out = torch.empty((max(n, 1),), dtype=torch.uint8, device=W.device)
    _cuda(out, "out", torch.uint8)
    _need(SW, "SW", N * (K // 16))
    _need(out, "out", n)
    _check("nvfp4_w4a16_prepare", load_library().nvfp4_w4a16_prepare(
        _ptr(W), _ptr(SW), N, K, _ptr(out), _stream(stream)))
    return out


def w4a16_linear(x, Wprep, alpha: float, N: int, out=None, stream=None):
    """y = bf16(alpha * x * dequant(W)^T); x bf16 [M, K]."""
    import torch

    _cuda(x, "x", torch.bfloat16)
    _cuda(Wprep, "Wprep", torch.uint8)
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    _need(Wprep, "Wprep", w4a16_prepared_bytes(int(N), K))
    _need(out, "out", 2 * M * int(N))
    _check("nvfp4_w4a16_linear", load_library().nvfp4_w4a16_linear(
        _ptr(x), _ptr(Wprep), float(alpha), _ptr(out), M, int(N), K, _stream(stream)))
    return out


def w4a16_linear_colscale(x, Wprep, alpha_col, N: int, out=None, stream=None):
    """y = bf16(alpha_col[n] * x * dequant(W)^T); alpha_col float32 [N] on the device."""
    import torch

    _cuda(x, "x", torch.bfloat16)
    _cuda(Wprep, "Wprep", torch.uint8)
    _cuda(alpha_col, "alpha_col", torch.float32)
    if alpha_col.numel() != N:
        raise ValueError(f"alpha_col holds {alpha_col.numel()} scales, needs {N}")
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    _need(Wprep, "Wprep", w4a16_prepared_bytes(int(N), K))
    _need(out, "out", 2 * M * int(N))
    _check("nvfp4_w4a16_linear_colscale", load_library().nvfp4_w4a16_linear_colscale(
        _ptr(x), _ptr(Wprep), _ptr(alpha_col), _ptr(out), M, int(N), K, _stream(stream)))
    return out


def w4a16_streamk_workspace_bytes() -> int:
    return int(load_library().nvfp4_w4a16_streamk_workspace_bytes())


def w4a16_linear_streamk(x, Wprep, alpha: float, N: int, workspace, alpha_col=None, out=None, stream=None):
    """nvfp4_w4a16_linear_streamk: the work split evenly over the SMs; workspace
    is a zero-filled uint8 device tensor of w4a16_streamk_workspace_bytes() bytes."""
    import torch

    _cuda(x, "x", torch.bfloat16)
    _cuda(Wprep, "Wprep", torch.uint8)
    _cuda(workspace, "workspace", torch.uint8)
    if alpha_col is not None:
        _cuda(alpha_col, "alpha_col", torch.float32)
        if alpha_col.numel() != N:
            raise ValueError(f"alpha_col holds {alpha_col.numel()} scales, needs {N}")
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    _need(Wprep, "Wprep", w4a16_prepared_bytes(int(N), K))
    _need(out, "out", 2 * M * int(N))
    _check("nvfp4_w4a16_linear_streamk", load_library().nvfp4_w4a16_linear_streamk(
        _ptr(x), _ptr(Wprep), float(alpha), _ptr(alpha_col) if alpha_col is not None else None, _ptr(out), M,
        int(N), K, _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


MMA_KINDS = {"nvf4": 0, "bf16": 1, "fp8": 2}


def mma_ceiling(kind: str = "nvf4", iters: int = 8192, stream=None):
    """nvfp4_mma_ceiling: (TFLOP/s, median cycles per instruction) of back-to-back
    M = 256, N = 256 CTA-pair MMAs of `kind` ('nvf4', 'bf16' or 'fp8')."""
    tf, cyc = ctypes.c_double(0.0), ctypes.c_double(0.0)
    _check("nvfp4_mma_ceiling", load_library().nvfp4_mma_ceiling(
        MMA_KINDS[kind], int(iters), ctypes.byref(tf), ctypes.byref(cyc), _stream(stream)))
    return tf.value, cyc.value


def test_streamk_fault(skip_publish: bool, flag_wait_ns: int = 0) -> None:
    """Tests only: make the stream-K flag waits run out (see nvfp4_test_streamk_fault)."""
    _check("nvfp4_test_streamk_fault",
           load_library().nvfp4_test_streamk_fault(1 if skip_publish else 0, int(flag_wait_ns)))


def device_error(clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return (optionally clear) the device-side error status."""
    return int(load_library().nvfp4_device_error(_stream(stream), 1 if clear else 0))

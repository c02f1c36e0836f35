"""The timeout path of the GEMM kernels, made to run without any fault: the stream-K
fault injection (nvfp4_test_streamk_fault) makes the pairs that start a shared tile
skip publishing their partial, so the pairs that finish it wait on a flag that
nothing sets.  With a 1 ms limit those waits run out: the launch must end by itself,
report NVFP4_ERR_TIMEOUT through nvfp4_device_error, and leave the device usable --
the next call (workspace re-zeroed, or reset_scratch for the static-array entry)
must give the oracle's result."""

import time

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_gb300 as nv
from oracle import nvfp4_oracle as O
from synthetic import generators as G
from gpu_util import assert_within, corner_tiles, dev, host_f64, sample_points

pytestmark = pytest.mark.gpu

TIMEOUT = -6  # NVFP4_ERR_TIMEOUT


def _check(D, A, SFA, B, SFB, alpha, M, N, what):
    rows, cols = sample_points(M, N, 512)
    ref, abs_sum = O.gemm_at(A, SFA, B, SFB, alpha, rows, cols)
    assert_within(host_f64(D[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]), ref, abs_sum, alpha,
                  what + " samples")
    for r0, r1, c0, c1 in corner_tiles(M, N):
        ref, abs_sum = O.gemm_tile(A, SFA, B, SFB, alpha, r0, r1, c0, c1)
        assert_within(host_f64(D[r0:r1, c0:c1]), ref, abs_sum, alpha, f"{what} tile {(r0, c0)}")


def _run_injected(call):
    """Run `call` with the flag waits set to give up after 1 ms and nothing published;
    return (device error, seconds until the stream drained)."""
    assert nv.device_error() == 0
    try:
        nv.test_streamk_fault(True, 1_000_000)
        t0 = time.time()
        call()
        torch.cuda.synchronize()  # the launch ended by itself
        elapsed = time.time() - t0
        err = nv.device_error()
    finally:
        nv.test_streamk_fault(False, 0)
    return err, elapsed


def test_streamk_flag_wait_times_out_and_the_next_call_is_correct():
    # 1024 x 5120 x 5120: 80 tiles of 256 x 256 on about 76 pairs, so the stream-K
    # schedule shares tiles between pairs (the same layer the no-allocation test uses).
    M, N, K = 1024, 5120, 5120
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=21)
    a, sfa, b, sfb = dev(A), nv.pack_scales(dev(SFA), K), dev(B), nv.pack_scales(dev(SFB), K)
    alpha = 1.25
    ws = torch.zeros(nv.gemm_streamk_workspace_bytes(), dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    err, elapsed = _run_injected(lambda: nv.gemm_streamk(a, sfa, b, sfb, alpha, M, N, K, ws, out=D))
    assert err == TIMEOUT
    assert elapsed < 5.0

    ws.zero_()
    D.zero_()
    nv.gemm_streamk(a, sfa, b, sfb, alpha, M, N, K, ws, out=D)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    _check(D, A, SFA, B, SFB, alpha, M, N, "after a timeout")
    want = D.clone()

    # The static-array entry: the same timeout, then reset_scratch.
    err, elapsed = _run_injected(lambda: nv.gemm_streamk_noalloc(a, sfa, b, sfb, alpha, M, N, K, out=D))
    assert err == TIMEOUT
    assert elapsed < 5.0
    D.zero_()
    nv.gemm_streamk_noalloc(a, sfa, b, sfb, alpha, M, N, K, out=D, reset_scratch=True)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(D.view(torch.int16), want.view(torch.int16))


def test_injection_off_leaves_results_unchanged():
    # Turning the hook on and off again restores the normal schedule bit for bit.
    M, N, K = 1024, 5120, 5120
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=22)
    a, sfa, b, sfb = dev(A), nv.pack_scales(dev(SFA), K), dev(B), nv.pack_scales(dev(SFB), K)
    ws = torch.zeros(nv.gemm_streamk_workspace_bytes(), dtype=torch.uint8, device="cuda")
    D1 = nv.gemm_streamk(a, sfa, b, sfb, 0.75, M, N, K, ws)
    nv.test_streamk_fault(True, 1_000_000)
    nv.test_streamk_fault(False, 0)
    D2 = nv.gemm_streamk(a, sfa, b, sfb, 0.75, M, N, K, ws)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(D1.view(torch.int16), D2.view(torch.int16))

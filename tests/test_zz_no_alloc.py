"""nvfp4_gemm_streamk_noalloc: the stream-K GEMM on the library's static per-device
workspace.  Two calls in a row must give the bits of nvfp4_gemm_streamk on a caller
workspace, whether this file runs alone or after every other test."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import nvfp4_block_scaled_gb300 as nv
from synthetic import generators as G

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _operands(M, N, K, seed):
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=seed)
    return dev(A), nv.pack_scales(dev(SFA), K), dev(B), nv.pack_scales(dev(SFB), K)


def _bits(D):
    return D.view(torch.int16)


@pytest.mark.parametrize("M,N,K", [(2304, 2304, 8192), (1024, 5120, 5120), (2304, 2304, 1024)])
def test_noalloc_two_calls_match_caller_workspace(M, N, K):
    # the first two shapes run the stream-K split, the last is declined (data-parallel)
    a, sfa, b, sfb = _operands(M, N, K, seed=M + N + K)
    alpha = G.alpha_uniform(K)
    ws = torch.zeros(nv.gemm_streamk_workspace_bytes(), dtype=torch.uint8, device="cuda")
    want = nv.gemm_streamk(a, sfa, b, sfb, alpha, M, N, K, ws)
    D1 = nv.gemm_streamk_noalloc(a, sfa, b, sfb, alpha, M, N, K)
    D2 = nv.gemm_streamk_noalloc(a, sfa, b, sfb, alpha, M, N, K)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(_bits(D1), _bits(want))
    assert torch.equal(_bits(D2), _bits(want))


def test_noalloc_reset_scratch_gives_the_same_bits():
    M, N, K = 2304, 2304, 8192
    a, sfa, b, sfb = _operands(M, N, K, seed=5)
    D1 = nv.gemm_streamk_noalloc(a, sfa, b, sfb, 1.5, M, N, K)
    D2 = nv.gemm_streamk_noalloc(a, sfa, b, sfb, 1.5, M, N, K, reset_scratch=True)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert torch.equal(_bits(D1), _bits(D2))


def test_noalloc_rejects_bad_arguments_like_the_workspace_entry():
    M = N = K = 512
    a, sfa, b, sfb = _operands(M, N, K, seed=9)
    with pytest.raises(nv.NVFP4Error) as e:
        nv.gemm_streamk_noalloc(a, sfa, b, sfb, float("nan"), M, N, K)
    assert e.value.status == -1


def test_noalloc_stream_k_result_matches_the_oracle():
    # A 1024-token layer (80 tiles of 256 x 256 on about 76 CTA pairs): the stream-K
    # split runs through the static array, so its bits differ from the data-parallel
    # nvfp4_gemm somewhere (a different FP32 summation order on the shared tiles),
    # and sampled outputs and the corner tiles are within the tolerance of the exact
    # reference.
    from gpu_util import assert_within, corner_tiles, host_f64, sample_points
    from oracle import nvfp4_oracle as O

    M, N, K = 1024, 5120, 5120
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=11)
    a, sfa, b, sfb = dev(A), nv.pack_scales(dev(SFA), K), dev(B), nv.pack_scales(dev(SFB), K)
    alpha = G.alpha_uniform(11)
    D = nv.gemm_streamk_noalloc(a, sfa, b, sfb, alpha, M, N, K)
    Ddp = nv.gemm(a, sfa, b, sfb, alpha, M, N, K)
    torch.cuda.synchronize()
    assert nv.device_error() == 0
    assert not torch.equal(_bits(D), _bits(Ddp)), "the stream-K schedule did not run"
    rows, cols = sample_points(M, N, 512)
    ref, abs_sum = O.gemm_at(A, SFA, B, SFB, alpha, rows, cols)
    assert_within(host_f64(D[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]), ref, abs_sum, alpha,
                  "no-alloc stream-K samples")
    for r0, r1, c0, c1 in corner_tiles(M, N):
        ref, abs_sum = O.gemm_tile(A, SFA, B, SFB, alpha, r0, r1, c0, c1)
        assert_within(host_f64(D[r0:r1, c0:c1]), ref, abs_sum, alpha, f"no-alloc tile {(r0, c0)}")

"""Concurrent first use from several host threads: the library's once-per-device setup
(kernel attributes, occupancy queries) is reached by four threads at the same time,
each on its own stream, in a fresh process.  Every result must equal a run of the
same calls from one thread."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
import nvfp4_block_scaled_gb300 as nv
from synthetic import generators as G

d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
cases = []
for i, (M, N, K, cfg) in enumerate([(1024, 2560, 1024, 3), (256, 512, 1024, 5), (512, 4096, 512, 1), (128, 256, 512, 4)]):
    A, SFA, B, SFB = G.gemm_square_inputs(M, N, K, seed=i)
    cases.append((d(A), nv.pack_scales(d(SFA), K), d(B), nv.pack_scales(d(SFB), K), M, N, K, cfg))
W = G.packed_codes_uniform(1024, 512, 0, "W")
SW = G.scales_uniform_normal(1024, 512, 0, "SW")
wp = nv.w4a16_prepare(d(W), d(SW))
x = d(G.bf16_normal(4, 512, 0, "x").view(np.int16)).view(torch.bfloat16)
torch.cuda.synchronize()

results = [None] * 5
errors = []
start = threading.Barrier(5)

def work(i):
    try:
        s = torch.cuda.Stream()
        start.wait()
        with torch.cuda.stream(s):
            if i < 4:
                a, sa, b, sb, M, N, K, cfg = cases[i]
                out = nv.gemm(a, sa, b, sb, 1.0, M, N, K, config=cfg, stream=s)
            else:
                out = nv.w4a16_linear(x, wp, 0.5, 1024, stream=s)
        s.synchronize()
        results[i] = out.view(torch.int16).cpu()
    except Exception as e:
        errors.append(repr(e))

threads = [threading.Thread(target=work, args=(i,)) for i in range(5)]
for t in threads: t.start()
for t in threads: t.join()
assert not errors, errors
assert nv.device_error() == 0
# the same calls again, one after the other on the default stream
for i in range(4):
    a, sa, b, sb, M, N, K, cfg = cases[i]
    ref = nv.gemm(a, sa, b, sb, 1.0, M, N, K, config=cfg).view(torch.int16).cpu()
    assert torch.equal(ref, results[i]), i
ref = nv.w4a16_linear(x, wp, 0.5, 1024).view(torch.int16).cpu()
assert torch.equal(ref, results[4])
print("ok")
"""


def test_concurrent_first_use_from_four_threads():
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")

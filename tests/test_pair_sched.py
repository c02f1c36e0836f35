"""The CTA-pair GEMM's work schedule (csrc/pair_sched.h), compiled for the host and
checked over many (tiles, pairs, K-blocks) shapes: every (tile, K-block) unit is
computed by exactly one pair; under stream-K a pair has at most one head piece (the
start of a tile, right after its data-parallel tiles) and one tail piece (the end of
a tile, its last segment), and every tail finishes exactly the head of the pair
before it, which is what the kernel's fix-up relies on.  No GPU."""

import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "nvfp4_block_scaled_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <vector>
#include "pair_sched.h"
using nvfp4::sched::PairSched;

static int check(int tiles, int P, int KB, bool sk) {
  std::vector<int> cover(static_cast<size_t>(tiles) * KB, 0);
  std::vector<int> head_t(P, -1), head_k(P, -1), tail_t(P, -1), tail_k(P, -1);
  for (int p = 0; p < P; ++p) {
    PairSched s;
    s.init(p, P, tiles, KB, sk ? 1 : 0);
    const int n = s.count();
    int stage = 0;  // 0: data-parallel tiles, 1: after the head, 2: after the tail
    for (int i = 0; i < n; ++i) {
      int t, k0, k1, kind;
      if (sk) s.seg<true>(i, t, k0, k1, kind); else s.seg<false>(i, t, k0, k1, kind);
      if (t < 0 || t >= tiles || k0 < 0 || k1 > KB || k0 >= k1) return 1;
      for (int k = k0; k < k1; ++k) ++cover[static_cast<size_t>(t) * KB + k];
      if (stage == 2) return 2;  // nothing after the tail
      if (kind == PairSched::kFull) {
        if (k0 != 0 || k1 != KB) return 3;
      } else if (kind == PairSched::kHead) {
        if (!sk || k0 != 0 || k1 >= KB || stage != 0 || head_t[p] >= 0) return 4;
        head_t[p] = t; head_k[p] = k1; stage = 1;
      } else if (kind == PairSched::kTail) {
        if (!sk || k0 == 0 || k1 != KB || i != n - 1) return 5;
        tail_t[p] = t; tail_k[p] = k0; stage = 2;
      } else {
        return 6;
      }
    }
  }
  for (int c : cover)
    if (c != 1) return 7;
  for (int p = 0; p < P; ++p) {
    if (tail_t[p] >= 0 && (p == 0 || head_t[p - 1] != tail_t[p] || head_k[p - 1] != tail_k[p])) return 8;
    if (head_t[p] >= 0 && (p + 1 >= P || tail_t[p + 1] != head_t[p])) return 9;
  }
  return 0;
}

int main() {
  const int Ps[] = {1, 2, 3, 7, 37, 74, 76, 80};
  const int KBs[] = {1, 2, 3, 4, 16, 20, 32, 68};
  long cases = 0, sk_cases = 0, splits = 0;
  for (int P : Ps)
    for (int KB : KBs)
      for (int tiles = 1; tiles <= 400; ++tiles) {
        int r = check(tiles, P, KB, false);
        if (r) { std::printf("FAIL dp tiles=%d P=%d KB=%d code=%d\n", tiles, P, KB, r); return 1; }
        ++cases;
        if (tiles > P && tiles % P != 0) {  // the shapes the kernel runs with stream-K
          r = check(tiles, P, KB, true);
          if (r) { std::printf("FAIL sk tiles=%d P=%d KB=%d code=%d\n", tiles, P, KB, r); return 1; }
          ++sk_cases;
          for (int p = 0; p < P; ++p) {
            PairSched s;
            s.init(p, P, tiles, KB, 1);
            splits += s.has_head;
          }
        }
      }
  std::printf("ok %ld %ld %ld\n", cases, sk_cases, splits);
  return 0;
}
"""


def test_pair_schedule_covers_every_unit_once_and_pairs_heads_with_tails():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "sched_check.cc")
        exe = os.path.join(d, "sched_check")
        with open(src, "w") as f:
            f.write(HARNESS)
        subprocess.run([cxx, "-std=c++17", "-O2", "-I", CSRC, src, "-o", exe], check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    ok, cases, sk_cases, splits = r.stdout.split()
    assert ok == "ok" and int(sk_cases) > 1000 and int(splits) > 1000

"""The W4A16 tensor-core stream-K kernel's unit ranges (csrc/sk_units.h), compiled for
the host and checked over many (token tiles, groups, K-steps, blocks) shapes, for the
invariants its tickets and fix-up rely on (TileLang PR #3290, Design: contiguous (tile, k-tile)
ranges, a deterministic fix-up):

- the G ranges partition the U units, and cta_of finds the block of every unit;
- a block's range meets at most two groups only partly: the group of its first unit
  and that of its last; the groups in between it covers whole;
- every block that computes part of a split group takes exactly one ticket for it
  (the kernel's rule: one ticket for the first unit's group if split, one for the last
  unit's group if split and different), so the number of tickets equals the number of
  parts cta_of(last unit) - cta_of(first unit) + 1;
- the slot a part is written to (2b for the block's first segment, 2b + 1 otherwise)
  is the slot part_slot gives the block that adds the parts, and no two parts share
  a slot.
No GPU."""

import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "nvfp4_block_scaled_gb300", "csrc")

HARNESS = r"""
#include <cstdint>
#include <cstdio>
#include <map>
#include <set>
#include <utility>
#include <vector>
#include "sk_units.h"
using namespace nvfp4::sku;

// U = groups * KS units (token tiles folded into groups), G blocks.
static int check(int64_t groups, int KS, int G) {
  const int64_t U = groups * KS;
  if (unit_start(0, G, U) != 0 || unit_start(G, G, U) != U) return 1;
  for (int b = 0; b < G; ++b)
    if (unit_start(b + 1, G, U) <= unit_start(b, G, U)) return 2;  // G <= U: no empty range
  // cta_of on every unit (sampled when U is large: every range end and a stride)
  const int64_t stride = U > 200000 ? U / 50000 : 1;
  for (int64_t u = 0; u < U; u += stride) {
    const int b = cta_of(u, G, U);
    if (!(unit_start(b, G, U) <= u && u < unit_start(b + 1, G, U))) return 3;
  }
  for (int b = 0; b < G; ++b) {
    const int64_t e = unit_start(b + 1, G, U) - 1;
    if (cta_of(unit_start(b, G, U), G, U) != b || cta_of(e, G, U) != b) return 3;
  }
  std::map<int64_t, int> tickets;               // split group -> tickets taken
  std::map<int64_t, std::set<int>> writer_slot; // split group -> slots written by its parts
  std::set<int> used;
  for (int b = 0; b < G; ++b) {
    const int64_t u0 = unit_start(b, G, U), u1 = unit_start(b + 1, G, U);
    // segments, as the kernel walks them
    int nseg = 0, npartial = 0;
    for (int64_t su = u0; su < u1;) {
      const int64_t pg = su / KS;
      const int64_t s0 = su - pg * KS;
      const int64_t n = (KS - s0) < (u1 - su) ? (KS - s0) : (u1 - su);
      const bool whole = s0 == 0 && n == KS;
      if (!whole) {
        ++npartial;
        const bool first_seg = su == u0;
        const bool last_seg = su + n == u1;
        if (!first_seg && !last_seg) return 4;  // a partial group in the middle of a range
        const int slot = 2 * b + (first_seg ? 0 : 1);
        if (!used.insert(slot).second) return 5;  // two parts in one slot
        writer_slot[pg].insert(slot);
      }
      ++nseg;
      su += n;
    }
    if (npartial > 2) return 6;
    // tickets, as the kernel takes them (thread 0: first unit's group, thread 1: last unit's)
    for (int which = 0; which < 2; ++which) {
      const int64_t su = which == 0 ? u0 : u1 - 1;
      const int64_t pg = su / KS;
      const int64_t gu0 = pg * KS, gu1 = gu0 + KS;
      const bool split = u0 > gu0 || u1 < gu1;
      const bool distinct = which == 0 || (u0 / KS) != pg;
      if (split && distinct) ++tickets[pg];
    }
  }
  // every split group: one ticket per part, and the summing block reads the written slots
  for (auto& kv : writer_slot) {
    const int64_t pg = kv.first, gu0 = pg * KS;
    const int first = cta_of(gu0, G, U), last = cta_of(gu0 + KS - 1, G, U);
    if (tickets[pg] != last - first + 1) return 7;
    std::set<int> read;
    for (int p = first; p <= last; ++p) read.insert(part_slot(p, G, U, gu0));
    if (read != kv.second) return 8;
  }
  for (auto& kv : tickets)
    if (!writer_slot.count(kv.first)) return 9;  // a ticket for a group nobody split
  return 0;
}

int main() {
  long n = 0;
  const int kss[] = {4, 5, 8, 20, 80, 272};
  for (int ks : kss)
    for (int64_t groups = 1; groups <= 600; groups += (groups < 40 ? 1 : 37))
      for (int G = 1; G <= 152; G += (G < 16 ? 1 : 9)) {
        if (static_cast<int64_t>(G) > groups * ks) continue;
        const int r = check(groups, ks, G);
        ++n;
        if (r != 0) {
          std::printf("FAIL %d groups=%lld KS=%d G=%d\n", r, static_cast<long long>(groups), ks, G);
          return 1;
        }
      }
  std::printf("OK %ld\n", n);
  return 0;
}
"""


def test_tensor_core_streamk_unit_ranges():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "h.cpp")
        exe = os.path.join(d, "h")
        with open(src, "w") as f:
            f.write(HARNESS)
        subprocess.run([cxx, "-std=c++17", "-O2", "-I", CSRC, src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
        assert out.returncode == 0, out.stdout + out.stderr
        assert out.stdout.startswith("OK")

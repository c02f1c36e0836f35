// sk_units.h -- the unit ranges of the W4A16 tensor-core stream-K kernel, as plain code
// that compiles for the device and for the host (a host-side test checks the
// invariants the kernel's tickets and fix-up rely on).
//
// TileLang PR #3290, Design, the persistent stream-K kernel: U units (token tile, 128-row group,
// 64-K step), group-major, split into G contiguous ranges, one per block.  A block's
// range meets at most two groups only partly (the first and the last it touches);
// every group it covers in between goes to the output whole.  The part of a split
// group that a block computes is stored in slot 2b of the workspace if the group is
// the block's first segment, 2b + 1 if it is its last.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define NVFP4_SKU_HD __host__ __device__
#else
#define NVFP4_SKU_HD
#endif

namespace nvfp4 {
namespace sku {

// First unit of block i of G over U units (block G's "first unit" is U).
NVFP4_SKU_HD inline int64_t unit_start(int i, int G, int64_t U) { return static_cast<int64_t>(i) * U / G; }

// The block whose range holds unit u (0 <= u < U).
NVFP4_SKU_HD inline int cta_of(int64_t u, int G, int64_t U) {
  int i = static_cast<int>((u * G) / U);
  while (i + 1 < G && unit_start(i + 1, G, U) <= u) ++i;
  while (i > 0 && unit_start(i, G, U) > u) --i;
  return i;
}

// Slot holding block p's part of the group whose first unit is gu0: the group is p's
// first segment when p's range starts inside (or at the start of) it.
NVFP4_SKU_HD inline int part_slot(int p, int G, int64_t U, int64_t gu0) {
  return 2 * p + (unit_start(p, G, U) >= gu0 ? 0 : 1);
}

}  // namespace sku
}  // namespace nvfp4

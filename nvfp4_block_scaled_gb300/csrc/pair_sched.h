// pair_sched.h -- the work schedule of the CTA-pair GEMM kernel (data-parallel or
// stream-K), as plain code that compiles for the device and for the host (a host-side
// test checks its coverage invariants).
#pragma once

#include <cstdint>

// Member functions defined in the class are inline; on the device side they are
// host-and-device functions.
#if defined(__CUDACC__)
#define NVFP4_HD __host__ __device__
#else
#define NVFP4_HD
#endif

namespace nvfp4 {
namespace sched {

// Work of one pair, as a list of segments (tile, K-stage range, kind) that every
// role walks in the same order.
//   Data-parallel (SK = false): tiles pair, pair + P, pair + 2P, ..., all full.
//   Stream-K (SK = true; tiles >= P and not a multiple of P): the first
//   (tiles / P - 1) waves stay data-parallel (strided tiles keep a wave's operands
//   together in L2); the remaining R tiles (P <= R < 2P) form R x KB (tile, stage)
//   units split evenly over the P pairs.  Each pair's range holds at least KB units,
//   so a tile is shared by at most two pairs: pair p's range may end inside a tile
//   (its HEAD piece: stages [0, k_end), published to the workspace) and begin inside
//   the tile whose head pair p - 1 computed (its TAIL piece: stages [k_first, KB),
//   added to that head partial).  Order: data-parallel tiles, the head piece, the
//   whole stream-K tiles, the tail piece -- so a head is published long before the
//   pair that needs it gets there.
struct PairSched {
  enum { kFull = 0, kHead = 1, kTail = 2 };
  int p, P, tiles, KB;
  int dp;                       // data-parallel tiles of this pair
  int t_first, k_first, t_last, k_end, tf0, nfull, has_head, has_tail;

  NVFP4_HD void init(int p_, int P_, int tiles_, int KB_, int streamk) {
    p = p_; P = P_; tiles = tiles_; KB = KB_;
    has_head = has_tail = nfull = 0;
    tf0 = t_first = t_last = k_first = k_end = 0;
    if (!streamk) {
      dp = p < tiles ? (tiles - p + P - 1) / P : 0;
      return;
    }
    dp = tiles / P - 1;
    const int T0 = dp * P;
    const int64_t U = static_cast<int64_t>(tiles - T0) * KB;
    const int64_t u0 = static_cast<int64_t>(p) * U / P, u1 = static_cast<int64_t>(p + 1) * U / P;
    t_first = T0 + static_cast<int>(u0 / KB);
    k_first = static_cast<int>(u0 % KB);
    t_last = T0 + static_cast<int>((u1 - 1) / KB);
    k_end = static_cast<int>((u1 - 1) % KB) + 1;
    has_tail = k_first > 0;
    has_head = k_end < KB;
    tf0 = has_tail ? t_first + 1 : t_first;
    const int tf1 = has_head ? t_last - 1 : t_last;
    nfull = tf1 >= tf0 ? tf1 - tf0 + 1 : 0;
  }
  NVFP4_HD int count() const { return dp + has_head + nfull + has_tail; }
  template <bool SK>
  NVFP4_HD void seg(int s, int& tile, int& kb0, int& kb1, int& kind) const {
    if (!SK || s < dp) { tile = p + s * P; kb0 = 0; kb1 = KB; kind = kFull; return; }
    s -= dp;
    if (has_head) {
      if (s == 0) { tile = t_last; kb0 = 0; kb1 = k_end; kind = kHead; return; }
      --s;
    }
    if (s < nfull) { tile = tf0 + s; kb0 = 0; kb1 = KB; kind = kFull; return; }
    tile = t_first; kb0 = k_first; kb1 = KB; kind = kTail;
  }
};

}  // namespace sched
}  // namespace nvfp4

// gemm_w4a4.cu -- NVFP4 block-scaled GEMM on the sm_103a tcgen05 tensor cores.
//
// D[m,n] = bf16(alpha * sum_k (A[m,k] SFA[m,k/16]) (B[n,k] SFB[n,k/16])), FP32 accumulation.
//
// Structure (after Colfax Research, "Optimizing an NVFP4 Blockscaled GEMM on RTX
// PRO 6000 Blackwell GPU (SM120)": Version 1's warp-specialised persistent kernel
// with a TMA producer and an mbarrier ring, Version 2's swizzled raster, Versions
// 3/4's store path kept off the MMA issuer), rebuilt for tcgen05:
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) and the 512-byte scale
//               atoms (bulk copies) of one K block per pipeline stage.
//   warp 1      allocates TMEM; lane 0 issues tcgen05.cp (scale atoms -> TMEM) and
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X, then commits
//               the stage back to the producer and the accumulator to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld of the FP32 accumulator, alpha in FP32,
//               round-to-nearest-even to BF16, stores to D.
// Tiles are 128 x BN (BN = 128 or 256) per CTA; a persistent grid walks them in a
// grouped raster so that a wave shares A rows and B columns in L2.  Large shapes run
// the CTA-pair kernel (256 x 256 tiles), optionally with a stream-K schedule over a
// caller workspace; shapes with few tiles split K over a thread block cluster (the
// split-K kernel).  Every kernel supports programmatic dependent launch: its
// producer streams the first weight (B) stages before it waits for the previous
// grid in the stream, and loads A only after.  Every kernel also takes b_shift: with
// 1, A holds 2K codes (the two-pass activation, value and residual K-blocks
// interleaved) and A's K-block kb meets B's K-block kb >> 1, so both passes
// accumulate into one tile while the weight is read once.

#include <cuda_bf16.h>

#include "internal.h"
#include "pair_sched.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 256;               // K elements per stage
constexpr int kBKBytes = kBK / 2;      // packed bytes per row per stage (one 128-byte swizzle row)
constexpr int kMmaK = 64;              // K per tcgen05.mma (kind::mxf4nvf4)
constexpr int kKSteps = kBK / kMmaK;   // MMAs per stage
constexpr int kAtom = 512;             // bytes of one scale atom (128 rows x 64 K)
constexpr int kThreads = 192;

template <int BN, int STAGES, int ACC_BUFS>
struct Cfg {
  static constexpr int kBands = BN / 128;
  static constexpr int kABytes = kBM * kBKBytes;
  static constexpr int kBBytes = BN * kBKBytes;
  static constexpr int kSFABytes = kKSteps * kAtom;
  static constexpr int kSFBBytes = kBands * kKSteps * kAtom;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kABytes;
  static constexpr int kOffSFA = kOffB + STAGES * kBBytes;
  static constexpr int kOffSFB = kOffSFA + STAGES * kSFABytes;
  static constexpr int kOffBar = kOffSFB + STAGES * kSFBBytes;
  static constexpr int kNumBars = 2 * STAGES + 2 * ACC_BUFS;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for 1024-byte alignment
  // TMEM columns: accumulators, then per stage the SFA and SFB scale columns.
  static constexpr int kSFACols = kKSteps * 4;
  static constexpr int kSFBCols = kKSteps * 4 * kBands;
  static constexpr int kTmemSF = ACC_BUFS * BN;
  static constexpr int kTmemUsed = kTmemSF + STAGES * (kSFACols + kSFBCols);
  static constexpr int kTmemCols = kTmemUsed <= 128 ? 128 : kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Instruction descriptor, kind::mxf4nvf4: A and B E2M1 (format 1) K-major, dense,
// UE4M3 scales (bit 23 = 0), N >> 3 in bits 17..22, M >> 4 in bits 24..28.
template <int BN>
__host__ __device__ constexpr uint32_t idesc_nvf4_m128() {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(kBM >> 4) << 24);
}

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_n, int& mb,
                                            int& nb) {
  const int per_group = tiles_m * group_n;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int n0 = g * group_n;
  const int gw = min(group_n, tiles_n - n0);
  mb = r / gw;
  nb = n0 + (r - mb * gw);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// A copies held back until the previous grid in the stream has completed (the
// producers' side of programmatic dependent launch): up to N stages whose B
// copies are already in flight.  flush() waits for the grid dependency, then
// issues the held-back copies through load(stage, kb, m_block, n_atoms).
template <int N>
struct DeferredA {
  int n = 0;
  bool done = false;
  int st[N], kb[N], mb[N], nk[N];
  __device__ bool full() const { return !done && n == N; }
  __device__ void add(int s, int k, int m, int a) {
    st[n] = s; kb[n] = k; mb[n] = m; nk[n] = a;
    ++n;
  }
  template <typename F>
  __device__ void flush(F&& load) {
    griddep_wait();
    for (int i = 0; i < n; ++i) load(st[i], kb[i], mb[i], nk[i]);
    done = true;
  }
};

template <int BN, int STAGES, int ACC_BUFS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const uint8_t* __restrict__ SFA, const uint8_t* __restrict__ SFB,
                     __nv_bfloat16* __restrict__ D, float alpha, int M, int N, int K, int tiles_m,
                     int tiles_n, int group_n, int b_shift) {
  using C = Cfg<BN, STAGES, ACC_BUFS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::kOffBar;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_accf = bar_empty + 8 * STAGES;
  const uint32_t bar_acce = bar_accf + 8 * ACC_BUFS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < ACC_BUFS; ++a) {
      mbar_init(bar_accf + 8 * a, 1);
      mbar_init(bar_acce + 8 * a, 128);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  const int num_tiles = tiles_m * tiles_n;
  const int KB = (K + kBK - 1) / kBK;
  const int KG = K / kMmaK;           // scale atoms per 128-row band
  const int bands_n = (N + 127) / 128;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      // The first STAGES stages' B (weight) copies go out before waiting for the
      // previous grid in the stream (programmatic launch); their A copies, which
      // that grid may produce, are deferred until after the wait.
      DeferredA<STAGES> dfr;
      auto load_a = [&](int st, int kb, int mb, int nk) {
        const uint32_t fb = bar_full + 8 * st;
        tma_load_2d(sbase + C::kOffA + st * C::kABytes, &tmA, fb, kb * kBKBytes, mb * kBM, pol);
        bulk_load(sbase + C::kOffSFA + st * C::kSFABytes, SFA + (static_cast<size_t>(mb) * KG + kb * kKSteps) * kAtom,
                  nk * kAtom, fb, pol);
      };
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, tiles_m, tiles_n, group_n, mb, nb);
        int nbv = 0;
#pragma unroll
        for (int b = 0; b < C::kBands; ++b) nbv += (nb * C::kBands + b < bands_n) ? 1 : 0;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (dfr.full()) dfr.flush(load_a);
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag)) { ok = false; break; }
          const int nk = min(kKSteps, KG - kb * kKSteps);
          const uint32_t bytes = C::kABytes + C::kBBytes + nk * kAtom * (1 + nbv);
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, bytes);
          tma_load_2d(sbase + C::kOffB + stage * C::kBBytes, &tmB, fb, (kb >> b_shift) * kBKBytes, nb * BN, pol);
          for (int b = 0; b < nbv; ++b)
            bulk_load(sbase + C::kOffSFB + stage * C::kSFBBytes + b * kKSteps * kAtom,
                      SFB + (static_cast<size_t>(nb * C::kBands + b) * (KG >> b_shift) + (kb >> b_shift) * kKSteps) *
                                kAtom,
                      nk * kAtom, fb, pol);
          if (dfr.done) load_a(stage, kb, mb, nk); else dfr.add(stage, kb, mb, nk);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      if (!dfr.done) dfr.flush(load_a);
      // After an abort, wait (briefly, bounded) for the copies still in flight
      // before the thread block releases its shared memory.
      if (*abort_flag) {
        for (int i = 0; i < STAGES && issued > 0; ++i) {
          --issued;
          if (--stage < 0) { stage = STAGES - 1; phase ^= 1; }
          mbar_wait_for(bar_full + 8 * stage, phase, 10000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop on warp-uniform values (barrier waits by vote) and
    // lane 0, elected in each instruction, issues the scale copies and the MMAs.
    {
      griddep_wait();  // time-limited waits start once the previous grid is done
      constexpr uint32_t idesc = idesc_nvf4_m128<BN>();
      const uint32_t tm = warp_uniform(tmem);
      const uint32_t sb = warp_uniform(sbase);
      const uint32_t u_full = sb + (bar_full - sbase), u_empty = sb + (bar_empty - sbase);
      const uint32_t u_accf = sb + (bar_accf - sbase), u_acce = sb + (bar_acce - sbase);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        if (!warp_wait_vote(u_acce + 8 * acc, acc_phase ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tm + acc * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!warp_wait_vote(u_full + 8 * stage, phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const int nk = min(kKSteps, KG - kb * kKSteps);
          const uint32_t sfa_t = tm + C::kTmemSF + stage * (C::kSFACols + C::kSFBCols);
          const uint32_t sfb_t = sfa_t + C::kSFACols;
          const uint32_t sA = sb + C::kOffA + stage * C::kABytes;
          const uint32_t sB = sb + C::kOffB + stage * C::kBBytes;
          const uint32_t sSFA = sb + C::kOffSFA + stage * C::kSFABytes;
          const uint32_t sSFB = sb + C::kOffSFB + stage * C::kSFBBytes;
          for (int j = 0; j < nk; ++j) {
            tc_cp_32x128b_warpx4_elect(sfa_t + 4 * j, make_sdesc(sSFA + j * kAtom, 0, 128, 0));
#pragma unroll
            for (int b = 0; b < C::kBands; ++b)
              tc_cp_32x128b_warpx4_elect(sfb_t + 4 * (j * C::kBands + b),
                                         make_sdesc(sSFB + (b * kKSteps + j) * kAtom, 0, 128, 0));
          }
          for (int j = 0; j < nk; ++j) {
            const uint64_t adesc = make_sdesc(sA + j * (kMmaK / 2), 16, 1024, 2);
            const uint64_t bdesc = make_sdesc(sB + j * (kMmaK / 2), 16, 1024, 2);
            tc_mma_nvf4_elect(d_tmem, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + 4 * j * C::kBands,
                              (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit_elect(u_empty + 8 * stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_elect(u_accf + 8 * acc);
        if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    griddep_wait();
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, tiles_m, tiles_n, group_n, mb, nb);
      if (!warp_wait(bar_accf + 8 * acc, acc_phase, abort_flag)) break;
      tc_fence_after();
      const int row = mb * kBM + q * 32 + lane;
      const uint32_t t_base = tmem + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tc_ld_32x32b_x32(t_base + c * 32, v);
        tc_wait_ld();
        const int col0 = nb * BN + c * 32;
        if (row < M && col0 < N) {
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p[i] = pack_bf16x2(alpha * __uint_as_float(v[2 * i]), alpha * __uint_as_float(v[2 * i + 1]));
          uint4* dst = reinterpret_cast<uint4*>(D + static_cast<size_t>(row) * N + col0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (col0 + 8 * i < N) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar_acce + 8 * acc);
      if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}


// ------------------------------------------------------------------ split-K kernel
//
// For shapes whose output tiles cannot fill the SMs (few tokens: M = 128 against
// 5120..17408 weight rows gives 20..68 tiles of 128 x 256 for 152 SMs), K is split
// over a thread block cluster of S CTAs (S <= 8).  Every CTA of the cluster computes
// the same 128 x BN tile over a contiguous range of the K blocks, with the
// producer / MMA / epilogue roles of gemm_nvf4_kernel.  Its epilogue warps park the
// FP32 partial tile in the CTA's own shared memory (the drained operand ring), and
// after a cluster barrier CTA r finalises rows [128 r / S, 128 (r + 1) / S) of the
// tile: it reads the S partials through distributed shared memory, adds them in
// rank order (a fixed order: repeated calls are bit-identical), multiplies by alpha
// and stores BF16.  No global workspace is involved.
//
// Partial-tile layout: row r (TMEM lane) holds BN floats as BN/4 16-byte chunks;
// chunk c sits at position c ^ (r % 8), so the eight rows written by one phase of a
// warp's 16-byte stores fall in different banks.
// Twelve warps: producer, MMA issuer, then ten more that wait for the accumulator.
// Eight of them (two per TMEM lane quarter) push the partial tile; all twelve sum the
// owned columns.  The extra warps are there for latency hiding in those two phases,
// which are short dependent chains per warp.
constexpr int kSplitThreads = 384;

template <int BN, int STAGES>
__global__ void __launch_bounds__(kSplitThreads, 1)
    gemm_nvf4_splitk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const uint8_t* __restrict__ SFA, const uint8_t* __restrict__ SFB,
                            __nv_bfloat16* __restrict__ D, float alpha, int M, int N, int K, int S, int b_shift) {
  using C = Cfg<BN, STAGES, 1>;
  // The receive slots (at most S x 128 rows x (ceil(BN/8 / S) x 32 + 16) bytes, largest
  // for S = 6 or 7) fit in the drained operand ring, below the per-unit table at its end.
  static_assert(6 * 128 * (((BN / 8 + 5) / 6) * 32 + 16) + 8 * (BN / 8) <= C::kOffBar &&
                    7 * 128 * (((BN / 8 + 6) / 7) * 32 + 16) + 8 * (BN / 8) <= C::kOffBar &&
                    8 * 128 * (((BN / 8 + 7) / 8) * 32 + 16) + 8 * (BN / 8) <= C::kOffBar &&
                    5 * 128 * (((BN / 8 + 4) / 5) * 32 + 16) + 8 * (BN / 8) <= C::kOffBar,
                "partial-sum slots fit in the operand ring");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::kOffBar;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_accf = bar_empty + 8 * STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = blockIdx.x;  // the cluster spans gridDim.x == S CTAs: rank == blockIdx.x
  const int nb = blockIdx.y;
  const int mb = blockIdx.z;
  const int KB = (K + kBK - 1) / kBK;
  const int kb0 = rank * KB / S, kb1 = (rank + 1) * KB / S;
  const int KG = K / kMmaK;
  const int bands_n = (N + 127) / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_accf, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_normal();
      int nbv = 0;
#pragma unroll
      for (int b = 0; b < C::kBands; ++b) nbv += (nb * C::kBands + b < bands_n) ? 1 : 0;
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      DeferredA<STAGES> dfr;  // B first, A after the grid dependency (see gemm_nvf4_kernel)
      auto load_a = [&](int st, int kb, int m, int nk) {
        const uint32_t fb = bar_full + 8 * st;
        tma_load_2d(sbase + C::kOffA + st * C::kABytes, &tmA, fb, kb * kBKBytes, m * kBM, pol);
        bulk_load(sbase + C::kOffSFA + st * C::kSFABytes, SFA + (static_cast<size_t>(m) * KG + kb * kKSteps) * kAtom,
                  nk * kAtom, fb, pol);
      };
      for (int kb = kb0; kb < kb1; ++kb) {
        if (dfr.full()) dfr.flush(load_a);
        if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag)) break;
        const int nk = min(kKSteps, KG - kb * kKSteps);
        const uint32_t fb = bar_full + 8 * stage;
        mbar_arrive_expect_tx(fb, C::kABytes + C::kBBytes + nk * kAtom * (1 + nbv));
        tma_load_2d(sbase + C::kOffB + stage * C::kBBytes, &tmB, fb, (kb >> b_shift) * kBKBytes, nb * BN, pol);
        for (int b = 0; b < nbv; ++b)
          bulk_load(sbase + C::kOffSFB + stage * C::kSFBBytes + b * kKSteps * kAtom,
                    SFB + (static_cast<size_t>(nb * C::kBands + b) * (KG >> b_shift) + (kb >> b_shift) * kKSteps) *
                              kAtom,
                    nk * kAtom, fb, pol);
        if (dfr.done) load_a(stage, kb, mb, nk); else dfr.add(stage, kb, mb, nk);
        ++issued;
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      if (!dfr.done) dfr.flush(load_a);
      if (*abort_flag) {
        for (int i = 0; i < STAGES && issued > 0; ++i) {
          --issued;
          if (--stage < 0) { stage = STAGES - 1; phase ^= 1; }
          mbar_wait_for(bar_full + 8 * stage, phase, 10000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Whole warp, warp-uniform values, barrier waits by vote, lane 0 elected to issue.
    {
      griddep_wait();
      constexpr uint32_t idesc = idesc_nvf4_m128<BN>();
      const uint32_t tm = warp_uniform(tmem);
      const uint32_t sb = warp_uniform(sbase);
      const uint32_t u_full = sb + (bar_full - sbase), u_empty = sb + (bar_empty - sbase);
      const uint32_t u_accf = sb + (bar_accf - sbase);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!warp_wait_vote(u_full + 8 * stage, phase, abort_flag)) break;
        tc_fence_after();
        const int nk = min(kKSteps, KG - kb * kKSteps);
        const uint32_t sfa_t = tm + C::kTmemSF + stage * (C::kSFACols + C::kSFBCols);
        const uint32_t sfb_t = sfa_t + C::kSFACols;
        const uint32_t sA = sb + C::kOffA + stage * C::kABytes;
        const uint32_t sB = sb + C::kOffB + stage * C::kBBytes;
        const uint32_t sSFA = sb + C::kOffSFA + stage * C::kSFABytes;
        const uint32_t sSFB = sb + C::kOffSFB + stage * C::kSFBBytes;
        for (int j = 0; j < nk; ++j) {
          tc_cp_32x128b_warpx4_elect(sfa_t + 4 * j, make_sdesc(sSFA + j * kAtom, 0, 128, 0));
#pragma unroll
          for (int b = 0; b < C::kBands; ++b)
            tc_cp_32x128b_warpx4_elect(sfb_t + 4 * (j * C::kBands + b),
                                       make_sdesc(sSFB + (b * kKSteps + j) * kAtom, 0, 128, 0));
        }
        for (int j = 0; j < nk; ++j) {
          const uint64_t adesc = make_sdesc(sA + j * (kMmaK / 2), 16, 1024, 2);
          const uint64_t bdesc = make_sdesc(sB + j * (kMmaK / 2), 16, 1024, 2);
          tc_mma_nvf4_elect(tm, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + 4 * j * C::kBands,
                            (kb != kb0 || j != 0) ? 1u : 0u);
        }
        tc_commit_elect(u_empty + 8 * stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      tc_commit_elect(u_accf);  // also when the loop gave up: lets the epilogue proceed
    }
  } else {
    griddep_wait();
    warp_wait(bar_accf, 0, abort_flag);  // (gives up only together with the other roles)
  }

  // ------------------------------------------------------------ push the partial tile to its owners
  // The tile's columns form nu = BN/8 units of 8; CTA k owns units [k nu / S, (k+1) nu / S).
  // Owner k receives, in its ring, one slot per source rank: 128 rows x (its units x 8)
  // FP32, rows padded by 16 bytes (so the eight rows written by one phase of 16-byte
  // stores fall in different banks).  The stores are posted (no round trip).  A small
  // table (per unit: the shared::cluster address of row 0 of this CTA's slot at the
  // owner, and the owner's row pitch) is filled first, so the push loop itself does
  // no division.
  constexpr int kNu = BN / 8;

  // Every CTA's accumulator is complete (and its operand ring drained) past this
  // barrier, so the rings can receive the partial sums (and hold the table).
  tc_fence_before();
  __syncwarp();
  griddep_wait();  // D may still be written by the previous grid in the stream
  cluster_sync_all();
  tc_fence_after();

  uint32_t* unit_tab = reinterpret_cast<uint32_t*>(smem + C::kOffBar - 2 * 4 * kNu);
  if (threadIdx.x < kNu) {
    const int u = threadIdx.x;
    const int k = ((u + 1) * S - 1) / kNu;  // owner of unit u
    const int u0 = k * kNu / S, uk = (k + 1) * kNu / S - u0;
    const uint32_t pitch = static_cast<uint32_t>(uk * 32 + 16);
    const uint32_t off = static_cast<uint32_t>(rank) * 128u * pitch + static_cast<uint32_t>(u - u0) * 32u;
    unit_tab[2 * u] = map_to_rank(sbase + off, static_cast<uint32_t>(k));
    unit_tab[2 * u + 1] = pitch;
  }
  __syncthreads();

  if (warp >= 2 && warp < 10) {
    const int q = warp & 3;                 // TMEM lane quarter
    const int half = (warp - 2) >> 2;       // which half of the columns
    const uint32_t r = static_cast<uint32_t>(q * 32 + lane);
    const uint32_t t_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
    for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
      uint32_t v[32];
      tc_ld_32x32b_x32(t_base + c * 32, v);
      tc_wait_ld();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t dst = unit_tab[2 * (4 * c + i)] + r * unit_tab[2 * (4 * c + i) + 1];
        asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v[8 * i]),
                     "r"(v[8 * i + 1]), "r"(v[8 * i + 2]), "r"(v[8 * i + 3])
                     : "memory");
        asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 16), "r"(v[8 * i + 4]),
                     "r"(v[8 * i + 5]), "r"(v[8 * i + 6]), "r"(v[8 * i + 7])
                     : "memory");
      }
    }
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();  // every partial has landed at its owner

  // ------------------------------------------------------------ fixed-order sum of the owned columns
  // Item = one row x one 8-column unit (two 16-byte chunks per slot, one 16-byte
  // BF16 store); each thread takes two items at a time so their loads overlap.
  {
    const int u0 = rank * kNu / S, uk = (rank + 1) * kNu / S - u0;
    const uint32_t pitch = static_cast<uint32_t>(uk * 32 + 16);
    const uint32_t slot = 128u * pitch;
    const int items = 128 * uk;
    const int gcol0 = nb * BN + u0 * 8;
    for (int base = threadIdx.x; base < items; base += 2 * kSplitThreads) {
      float a[2][8];
      int row[2], un[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int idx = base + h * kSplitThreads;
        row[h] = idx / uk;  // uk is small; one division per item
        un[h] = idx - row[h] * uk;
#pragma unroll
        for (int e = 0; e < 8; ++e) a[h][e] = 0.f;
        if (idx < items) {
          const uint32_t off = sbase + static_cast<uint32_t>(row[h]) * pitch + static_cast<uint32_t>(un[h]) * 32u;
#pragma unroll 1
          for (int s = 0; s < S; ++s) {
            float4 lo, hi;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(lo.x), "=f"(lo.y), "=f"(lo.z), "=f"(lo.w)
                         : "r"(off + static_cast<uint32_t>(s) * slot));
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(hi.x), "=f"(hi.y), "=f"(hi.z), "=f"(hi.w)
                         : "r"(off + static_cast<uint32_t>(s) * slot + 16u));
            a[h][0] += lo.x; a[h][1] += lo.y; a[h][2] += lo.z; a[h][3] += lo.w;
            a[h][4] += hi.x; a[h][5] += hi.y; a[h][6] += hi.z; a[h][7] += hi.w;
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int idx = base + h * kSplitThreads;
        const int grow = mb * kBM + row[h];
        const int gcol = gcol0 + un[h] * 8;
        if (idx < items && grow < M && gcol < N)
          *reinterpret_cast<uint4*>(D + static_cast<size_t>(grow) * N + gcol) =
              make_uint4(pack_bf16x2(alpha * a[h][0], alpha * a[h][1]), pack_bf16x2(alpha * a[h][2], alpha * a[h][3]),
                         pack_bf16x2(alpha * a[h][4], alpha * a[h][5]), pack_bf16x2(alpha * a[h][6], alpha * a[h][7]));
      }
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ CTA-pair kernel
//
// One pair of CTAs (a cluster of 2) computes a 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 64 per instruction).  Each CTA
// stages its own 128 rows of A and its own 128 rows of B.
//
// Operand delivery: four stages of K = 256; per stage A and B arrive as one 16 KB
// box each (128 rows x 128 bytes, 128-byte swizzle), the scale atoms as one SFA box
// (4 atoms, 2 KB) and one SFB box (4 atoms of each of the tile's two bands, 4 KB).
// All of both CTAs' copies complete on the leader's "full" barrier.
//
// What bounds the tensor pipe here (measured on GB300 with MMA-only loops): one
// 256 x 256 x 64 MMA occupies each SM of the pair for 128 cycles (16384 FP4 MACs per
// SM per cycle, 4x the BF16 rate), and a stage needs 12 tcgen05.cp of 512-byte scale
// atoms besides its 4 MMAs.  How fast a warp can issue them depends on how the code
// is written: a lone lane with operands the compiler cannot prove warp-uniform issues
// one copy per ~64 cycles (~128 while MMAs run), a converged warp with warp-uniform
// operands and elect.sync one per ~29 cycles.  So the MMA warp and the copy warps run
// their loops as whole warps (values broadcast from lane 0, barrier waits by vote,
// lane 0 elected in each tcgen05 instruction); this took the kernel from 193 to
// 175 us at 8192^3.  The copies are spread over six warps, placed on the three
// sub-partitions that do not hold the MMA warp, two copies per warp per stage (three
// warps with four copies each measured 224 us).  They are ordered before the stage's
// MMAs without waiting for their completion: each copy warp issues its copies,
// executes tcgen05.fence::before_thread_sync and arrives on the stage's "sf"
// barrier; the MMA warp waits for it and executes tcgen05.fence::after_thread_sync
// before its MMAs, which places the MMAs after the copies in the tensor pipe.  The
// MMA warp then issues the stage's four MMAs from precomputed descriptors and
// releases the stage to both CTAs with a multicast commit.  Eight epilogue warps per
// CTA drain the accumulator (128 lanes x 256 columns) into a 128-byte-swizzled BF16
// staging tile, loading the next 32-column chunk from TMEM while converting the
// current one; the accumulator is released as soon as the last chunk is in
// registers (it is single-buffered: two 256-column accumulators would leave no TMEM
// columns for the scale slots), and D goes out with TMA stores.
//
// Tile schedules: static (pair p takes tiles p, p + P, ... of the grouped raster),
// stream-K (pair_sched.h), or cluster launch control (Colfax Research's SM120 NVFP4
// GEMM article, Appendix): the grid holds one cluster per tile, a running pair starts
// with its own tile and then cancels pending clusters and takes theirs.  Warp 13 (otherwise idle) of the leader issues
// clusterlaunchcontrol.try_cancel with the response multicast to both CTAs into a
// two-slot ring once every consuming role (27 warps or threads over the pair) has
// read the slot's previous response; the follower's warp 13 arms its own barrier for
// each response.  Measured on GB300 against the static schedule: no gain (8192^3
// 177.9 against 172.7 us; 1024 x 5120 x 17408 59.1 against 58.0), so it is an
// explicit configuration, not the automatic choice.
namespace pair {

constexpr int kStages = 5;
constexpr int kBKP = 256;                        // K per stage
constexpr int kStepsP = kBKP / kMmaK;            // 4 MMAs per stage
constexpr int kEpiWarps = 8;
constexpr int kFirstEpiWarp = 2;
constexpr int kSFWarp = kFirstEpiWarp + kEpiWarps;  // first of the warps issuing the scale copies
constexpr int kSFWarps = 6;                         // warps 10, 11, 12, 14, 15, 16 (not sub-partition 1)
constexpr int kSFCopies = 3 * kStepsP;              // per stage: SFA, SFB band 0, SFB band 1 per MMA
constexpr int kAWarp = kSFWarp + kSFWarps + (kSFWarps - 1) / 3 + 1;  // 18: the A producer (sub-partition 2)
constexpr int kNumWarps = kAWarp + 1;
constexpr int kThreads = 32 * kNumWarps;
// Copy-warp index of warp `w` (>= kSFWarp): the warps whose id is 1 mod 4 share the
// MMA warp's sub-partition and issue no copies (-1).
__host__ __device__ constexpr int sf_warp_index(int w) {
  return (w & 3) == 1 ? -1 : w - kSFWarp - (w - kSFWarp) / 4;
}
static_assert(sf_warp_index(kAWarp - 2) == kSFWarps - 1 && (kAWarp & 3) == 2, "warp roles");
constexpr int kABytes = 128 * (kBKP / 2);        // 16 KB: 128 rows x 128 B
constexpr int kBBytes = 128 * (kBKP / 2);        // 16 KB
constexpr int kSubTile = 128 * 128;              // 16 KB
constexpr int kSFABytes = kStepsP * kAtom;       // 2 KB
constexpr int kSFBBytes = 2 * kStepsP * kAtom;   // 4 KB: [band][atom]
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffSFA = kOffB + kStages * kBBytes;
constexpr int kOffSFB = kOffSFA + kStages * kSFABytes;
constexpr int kOffOut = kOffSFB + kStages * kSFBBytes;  // 2 boxes of 128 rows x 128 B (64 bf16 columns)
constexpr int kOutBox = 128 * 128;
constexpr int kOffBar = kOffOut + 2 * kOutBox;
constexpr int kClcSlots = 2;          // CLC response ring
constexpr int kClcConsumers = 17 + 10; // leader: 2 producers, MMA, 6 copy, 8 epilogue warps; follower: 2 + 8
constexpr int kNumBars = 4 * kStages + 5 + 2 * kClcSlots;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffResp = (kOffMisc + 16 + 15) / 16 * 16;
constexpr int kSmemBytes = kOffResp + 16 * kClcSlots + 1024;
static_assert(kOffOut % 1024 == 0 && kOffB % 1024 == 0, "swizzled tiles must be 1024-byte aligned");
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr int kTmemCols = 512;
constexpr int kSFACols = kStepsP * 4;   // MMA j reads SFA columns [4j, 4j + 4)
constexpr int kSFBCols = kStepsP * 8;   // MMA j reads SFB columns [8j, 8j + 8) (band 0 then band 1)
constexpr int kSFSlotCols = kSFACols + kSFBCols;
constexpr int kTmemSF = 256;
static_assert(kTmemSF + kStages * kSFSlotCols <= kTmemCols, "TMEM budget");

constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(256 >> 3) << 17) |
                            (static_cast<uint32_t>(256 >> 4) << 24);

// The pair schedule is in pair_sched.h, shared with a host-side test.
using ::nvfp4::sched::PairSched;

// Fault injection for tests (off unless nvfp4_test_streamk_fault turns it on): the
// head pairs of the stream-K schedule skip publishing their partials, and the flag
// waits give up after g_flag_wait_ns, so that a test can make those waits run out and
// check the timeout path without faulting or hanging anything.
__device__ int g_test_skip_publish = 0;
__device__ unsigned long long g_flag_wait_ns = kWaitLimitNs;

// Bounded wait (2 s unless a test shortened it) for a stream-K flag to read 1
// (acquire, GPU scope).
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, volatile int* abort) {
  const uint64_t limit = g_flag_wait_ns;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v == 1u) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit) {
      *abort = 1;
      record_device_error(kDevErrTimeout);
      return false;
    }
  }
}

// SK: the stream-K schedule is compiled in (the data-parallel instantiation carries
// none of its code or registers).
template <bool SK, bool CLC = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                          const __grid_constant__ CUtensorMap tmD, float alpha, int K, int tiles_m, int tiles_n,
                          int group_n, float* __restrict__ ws, uint32_t* __restrict__ flags, int b_shift) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + kOffBar;             // both CTAs' A and B bytes (leader's copy is used)
  const uint32_t bar_empty = bar_full + 8 * kStages;     // stage released by the MMAs (both CTAs)
  const uint32_t bar_accf = bar_empty + 8 * kStages;
  const uint32_t bar_acce = bar_accf + 8;
  const uint32_t bar_sf = bar_acce + 8;                 // stage's scales are in TMEM (leader)
  const uint32_t bar_pub = bar_sf + 8 * kStages;        // stream-K: this CTA's head partial is written
  const uint32_t bar_seen = bar_pub + 8;                // stream-K: the head partial of the tail is ready
  const uint32_t bar_fsf = bar_seen + 8;                // both CTAs' scale atoms of the stage (leader's copy)
  const uint32_t bar_drain = bar_fsf + 8 * kStages;     // every tcgen05 op of the launch has completed
  const uint32_t bar_clcf = bar_drain + 8;              // CLC response of a ring slot has landed
  const uint32_t bar_clce = bar_clcf + 8 * kClcSlots;   // every consumer has read it (leader's copy is used)
  const uint32_t resp0 = sbase + kOffResp;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_id = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_accf, 1);
    mbar_init(bar_acce, 2 * kEpiWarps);
    for (int s = 0; s < kStages; ++s) mbar_init(bar_fsf + 8 * s, 1);
    mbar_init(bar_drain, 1 + kSFWarps);  // the MMA thread and the copy warps, once each
    for (int s = 0; s < kStages; ++s) mbar_init(bar_sf + 8 * s, kSFWarps);
    mbar_init(bar_pub, kEpiWarps);  // each used at most once per launch (phase 0)
    mbar_init(bar_seen, 1);
    for (int s = 0; s < kClcSlots; ++s) {
      mbar_init(bar_clcf + 8 * s, 1);
      mbar_init(bar_clce + 8 * s, kClcConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmSFA);
    prefetch_tensormap(&tmSFB);
    prefetch_tensormap(&tmD);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  const int num_tiles = tiles_m * tiles_n;
  const int KB = (K + kBKP - 1) / kBKP;
  const int KG = K / kMmaK;  // scale atoms per 128-row band
  PairSched sched;
  sched.init(pair_id, num_pairs, num_tiles, KB, SK ? 1 : 0);
  const int nseg = sched.count();

  // Tile i of this pair's sequence: the static schedule, or (CLC) the pair's own tile
  // and then the tiles of the clusters it cancelled.  Every consuming role reads each
  // CLC response once, in order, and releases its ring slot.
  auto clc_query = [&](uint32_t addr, int& tile) -> bool {
    uint32_t ok = 0;
    asm volatile(
        "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
        "ld.shared.b128 r, [%1];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr)
        : "memory");
    if (ok) {
      uint32_t x;
      asm volatile(
          "{\n\t.reg .b128 r;\n\t"
          "ld.shared.b128 r, [%1];\n\t"
          "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, r;\n\t}"
          : "=r"(x)
          : "r"(addr)
          : "memory");
      tile = static_cast<int>(x >> 1);
    }
    return ok != 0;
  };
  auto clc_next = [&](int i, bool warp_wide) -> int {
    const int slot = i & (kClcSlots - 1);
    const uint32_t ph = static_cast<uint32_t>(i / kClcSlots) & 1u;
    const bool got = warp_wide ? warp_wait_vote<true>(bar_clcf + 8 * slot, ph, abort_flag)
                               : mbar_wait_spin<true>(bar_clcf + 8 * slot, ph, abort_flag);
    int t = -1;
    if (got && !clc_query(resp0 + 16 * slot, t)) t = -1;
    if (warp_wide) __syncwarp();
    if (!warp_wide || lane == 0) {
      if (leader) mbar_arrive(bar_clce + 8 * slot);
      else mbar_arrive_cluster(map_to_rank(bar_clce + 8 * slot, 0));
    }
    return t;
  };
  auto next_seg = [&](int s, int& t, int& kb0, int& kb1, int& kind, bool warp_wide) -> bool {
    if (!CLC) {
      if (s >= nseg) return false;
      sched.template seg<SK>(s, t, kb0, kb1, kind);
      return true;
    }
    t = s == 0 ? static_cast<int>(blockIdx.x >> 1) : clc_next(s - 1, warp_wide);
    kb0 = 0;
    kb1 = KB;
    kind = PairSched::kFull;
    return t >= 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer of B (both CTAs)
    // Issuing a tiled TMA load takes the issuing thread ~140 cycles, so one thread
    // cannot issue a stage's four loads in the 512 cycles its MMAs take: this warp
    // issues the weight side (B, SFB) and arms the stage's full barrier, warp kAWarp
    // the activation side (A, SFA).  The weight loads may be issued before the
    // previous grid in the stream has completed (programmatic launch).
    if (lane == 0) {
      const uint32_t full_leader = map_to_rank(bar_full, 0);
      const uint32_t fsf_leader = map_to_rank(bar_fsf, 0);
      // The operands (A, B and their scales, read by many tiles) are kept in L2 ahead
      // of D, which streams out once.
      const uint64_t keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int issued = 0;
      for (int s = 0; ok; ++s) {
        int t, kb0, kb1, kind;
        if (!next_seg(s, t, kb0, kb1, kind, false)) break;
        int mt, nt;
        tile_coords(t, tiles_m, tiles_n, group_n, mt, nt);
        const int b_row = nt * 256 + static_cast<int>(rank) * 128;
        for (int kb = kb0; kb < kb1; ++kb) {
          // The first kStages stages are free; the wait for the next one can only end
          // after the MMAs, which wait for the previous grid: wait for it here too, so
          // that the time limit counts from its completion.
          if (++issued == kStages + 1) griddep_wait();
          if (!mbar_wait_spin<true>(bar_empty + 8 * stage, phase ^ 1, abort_flag)) { ok = false; break; }
          // The scale atoms complete on their own barrier and go first, so that the
          // scale copies into TMEM overlap the arrival of the A and B tiles.
          if (leader) {
            mbar_arrive_expect_tx(bar_fsf + 8 * stage, 2 * (kSFABytes + kSFBBytes));
            mbar_arrive_expect_tx(bar_full + 8 * stage, 2 * (kABytes + kBBytes));
          }
          tma_load_3d_pair_hint(sbase + kOffSFB + stage * kSFBBytes, &tmSFB, fsf_leader + 8 * stage, 0,
                                (kb >> b_shift) * kStepsP, nt * 2, keep);
          tma_load_3d_pair_hint(sbase + kOffB + stage * kBBytes, &tmB, full_leader + 8 * stage, 0, b_row,
                                (kBKP / 256) * (kb >> b_shift), keep);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      // Drain: wait until every stage has been released once more, so that no commit
      // arrival (and no copy of this CTA) is still in flight when the CTA exits.
      if (issued <= kStages) griddep_wait();
      for (int i = 0; i < kStages && !*abort_flag; ++i) {
        if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag)) break;
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (*abort_flag && leader) {
        for (int i = 0; i < kStages; ++i) {
          mbar_wait_for(bar_full + 8 * i, 0, 10000000ull);
          mbar_wait_for(bar_fsf + 8 * i, 0, 10000000ull);
        }
      }
    }
  } else if (warp == kAWarp) {
    // ------------------------------------------------------------ TMA producer of A (both CTAs)
    // The activations may be written by the previous grid in the stream: wait for it.
    if (lane == 0) {
      griddep_wait();
      const uint32_t full_leader = map_to_rank(bar_full, 0);
      const uint32_t fsf_leader = map_to_rank(bar_fsf, 0);
      const uint64_t keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int s = 0; ok; ++s) {
        int t, kb0, kb1, kind;
        if (!next_seg(s, t, kb0, kb1, kind, false)) break;
        int mt, nt;
        tile_coords(t, tiles_m, tiles_n, group_n, mt, nt);
        const int a_row = mt * 256 + static_cast<int>(rank) * 128;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_spin<true>(bar_empty + 8 * stage, phase ^ 1, abort_flag)) { ok = false; break; }
          tma_load_3d_pair_hint(sbase + kOffSFA + stage * kSFABytes, &tmSFA, fsf_leader + 8 * stage, 0, kb * kStepsP,
                                mt * 2 + static_cast<int>(rank), keep);
          tma_load_3d_pair_hint(sbase + kOffA + stage * kABytes, &tmA, full_leader + 8 * stage, 0, a_row,
                                (kBKP / 256) * kb, keep);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    // The whole warp runs the loop on warp-uniform values (barrier waits by vote) and
    // lane 0, elected in each instruction, issues.
    if (leader) {
      griddep_wait();  // time-limited waits start once the previous grid is done
      const uint32_t tm = warp_uniform(tmem);
      const uint32_t sb = warp_uniform(sbase);
      // (each barrier address rebased on the uniform shared-memory base)
      const uint32_t u_full = sb + (bar_full - sbase), u_empty = sb + (bar_empty - sbase);
      const uint32_t u_accf = sb + (bar_accf - sbase), u_acce = sb + (bar_acce - sbase);
      const uint32_t u_sf = sb + (bar_sf - sbase), u_drain = sb + (bar_drain - sbase);
      // Descriptors of stage 0, K-step 0; stage s, K-step j adds s * 16 KB + j * 32 bytes
      // to the start address (16-byte units in the low bits).
      const uint64_t adesc0 = make_sdesc(sb + kOffA, 16, 1024, 2);
      const uint64_t bdesc0 = make_sdesc(sb + kOffB, 16, 1024, 2);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int s = 0; ok; ++s) {
        int t, kb0, kb1, kind;
        if (!next_seg(s, t, kb0, kb1, kind, true)) break;
        if (!warp_wait_vote<true>(u_acce, acc_phase ^ 1, abort_flag)) break;
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb) {
          // The copy warps arrive only after the stage's operands landed (they wait
          // for its full barrier) and their scale copies were issued.
          if (!warp_wait_vote(u_sf + 8 * stage, phase, abort_flag)) { ok = false; break; }
          if (!warp_wait_vote<true>(u_full + 8 * stage, phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sf_t = tm + kTmemSF + stage * kSFSlotCols;
          const uint64_t ad = adesc0 + static_cast<uint64_t>(stage * (kABytes >> 4));
          const uint64_t bd = bdesc0 + static_cast<uint64_t>(stage * (kBBytes >> 4));
          if (KG - kb * kStepsP >= kStepsP) {
            tc_mma_nvf4_pair_elect(tm, ad, bd, kIdesc, sf_t, sf_t + kSFACols, kb != kb0 ? 1u : 0u);
#pragma unroll
            for (int j = 1; j < kStepsP; ++j)
              tc_mma_nvf4_pair_elect(tm, ad + 2 * j, bd + 2 * j, kIdesc, sf_t + 4 * j, sf_t + kSFACols + 8 * j, 1u);
          } else {
            const int nk = KG - kb * kStepsP;
            for (int j = 0; j < nk; ++j)
              tc_mma_nvf4_pair_elect(tm, ad + 2 * j, bd + 2 * j, kIdesc, sf_t + 4 * j, sf_t + kSFACols + 8 * j,
                                     (kb != kb0 || j != 0) ? 1u : 0u);
          }
          tc_commit_pair_mc_elect(u_empty + 8 * stage, 0x3);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair_mc_elect(u_accf, 0x3);
        acc_phase ^= 1;
      }
      tc_commit_pair_mc_elect(u_drain, 0x3);  // see the teardown
    }
  } else if (warp >= kSFWarp) {
    // ------------------------------------------------------------ scale copies (leader CTA)
    // Move each landed stage's scale atoms into its TMEM slot (tcgen05.cp, both CTAs
    // of the pair) and signal the MMA issuer.  Copy c of a stage (0..11) is SFA of MMA
    // c (c < 4) or band (c / 4 - 1) of SFB of MMA c % 4; warp i takes the copies with
    // c % 6 == i.  The slot is free: the stage only refills (and its full barrier only
    // completes) after the MMAs that read the slot have committed.
    // The whole warp runs the loop on warp-uniform values; lane 0 issues (elected).
    const int cw = static_cast<int>(warp_uniform(static_cast<uint32_t>(sf_warp_index(warp))));
    if (CLC && warp == kSFWarp + 3) {
      // CLC scheduler: the leader cancels one pending cluster per ring slot once every
      // consumer has read the slot's previous response (multicast to both CTAs); the
      // follower arms its own barrier for each response.  Stops after a response that
      // cancelled nothing.
      if (lane == 0) {
        for (int i = 0;; ++i) {
          const int slot = i & (kClcSlots - 1);
          const uint32_t ph = static_cast<uint32_t>(i / kClcSlots) & 1u;
          if (leader && i >= kClcSlots && !mbar_wait_spin<true>(bar_clce + 8 * slot, ph ^ 1u, abort_flag)) break;
          mbar_arrive_expect_tx(bar_clcf + 8 * slot, 16);
          if (leader)
            asm volatile(
                "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.multicast::cluster::all.b128 [%0], [%1];" ::"r"(
                    resp0 + 16 * slot),
                "r"(bar_clcf + 8 * slot)
                : "memory");
          if (!mbar_wait_spin<true>(bar_clcf + 8 * slot, ph, abort_flag)) break;
          int t;
          if (!clc_query(resp0 + 16 * slot, t)) break;
        }
      }
    } else if (leader && cw >= 0) {
      griddep_wait();
      const uint32_t tm = warp_uniform(tmem);
      const uint32_t sb = warp_uniform(sbase);
      const uint32_t u_fsf = sb + (bar_fsf - sbase), u_sf = sb + (bar_sf - sbase);
      const uint32_t u_drain = sb + (bar_drain - sbase);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int s = 0; ok; ++s) {
        int t, kb0, kb1, kind;
        if (!next_seg(s, t, kb0, kb1, kind, true)) break;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!warp_wait_vote<true>(u_fsf + 8 * stage, phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const int nk = min(kStepsP, KG - kb * kStepsP);
          const uint32_t sf_t = tm + kTmemSF + stage * kSFSlotCols;
          const uint32_t sSFA = sb + kOffSFA + stage * kSFABytes;
          const uint32_t sSFB = sb + kOffSFB + stage * kSFBBytes;
#pragma unroll
          for (int c = cw; c < kSFCopies; c += kSFWarps) {
            const int j = c % kStepsP, k = c / kStepsP;
            if (j < nk) {
              if (k == 0)
                tc_cp_32x128b_warpx4_pair_elect(sf_t + 4 * j, make_sdesc(sSFA + j * kAtom, 0, 128, 0));
              else
                tc_cp_32x128b_warpx4_pair_elect(sf_t + kSFACols + 8 * j + 4 * (k - 1),
                                                make_sdesc(sSFB + ((k - 1) * kStepsP + j) * kAtom, 0, 128, 0));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(u_sf + 8 * stage);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      tc_commit_pair_mc_elect(u_drain, 0x3);  // see the teardown
    }
  } else {
    // ------------------------------------------------------------ epilogue (8 warps, both CTAs)
    griddep_wait();
    const int q = warp & 3;                        // TMEM lane quarter of this warp
    const int h = (warp - kFirstEpiWarp) >> 2;     // column half (0: columns 0..127, 1: 128..255)
    const uint32_t acce_leader = map_to_rank(bar_acce, 0);
    const uint32_t out_base = sbase + kOffOut;
    const uint64_t stream_out = policy_evict_first();
    const int r = q * 32 + lane;                   // accumulator row = TMEM lane
    uint32_t acc_phase = 0;
    bool stored = false;
    // Hand the accumulator back to the MMA issuer (every warp's TMEM loads have
    // completed: tcgen05.wait::ld).  The follower's warps arrive with relaxed
    // semantics: an arrival with release semantics at cluster scope waited ~700 ns
    // (measured) for the SM's memory traffic in flight, while the accumulator's
    // values are already in registers and nothing else needs ordering.
    auto release_acc = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(bar_acce);
        else mbar_arrive_relaxed_cluster(acce_leader);
      }
    };
    // Stream-K workspace slots: one 128 KB FP32 partial per (pair, rank) and one flag
    // each.  A slot is laid out in the epilogue's own register order, [warp][32-column
    // chunk][float4 i][lane], so that both the publishing and the finishing CTA (same
    // rank, hence the same TMEM lanes and warp roles) move it with whole 512-byte warp
    // accesses.
    const size_t slot_f4 = 128 * 256 / 4;
    const int ew = warp - kFirstEpiWarp;           // epilogue warp 0..7
    for (int s = 0;; ++s) {
      int t, kb0, kb1, kind;
      if (!next_seg(s, t, kb0, kb1, kind, true)) break;
      int mt, nt;
      tile_coords(t, tiles_m, tiles_n, group_n, mt, nt);
      const float4* part = nullptr;  // the head pair's partial of this tile (tail piece)
      float4 hp[8];                  // its current 32-column chunk
      if (SK && kind == PairSched::kTail) {
        // While this pair's own MMAs still run: one thread watches the flag, resets it
        // for the next call (the head pair publishes this slot once per launch) and
        // releases the other warps, which fetch their first chunk of the partial.
        uint32_t* flag = flags + (pair_id - 1) * 2 + rank;
        if (warp == kFirstEpiWarp && lane == 0 && wait_flag(flag, abort_flag)) {
          asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(0u) : "memory");
          mbar_arrive(bar_seen);
        }
        if (!warp_wait(bar_seen, 0, abort_flag)) break;
        part = reinterpret_cast<const float4*>(ws) + (static_cast<size_t>(pair_id - 1) * 2 + rank) * slot_f4 +
               static_cast<size_t>(ew) * (4 * 8 * 32) + lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) hp[i] = __ldcg(part + i * 32);
      }
      if (!warp_wait_vote<true>(bar_accf, acc_phase, abort_flag)) break;
      tc_fence_after();
      if (SK && kind == PairSched::kHead) {
        // ---- head piece: publish the FP32 partial tile for the pair that finishes it
        float4* dst = reinterpret_cast<float4*>(ws) + (static_cast<size_t>(pair_id) * 2 + rank) * slot_f4 +
                      static_cast<size_t>(ew) * (4 * 8 * 32) + lane;
#pragma unroll 1
        for (int c32 = 0; c32 < 4; ++c32) {
          const int col0 = h * 128 + c32 * 32;
          uint32_t v[32];
          tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + col0, v);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            __stcg(dst + (c32 * 8 + i) * 32, make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                         __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
        }
        // The accumulator is read out: hand it back before the stores drain.
        release_acc();
        __threadfence();  // this warp's stores are visible at GPU scope before its arrival
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pub);
        if (warp == kFirstEpiWarp && lane == 0 && mbar_wait(bar_pub, 0, abort_flag) && !g_test_skip_publish) {
          __threadfence();
          asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flags + pair_id * 2 + rank), "r"(1u) : "memory");
        }
        acc_phase ^= 1;
        continue;
      }
      if (stored) {  // the previous tile's stores must have finished reading the staging tile
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
      }
      // Drain the accumulator in four 32-column chunks, two TMEM loads per wait: the
      // first two chunks are converted and staged while nothing else is in flight, and
      // the accumulator goes back to the MMA issuer as soon as the last two are in
      // registers.
      const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * 128);
      auto stage_chunk = [&](uint32_t (&v)[32], int c32) {
        if (part != nullptr) {
          // fixed order: this pair's stages, then the head pair's partial (chunk 0's
          // partial was fetched while the MMAs ran)
          float4 hq[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) hq[i] = c32 == 0 ? hp[i] : __ldcg(part + (c32 * 8 + i) * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) + hq[i].x);
            v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + hq[i].y);
            v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + hq[i].z);
            v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + hq[i].w);
          }
        }
        const uint32_t box = out_base + h * kOutBox + r * 128;  // one box per column half, used twice
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c = (c32 & 1) * 4 + cc;   // 16-byte chunk (8 columns) within the 128-byte box row
          uint32_t p0 = pack_bf16x2(alpha * __uint_as_float(v[8 * cc + 0]), alpha * __uint_as_float(v[8 * cc + 1]));
          uint32_t p1 = pack_bf16x2(alpha * __uint_as_float(v[8 * cc + 2]), alpha * __uint_as_float(v[8 * cc + 3]));
          uint32_t p2 = pack_bf16x2(alpha * __uint_as_float(v[8 * cc + 4]), alpha * __uint_as_float(v[8 * cc + 5]));
          uint32_t p3 = pack_bf16x2(alpha * __uint_as_float(v[8 * cc + 6]), alpha * __uint_as_float(v[8 * cc + 7]));
          const uint32_t addr = box + ((c ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(p0), "r"(p1), "r"(p2), "r"(p3)
                       : "memory");
        }
      };
      // The staging box of a column half holds 64 columns: the first two chunks go out
      // with one TMA store while the last two are loaded, and are staged once that
      // store has read the box.
      const int row0 = mt * 256 + static_cast<int>(rank) * 128 + q * 32;
      const uint32_t box_rows = out_base + h * kOutBox + q * 32 * 128;
      uint32_t va[32], vb[32];
      if (part == nullptr) {
        // Two loads per wait (one TMEM round trip per 64 columns, measured 2 % faster
        // than one per chunk): chunks 0 and 1, staged, then chunks 2 and 3.
        tc_ld_32x32b_x32(trow, va);
        tc_ld_32x32b_x32(trow + 32, vb);
        tc_wait_ld(va);
        tc_bind(vb);
        stage_chunk(va, 0);
        stage_chunk(vb, 1);
        tc_ld_32x32b_x32(trow + 64, va);
        tc_ld_32x32b_x32(trow + 96, vb);
        tc_wait_ld(va);
        tc_bind(vb);
      } else {
        // stream-K tail: the head pair's partial is added chunk by chunk
        tc_ld_32x32b_x32(trow, va);
        tc_wait_ld(va);
        tc_ld_32x32b_x32(trow + 32, vb);
        stage_chunk(va, 0);
        tc_wait_ld(vb);
        tc_ld_32x32b_x32(trow + 64, va);
        stage_chunk(vb, 1);
        tc_wait_ld(va);
        tc_ld_32x32b_x32(trow + 96, vb);
        tc_wait_ld(vb);
      }
      // Accumulator read out: hand it back to the MMA issuer (before any store of this
      // tile is in flight: an arrival issued behind a TMA store was measured to reach
      // its waiter ~1 us late).
      release_acc();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d_hint(&tmD, box_rows, nt * 256 + h * 128, row0, stream_out);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
      __syncwarp();
      stage_chunk(va, 2);
      stage_chunk(vb, 3);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d_hint(&tmD, box_rows, nt * 256 + h * 128 + 64, row0, stream_out);
        bulk_commit_group();
      }
      stored = true;
      acc_phase ^= 1;
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  // Before TMEM is released and the CTAs exit, every MMA and scale copy issued in this
  // launch must have completed: the issuing threads' final commits arrive on both
  // CTAs' drain barrier.  In a normal run the epilogue has already waited for the last
  // MMAs; after a timed-out wait the roles stop early and this is what keeps the
  // tensor pipe from writing freed TMEM or reading a departed CTA's shared memory.
  if (threadIdx.x == 0) mbar_wait_for(bar_drain, 0, 200000000ull);
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace pair

// ------------------------------------------------------------------ host side

struct ConfigEntry {
  const char* name;
  int bn;
};

constexpr ConfigEntry kConfigs[] = {
    {"1cta_128x256_s3_acc1", 256},
    {"1cta_128x128_s4_acc2", 128},
    {"2cta_256x256_k256x4 (K % 256 == 0; other K run 1cta_128x256)", 256},
    {"1cta_128x256_splitk (K split over a cluster of up to 8 CTAs, fixed-order DSMEM reduction)", 256},
    {"1cta_128x128_splitk (K split over a cluster of up to 8 CTAs, fixed-order DSMEM reduction)", 128},
    {"2cta_256x256_k256x4_clc (CTA pairs, dynamic tile scheduling by cluster launch control)", 256},
};
constexpr int kNumConfigs = sizeof(kConfigs) / sizeof(kConfigs[0]);

// Programmatic dependent launch: the kernel may start while the previous kernel in
// the stream finishes; it streams its first weight stages and waits
// (griddepcontrol.wait) before it reads A or writes D.
inline void set_programmatic(cudaLaunchAttribute& a) {
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
}

template <int BN, int STAGES, int ACC_BUFS>
nvfp4_status run(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB, float alpha,
                 void* D, int64_t M, int64_t N, int64_t K, cudaStream_t stream, const DeviceInfo& dev,
                 int b_shift = 0) {
  using C = Cfg<BN, STAGES, ACC_BUFS>;
  auto kern = gemm_nvf4_kernel<BN, STAGES, ACC_BUFS>;
  static PerDeviceOnce smem_attr;
  if (!smem_attr.get(dev.device, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) == cudaSuccess;
      }))
    return NVFP4_ERR_CUDA;
  CUtensorMap ta, tb;
  nvfp4_status st = encode_tmap_u8_2d(&ta, A, K / 2, M, K / 2, kBKBytes, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != NVFP4_OK) return st;
  st = encode_tmap_u8_2d(&tb, B, (K >> b_shift) / 2, N, (K >> b_shift) / 2, kBKBytes, BN,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != NVFP4_OK) return st;
  const int tiles_m = static_cast<int>((M + kBM - 1) / kBM);
  const int tiles_n = static_cast<int>((N + BN - 1) / BN);
  const int num_tiles = tiles_m * tiles_n;
  const int grid = num_tiles < dev.num_sms ? num_tiles : dev.num_sms;
  const int group_n = tiles_n < 8 ? tiles_n : 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  set_programmatic(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return from_cuda(cudaLaunchKernelEx(&cfg, kern, ta, tb, SFA, SFB, static_cast<__nv_bfloat16*>(D), alpha,
                                      static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), tiles_m, tiles_n,
                                      group_n, b_shift));
}

// K split for a shape.  Clusters of S CTAs (one CTA per SM) must fit inside a GPC,
// so how many run at once is queried per S (cudaOccupancyMaxActiveClusters) rather
// than derived from the SM count.  The cost model: waves x (K blocks per CTA + 2),
// the 2 standing for the partial-sum exchange; S <= 8 (a portable cluster) and at
// least two K = 256 blocks per CTA when K allows.
int splitk_factor(int64_t tiles, int64_t K, const int (&active)[9]) {
  const int64_t KB = (K + kBK - 1) / kBK;
  int best = 1;
  int64_t best_cost = -1;
  for (int S = 1; S <= 8; ++S) {
    if (S > 1 && S > KB / 2) break;
    const int64_t act = active[S] > 0 ? active[S] : 1;
    const int64_t waves = (tiles + act - 1) / act;
    const int64_t cost = waves * ((KB + S - 1) / S + 2);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = S; }
  }
  return best;
}

template <int BN, int STAGES>
nvfp4_status run_splitk(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB, float alpha,
                        void* D, int64_t M, int64_t N, int64_t K, cudaStream_t stream, const DeviceInfo& dev,
                        int b_shift = 0) {
  using C = Cfg<BN, STAGES, 1>;
  auto kern = gemm_nvf4_splitk_kernel<BN, STAGES>;
  static PerDeviceOnce setup;
  static int active[64][9] = {};  // co-resident clusters of S CTAs, per device
  const int d = dev.device < 64 ? dev.device : 63;
  const int ok = setup.get(d, [&] {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return 0;
    for (int s = 1; s <= 8; ++s) {
      cudaLaunchConfig_t qc = {};
      qc.gridDim = dim3(s, 1, 1);
      qc.blockDim = dim3(kSplitThreads, 1, 1);
      qc.dynamicSmemBytes = C::kSmemBytes;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = s;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      qc.attrs = qa;
      qc.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &qc) != cudaSuccess) n = 0;
      active[d][s] = n > 0 ? n : dev.num_sms / s;
    }
    return 1;
  });
  if (!ok) return NVFP4_ERR_CUDA;
  const int64_t tiles_m = (M + kBM - 1) / kBM;
  const int64_t tiles_n = (N + BN - 1) / BN;
  if (tiles_m > 65535 || tiles_n > 65535)
    return run<BN, STAGES, 1>(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, b_shift);
  const int S = splitk_factor(tiles_m * tiles_n, K, active[d]);
  CUtensorMap ta, tb;
  nvfp4_status st = encode_tmap_u8_2d(&ta, A, K / 2, M, K / 2, kBKBytes, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != NVFP4_OK) return st;
  st = encode_tmap_u8_2d(&tb, B, (K >> b_shift) / 2, N, (K >> b_shift) / 2, kBKBytes, BN,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != NVFP4_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, static_cast<unsigned>(tiles_n), static_cast<unsigned>(tiles_m));
  cfg.blockDim = dim3(kSplitThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  set_programmatic(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return from_cuda(cudaLaunchKernelEx(&cfg, kern, ta, tb, SFA, SFB, static_cast<__nv_bfloat16*>(D), alpha,
                                      static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), S, b_shift));
}

// Pairs that can be co-resident (cudaOccupancyMaxActiveClusters for clusters of
// two), queried once per device; also sets the kernel's shared-memory limit.
int pair_slots(const DeviceInfo& dev) {
  static PerDeviceOnce slots;
  return slots.get(dev.device, [&] {
    auto kern = pair::gemm_nvf4_pair_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pair::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(pair::gemm_nvf4_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(pair::gemm_nvf4_pair_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair::kSmemBytes) != cudaSuccess)
      return -1;
    cudaLaunchConfig_t qc = {};
    qc.gridDim = dim3(dev.num_sms, 1, 1);
    qc.blockDim = dim3(pair::kThreads, 1, 1);
    qc.dynamicSmemBytes = pair::kSmemBytes;
    cudaLaunchAttribute qa[1];
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = 2;
    qa[0].val.clusterDim.y = 1;
    qa[0].val.clusterDim.z = 1;
    qc.attrs = qa;
    qc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &qc) != cudaSuccess || n < 1) n = dev.num_sms / 2;
    return n;
  });
}

// Stream-K workspace: one flag per (pair, rank), padded to 1 KB, then one 128 x 256
// FP32 partial tile per (pair, rank).
constexpr size_t kPartialBytes = 128 * 256 * 4;
constexpr int64_t kStreamKFixupKB = 16;
size_t streamk_flags_bytes(int pairs) { return ((static_cast<size_t>(pairs) * 2 * 4 + 1023) / 1024) * 1024; }
size_t streamk_bytes(int pairs) { return streamk_flags_bytes(pairs) + static_cast<size_t>(pairs) * 2 * kPartialBytes; }

// streamk: run the hybrid data-parallel / stream-K schedule (workspace required) when
// the tiles are not a whole number of waves; otherwise, or with streamk == false,
// the data-parallel schedule.
nvfp4_status run_pair(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB, float alpha,
                      void* D, int64_t M, int64_t N, int64_t K, cudaStream_t stream, const DeviceInfo& dev,
                      bool streamk = false, void* ws = nullptr, int b_shift = 0, bool clc = false) {
  const int slots = pair_slots(dev);
  if (slots < 0) return NVFP4_ERR_CUDA;
  CUtensorMap ta, tb, tsfa, tsfb, td;
  // A and B as [K/256 chunks][rows][128 bytes]: one box = 128 rows x one stage's chunks.
  nvfp4_status st = encode_tmap_u8_3d_chunks(&ta, A, M, K, 128, pair::kBKP / 256);
  if (st == NVFP4_OK) st = encode_tmap_u8_3d_chunks(&tb, B, N, K >> b_shift, 128, pair::kBKP / 256);
  // Packed scales as [bands][K/64 atoms][128 x u32]: SFA box = one stage's atoms of one
  // band, SFB box = one stage's atoms of two bands.
  if (st == NVFP4_OK) st = encode_tmap_sf_3d(&tsfa, SFA, M, K, pair::kStepsP, 1);
  if (st == NVFP4_OK) st = encode_tmap_sf_3d(&tsfb, SFB, N, K >> b_shift, pair::kStepsP, 2);
  if (st == NVFP4_OK)
    st = encode_tmap_2d(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, N, M, N * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != NVFP4_OK) return st;
  const int tiles_m = static_cast<int>((M + 255) / 256);
  const int tiles_n = static_cast<int>((N + 255) / 256);
  const int num_tiles = tiles_m * tiles_n;
  int use_sk = (streamk && ws != nullptr && num_tiles > slots && num_tiles % slots != 0) ? 1 : 0;
  if (use_sk) {
    // Cost per pair in K-blocks: data-parallel waves against whole waves plus an even
    // share of the rest plus the fix-up.  The fix-up (one partial written, one read
    // back, about four microseconds) and the stream-K instantiation's slower
    // data-parallel waves are charged together as 16 K-blocks, the value at which the
    // measured 4096^3, 8192^3 and 8192 x 5120 x 5120 cases stay data-parallel and the
    // 1024-token layers with 80 tiles split.  Ties stay data-parallel.
    const int64_t KB = K / pair::kBKP;
    const int64_t waves = (num_tiles + slots - 1) / slots;
    const int64_t whole = num_tiles / slots - 1;
    const int64_t units = (num_tiles - whole * slots) * KB;
    const int64_t sk_cost = whole * KB + (units + slots - 1) / slots + kStreamKFixupKB;
    use_sk = sk_cost < waves * KB ? 1 : 0;
  }
  const int pairs = clc ? num_tiles : use_sk ? slots : (num_tiles < slots ? num_tiles : slots);
  const int group_n = tiles_n < 8 ? tiles_n : 8;
  uint32_t* flags = use_sk ? static_cast<uint32_t*>(ws) : nullptr;
  float* part = use_sk ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + streamk_flags_bytes(slots)) : nullptr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(pair::kThreads, 1, 1);
  cfg.dynamicSmemBytes = pair::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  set_programmatic(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  auto kern = clc ? pair::gemm_nvf4_pair_kernel<false, true>
                 : use_sk ? pair::gemm_nvf4_pair_kernel<true> : pair::gemm_nvf4_pair_kernel<false>;
  return from_cuda(cudaLaunchKernelEx(&cfg, kern, ta, tb, tsfa, tsfb, td, alpha, static_cast<int>(K), tiles_m,
                                      tiles_n, group_n, part, flags, b_shift));
}

}  // namespace

nvfp4_status gemm_test_streamk_fault(int skip_publish, unsigned long long flag_wait_ns) {
  const int skip = skip_publish != 0 ? 1 : 0;
  const unsigned long long limit = flag_wait_ns != 0 ? flag_wait_ns : kWaitLimitNs;
  if (cudaMemcpyToSymbol(pair::g_test_skip_publish, &skip, sizeof(skip)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaMemcpyToSymbol(pair::g_flag_wait_ns, &limit, sizeof(limit)) != cudaSuccess) return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

int read_device_error_gemm(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (clear && v != 0) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_device_error, &z, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  return v;
}

int gemm_num_configs() { return kNumConfigs; }

const char* gemm_config_name(int config) {
  if (config < 1 || config > kNumConfigs) return nullptr;
  return kConfigs[config - 1].name;
}

int gemm_choose_config(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
  // Few output tiles (at most half the SMs busy with 128 x 256 tiles) and at least
  // two K = 256 blocks: split K over a cluster.  Otherwise CTA pairs (256 x 256
  // tiles, four K = 256 stages) whenever the tile is filled in both dimensions and K
  // allows the 3-D operand boxes; 128 x 256 single-CTA tiles for skinny M; 128 x 128
  // when N is narrow.
  const int64_t tiles256 = ((M + 127) / 128) * ((N + 255) / 256);
  const int64_t tiles128 = ((M + 127) / 128) * ((N + 127) / 128);
  const int64_t tiles_pair = ((M + 255) / 256) * ((N + 255) / 256);
  // One nearly full wave of CTA pairs (256 x 256 tiles on at least 3/4 of the pairs)
  // beats splitting K, up to K = 8192: measured (graph replay) at M = 128, N = 17408,
  // K = 5120 (68 tiles on 76 pairs): 13.5 us against 17.0 (split over 128 x 256 tiles)
  // and 15.5 (over 128 x 128).  With 20 to 24 pair tiles (N = 5120, 6144) split-K wins.
  if (K % 256 == 0 && K <= 8192 && M > 64 && N > 128 && 4 * tiles_pair >= 3 * (dev.num_sms / 2)) return 3;
  // Split K over 128 x 128 tiles unless those alone nearly fill the SMs (then over
  // 128 x 256 tiles, whose smaller split moves fewer partial sums): measured on the
  // 128-token layer shapes, e.g. 11.8 us against 17.4 us at N = K = 5120.
  if (2 * tiles256 <= dev.num_sms && K >= 512) return (5 * tiles128 >= 4 * dev.num_sms && N > 128) ? 4 : 5;
  if (K % 256 == 0 && M > 128 && N > 128) return 3;
  if (N <= 128 || tiles256 < dev.num_sms / 2) return 2;
  return 1;
}

size_t gemm_streamk_workspace_bytes(const DeviceInfo& dev) {
  const int slots = pair_slots(dev);
  return slots > 0 ? streamk_bytes(slots) : 0;
}

nvfp4_status launch_gemm_streamk(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                                 float alpha, void* D, int64_t M, int64_t N, int64_t K, void* ws,
                                 cudaStream_t stream, const DeviceInfo& dev) {
  // The stream-K schedule belongs to the CTA-pair kernel; shapes that do not run it
  // take the automatic configuration (and leave the workspace untouched).
  const int config = gemm_choose_config(M, N, K, dev);
  if (config != 3 || K % 256 != 0) return launch_gemm(config, A, SFA, B, SFB, alpha, D, M, N, K, stream, dev);
  return run_pair(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, true, ws);
}

nvfp4_status launch_gemm(int config, const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
                         const uint8_t* SFB, float alpha, void* D, int64_t M, int64_t N, int64_t K,
                         cudaStream_t stream, const DeviceInfo& dev, int b_shift) {
  switch (config) {
    case 1: return run<256, 3, 1>(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, b_shift);
    case 2: return run<128, 4, 2>(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, b_shift);
    case 3:
      if (K % 256 != 0) return run<256, 3, 1>(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, b_shift);
      return run_pair(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, false, nullptr, b_shift);
    case 4: return run_splitk<256, 3>(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, b_shift);
    case 5: return run_splitk<128, 4>(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, b_shift);
    case 6:
      if (K % 256 != 0) return run<256, 3, 1>(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, b_shift);
      return run_pair(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev, false, nullptr, b_shift, true);
    default: return NVFP4_ERR_INVALID_ARG;
  }
}

nvfp4_status launch_gemm_two_pass(const uint8_t* A2, const uint8_t* SFA2, const uint8_t* B, const uint8_t* SFB,
                                  float alpha, void* D, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                                  const DeviceInfo& dev) {
  // The activation operand holds 2K codes (value and residual K-blocks interleaved),
  // so every kernel runs over 2K with the weight's K-block index halved: each weight
  // stage is used by one value and one residual K-block, into one accumulator.
  const int64_t K2 = 2 * K;
  return launch_gemm(gemm_choose_config(M, N, K2, dev), A2, SFA2, B, SFB, alpha, D, M, N, K2, stream, dev, 1);
}

}  // namespace nvfp4

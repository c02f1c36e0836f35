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
// grouped raster so that a wave shares A rows and B columns in L2.

#include <cuda_bf16.h>

#include "internal.h"
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

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  int ok = 1;
  if (lane_id() == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int BN, int STAGES, int ACC_BUFS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const uint8_t* __restrict__ SFA, const uint8_t* __restrict__ SFB,
                     __nv_bfloat16* __restrict__ D, float alpha, int M, int N, int K, int tiles_m,
                     int tiles_n, int group_n) {
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
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, tiles_m, tiles_n, group_n, mb, nb);
        int nbv = 0;
#pragma unroll
        for (int b = 0; b < C::kBands; ++b) nbv += (nb * C::kBands + b < bands_n) ? 1 : 0;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag)) { ok = false; break; }
          const int nk = min(kKSteps, KG - kb * kKSteps);
          const uint32_t bytes = C::kABytes + C::kBBytes + nk * kAtom * (1 + nbv);
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, bytes);
          tma_load_2d(sbase + C::kOffA + stage * C::kABytes, &tmA, fb, kb * kBKBytes, mb * kBM, pol);
          tma_load_2d(sbase + C::kOffB + stage * C::kBBytes, &tmB, fb, kb * kBKBytes, nb * BN, pol);
          bulk_load(sbase + C::kOffSFA + stage * C::kSFABytes,
                    SFA + (static_cast<size_t>(mb) * KG + kb * kKSteps) * kAtom, nk * kAtom, fb, pol);
          for (int b = 0; b < nbv; ++b)
            bulk_load(sbase + C::kOffSFB + stage * C::kSFBBytes + b * kKSteps * kAtom,
                      SFB + (static_cast<size_t>(nb * C::kBands + b) * KG + kb * kKSteps) * kAtom,
                      nk * kAtom, fb, pol);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
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
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_nvf4_m128<BN>();
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        if (!mbar_wait(bar_acce + 8 * acc, acc_phase ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const int nk = min(kKSteps, KG - kb * kKSteps);
          const uint32_t sfa_t = tmem + C::kTmemSF + stage * (C::kSFACols + C::kSFBCols);
          const uint32_t sfb_t = sfa_t + C::kSFACols;
          const uint32_t sA = sbase + C::kOffA + stage * C::kABytes;
          const uint32_t sB = sbase + C::kOffB + stage * C::kBBytes;
          const uint32_t sSFA = sbase + C::kOffSFA + stage * C::kSFABytes;
          const uint32_t sSFB = sbase + C::kOffSFB + stage * C::kSFBBytes;
          for (int j = 0; j < nk; ++j) {
            tc_cp_32x128b_warpx4(sfa_t + 4 * j, make_sdesc(sSFA + j * kAtom, 0, 128, 0));
#pragma unroll
            for (int b = 0; b < C::kBands; ++b)
              tc_cp_32x128b_warpx4(sfb_t + 4 * (j * C::kBands + b),
                                   make_sdesc(sSFB + (b * kKSteps + j) * kAtom, 0, 128, 0));
          }
          for (int j = 0; j < nk; ++j) {
            const uint64_t adesc = make_sdesc(sA + j * (kMmaK / 2), 16, 1024, 2);
            const uint64_t bdesc = make_sdesc(sB + j * (kMmaK / 2), 16, 1024, 2);
            tc_mma_nvf4(d_tmem, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + 4 * j * C::kBands,
                        (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(bar_accf + 8 * acc);
        if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
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

// ------------------------------------------------------------------ host side

struct ConfigEntry {
  const char* name;
  int bn;
};

constexpr ConfigEntry kConfigs[] = {
    {"1cta_128x256_s3_acc1", 256},
    {"1cta_128x128_s4_acc2", 128},
};
constexpr int kNumConfigs = sizeof(kConfigs) / sizeof(kConfigs[0]);

template <int BN, int STAGES, int ACC_BUFS>
nvfp4_status run(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB, float alpha,
                 void* D, int64_t M, int64_t N, int64_t K, cudaStream_t stream, const DeviceInfo& dev) {
  using C = Cfg<BN, STAGES, ACC_BUFS>;
  auto kern = gemm_nvf4_kernel<BN, STAGES, ACC_BUFS>;
  static bool attr_set[64] = {};
  if (dev.device < 64 && !attr_set[dev.device]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    attr_set[dev.device] = true;
  }
  CUtensorMap ta, tb;
  nvfp4_status st = encode_tmap_u8_2d(&ta, A, K / 2, M, K / 2, kBKBytes, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != NVFP4_OK) return st;
  st = encode_tmap_u8_2d(&tb, B, K / 2, N, K / 2, kBKBytes, BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != NVFP4_OK) return st;
  const int tiles_m = static_cast<int>((M + kBM - 1) / kBM);
  const int tiles_n = static_cast<int>((N + BN - 1) / BN);
  const int num_tiles = tiles_m * tiles_n;
  const int grid = num_tiles < dev.num_sms ? num_tiles : dev.num_sms;
  const int group_n = tiles_n < 8 ? tiles_n : 8;
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(ta, tb, SFA, SFB, static_cast<__nv_bfloat16*>(D), alpha,
                                                   static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                                                   tiles_m, tiles_n, group_n);
  return from_cuda(cudaGetLastError());
}

}  // namespace

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
  (void)K;
  // Prefer the wide tile unless it leaves most SMs idle on a small problem.
  const int64_t tiles256 = ((M + 127) / 128) * ((N + 255) / 256);
  if (N <= 128 || tiles256 < dev.num_sms / 2) return 2;
  return 1;
}

nvfp4_status launch_gemm(int config, const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
                         const uint8_t* SFB, float alpha, void* D, int64_t M, int64_t N, int64_t K,
                         cudaStream_t stream, const DeviceInfo& dev) {
  switch (config) {
    case 1: return run<256, 3, 1>(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev);
    case 2: return run<128, 4, 2>(A, SFA, B, SFB, alpha, D, M, N, K, stream, dev);
    default: return NVFP4_ERR_INVALID_ARG;
  }
}

}  // namespace nvfp4

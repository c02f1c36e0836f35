// mma_ceiling.cu -- diagnostic: the tensor-core instruction ceiling of this GPU.
//
// Every CTA pair issues `iters` tcgen05.mma.cta_group::2 instructions of one kind
// (M = 256 across the pair, N = 256, operands resident in shared memory, FP32
// accumulator in TMEM) back to back from one thread, and times the span.  Kinds:
// the block-scaled FP4 MMA of the GEMM (kind::mxf4nvf4, scale_vec::4X, K = 64 per
// instruction), BF16 (kind::f16, K = 16) and E4M3 (kind::f8f6f4, K = 32).  The
// ratio of their rates is the hardware's own FP4 : BF16 : FP8 ratio, which is what
// the FP4 roofline denominator should scale the measured BF16 peak by.  The operand
// values are a fixed finite pattern and every scale is 1.0; the accumulator is never
// read.  Waits are bounded (2 s); a timeout is reported as NVFP4_ERR_TIMEOUT.

#include <algorithm>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kKindNvf4 = 0, kKindBf16 = 1, kKindFp8 = 2;
constexpr int kTileBytes = 128 * 128;         // 128 rows x 128 bytes, 128-byte swizzle
constexpr int kOffA = 0;                      // 4 A tiles
constexpr int kOffB = 4 * kTileBytes;         // 4 B tiles (128 rows of this CTA's half of N = 256)
constexpr int kOffSF = 8 * kTileBytes;        // scale atoms (all 1.0)
constexpr int kSFBytes = 8192;
constexpr int kOffBar = kOffSF + kSFBytes;
constexpr int kSmem = kOffBar + 64 + 1024;
constexpr int kMaxUnits = 128;                // CTA pairs per launch

__device__ unsigned long long g_ceiling_out[2 * kMaxUnits];  // per pair: clock cycles, ns
__device__ int g_ceiling_err;

__device__ __forceinline__ void mma_pair_plain(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc,
                                               int kind) {
  if (kind == kKindBf16)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

template <int KIND>
__global__ void __launch_bounds__(128, 1) mma_ceiling_kernel(int iters) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool leader = cluster_ctarank() == 0;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 56);
  const uint32_t bar_done = sb + kOffBar;
  for (int i = threadIdx.x; i < 8 * kTileBytes / 4; i += blockDim.x) {
    uint32_t h = static_cast<uint32_t>(i) * 2654435761u ^ (blockIdx.x * 97u);
    if (KIND == kKindBf16) h = 0x3F803F80u ^ (h & 0x007F007Fu);       // bf16 in [1, 2)
    else if (KIND == kKindFp8) h = (h & 0x3F3F3F3Fu) | 0x30303030u;   // finite E4M3
    reinterpret_cast<uint32_t*>(smem)[i] = h;                          // any E2M1 byte is finite
  }
  for (int i = threadIdx.x; i < kSFBytes / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(smem + kOffSF)[i] = 0x38383838u;     // UE4M3 1.0
  if (threadIdx.x == 0) {
    mbar_init(bar_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc_pair(smem_u32(slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (leader && warp == 1 && lane == 0) {
    const uint32_t sf0 = tmem + 256;  // 4 scale slots of 48 columns after the accumulator
    if (KIND == kKindNvf4) {
      for (int s = 0; s < 4; ++s)
        for (int j = 0; j < 4; ++j) {
          tc_cp_32x128b_warpx4_pair(sf0 + 48 * s + 4 * j, make_sdesc(sb + kOffSF + j * 512, 0, 128, 0));
          for (int b = 0; b < 2; ++b)
            tc_cp_32x128b_warpx4_pair(sf0 + 48 * s + 16 + 8 * j + 4 * b,
                                      make_sdesc(sb + kOffSF + 2048 + (b * 4 + j) * 512, 0, 128, 0));
        }
    }
    uint32_t idesc = (static_cast<uint32_t>(256 >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
    if (KIND == kKindNvf4) idesc |= (1u << 7) | (1u << 10);              // E2M1 x E2M1
    else if (KIND == kKindBf16) idesc |= (1u << 4) | (1u << 7) | (1u << 10);  // FP32 acc, BF16 x BF16
    else idesc |= (1u << 4);                                              // FP32 acc, E4M3 x E4M3
    const uint64_t a0 = make_sdesc(sb + kOffA, 16, 1024, 2), b0 = make_sdesc(sb + kOffB, 16, 1024, 2);
    tc_fence_after();
    const unsigned long long c0 = clock64();
    const uint64_t g0 = globaltimer_ns();
#pragma unroll 1
    for (int i = 0; i < iters; i += 4) {
      const int s = (i >> 2) & 3;  // tile (and scale slot) of this group of 4
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // 4 instructions along each 128-byte row
        const uint64_t ad = a0 + ((s * kTileBytes + j * 32) >> 4);
        const uint64_t bd = b0 + ((s * kTileBytes + j * 32) >> 4);
        const uint32_t acc = (i | j) ? 1u : 0u;
        if (KIND == kKindNvf4)
          tc_mma_nvf4_pair(tmem, ad, bd, idesc, sf0 + 48 * s + 4 * j, sf0 + 48 * s + 16 + 8 * j, acc);
        else
          mma_pair_plain(tmem, ad, bd, idesc, acc, KIND);
      }
    }
    tc_commit_pair_mc(bar_done, 0x1);
    if (!mbar_wait_for(bar_done, 0, kWaitLimitNs)) atomicExch(&g_ceiling_err, 1);
    const unsigned long long cyc = clock64() - c0;
    const uint64_t ns = globaltimer_ns() - g0;
    g_ceiling_out[2 * (blockIdx.x / 2)] = cyc;
    g_ceiling_out[2 * (blockIdx.x / 2) + 1] = ns;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

nvfp4_status mma_ceiling(int kind, int iters, double* tflops, double* cycles_per_mma, cudaStream_t stream,
                         const DeviceInfo& dev) {
  const int units = std::min(dev.num_sms / 2, kMaxUnits);
  if (units < 1 || static_cast<size_t>(kSmem) > dev.max_smem_optin) return NVFP4_ERR_UNSUPPORTED_DEVICE;
  void (*kern)(int) = kind == kKindNvf4 ? mma_ceiling_kernel<kKindNvf4>
                      : kind == kKindBf16 ? mma_ceiling_kernel<kKindBf16>
                                          : mma_ceiling_kernel<kKindFp8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_ceiling_err, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * units);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, iters) != cudaSuccess) return NVFP4_ERR_CUDA;
  std::vector<unsigned long long> h(2 * units);
  int err = 0;
  if (cudaMemcpyFromSymbolAsync(h.data(), g_ceiling_out, h.size() * sizeof(unsigned long long), 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&err, g_ceiling_err, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  if (err != 0) return NVFP4_ERR_TIMEOUT;
  std::vector<double> cyc(units);
  double max_ns = 0;
  for (int u = 0; u < units; ++u) {
    cyc[u] = static_cast<double>(h[2 * u]) / iters;
    max_ns = std::max(max_ns, static_cast<double>(h[2 * u + 1]));
  }
  std::sort(cyc.begin(), cyc.end());
  const double k = kind == kKindNvf4 ? 64 : kind == kKindBf16 ? 16 : 32;
  const double flops = 2.0 * 256 * 256 * k * iters * units;
  if (tflops != nullptr) *tflops = max_ns > 0 ? flops / max_ns * 1e-3 : 0.0;
  if (cycles_per_mma != nullptr) *cycles_per_mma = cyc[units / 2];
  return NVFP4_OK;
}

}  // namespace nvfp4

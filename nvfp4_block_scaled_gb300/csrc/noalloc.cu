// noalloc.cu -- nvfp4_gemm_streamk_noalloc: the stream-K GEMM with its scratch held
// in a static device array of this library instead of a caller workspace.
//
// The array lives in this translation unit's own module, so it is only brought in
// (with lazy module loading, the CUDA default) by the first call of this entry point.
// Nothing here allocates: the array's device address is looked up once per device
// with cudaGetSymbolAddress, and the call goes through nvfp4_gemm_streamk unchanged.
// The address and the "cleared" flag are cached per device ordinal for the life of
// the process: the entry point is not valid across cudaDeviceReset.

#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "nvfp4.h"

namespace {

// 20 MiB + 4 KiB: the stream-K flag words plus one 128 KB FP32 partial per CTA of a
// grid of up to 80 CTA pairs (a GB300 runs 76).
constexpr size_t kScratchBytes = (size_t{20} << 20) + 4096;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_streamk_scratch[kScratchBytes];

void* g_addr[kMaxDevices];
cudaError_t g_addr_err[kMaxDevices];
std::once_flag g_addr_once[kMaxDevices];
std::atomic<bool> g_cleared[kMaxDevices];

}  // namespace

extern "C" nvfp4_status nvfp4_gemm_streamk_noalloc(const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
                                                   const uint8_t* SFB, float alpha, void* D_bf16, int64_t M,
                                                   int64_t N, int64_t K, int reset_scratch,
                                                   nvfp4_stream_t stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::call_once(g_addr_once[dev], [dev]() {
    void* p = nullptr;
    g_addr_err[dev] = cudaGetSymbolAddress(&p, g_streamk_scratch);
    g_addr[dev] = g_addr_err[dev] == cudaSuccess ? p : nullptr;
  });
  if (g_addr_err[dev] != cudaSuccess || g_addr[dev] == nullptr) return NVFP4_ERR_CUDA;

  // The scratch this device's CTA-pair grid needs; more than the array holds is refused
  // before anything is enqueued.
  const size_t need = nvfp4_gemm_streamk_workspace_bytes();
  if (need == 0) return NVFP4_ERR_UNSUPPORTED_DEVICE;
  if (need > kScratchBytes) return NVFP4_ERR_UNSUPPORTED_DEVICE;

  // The flag words must read zero when a launch starts.  The first call on a device
  // clears the scratch on its stream, and so does a call with reset_scratch set (the
  // way back after a device-side timeout left flags raised).
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool first = !g_cleared[dev].exchange(true);
  if (first || reset_scratch != 0) {
    if (cudaMemsetAsync(g_addr[dev], 0, need, s) != cudaSuccess) {
      if (first) g_cleared[dev].store(false);
      return NVFP4_ERR_CUDA;
    }
  }
  return nvfp4_gemm_streamk(A, SFA, B, SFB, alpha, D_bf16, M, N, K, g_addr[dev], kScratchBytes, stream);
}

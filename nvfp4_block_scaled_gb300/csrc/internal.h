// internal.h -- host-side helpers shared by the translation units of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int cc_major = 0;
  int cc_minor = 0;
  size_t max_smem_optin = 0;
  size_t smem_per_sm = 0;
  bool ok = false;  // compute capability 10.3
};

// Cached properties of the current device (queried once per device).
nvfp4_status current_device(DeviceInfo* out);

// One-time setup per device (kernel attributes, occupancy queries) that host threads
// may reach concurrently: the first caller for a device runs `f`, callers arriving
// meanwhile wait for it, and every later call returns the same result.  Each call
// site owns its own instance (a function-local static).
struct PerDeviceOnce {
  std::once_flag flag[64];
  int result[64] = {};
  template <typename F>
  int get(int device, F&& f) {
    const int d = device >= 0 && device < 64 ? device : 63;
    std::call_once(flag[d], [&] { result[d] = f(); });
    return result[d];
  }
};

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline nvfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

// 2-D UINT8 tensor map over a row-major byte matrix [outer x inner] with the given
// row pitch, box [box_outer x box_inner], zero fill out of bounds.
nvfp4_status encode_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                               uint64_t row_pitch, uint32_t box_inner, uint32_t box_outer,
                               CUtensorMapSwizzle swizzle);

// Same, for any element type (inner/box_inner in elements, row_pitch in bytes).
nvfp4_status encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                            uint64_t outer, uint64_t row_pitch, uint32_t box_inner, uint32_t box_outer,
                            CUtensorMapSwizzle swizzle);

// 3-D UINT8 map over packed K-major codes [rows x K/2] viewed as [K/256][rows][128 B]
// (128-byte swizzle); K % 256 == 0.  A box is box_rows x box_chunks 128-byte chunks.
nvfp4_status encode_tmap_u8_3d_chunks(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t box_rows,
                                      uint32_t box_chunks);

// 3-D UINT32 map over a packed scale buffer viewed as [bands][K/64 atoms][128 words];
// a box is box_bands x box_atoms atoms (out-of-range atoms / bands read as zero).
nvfp4_status encode_tmap_sf_3d(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t box_atoms,
                               uint32_t box_bands);

// 3-D UINT64 map over a prepared W4A16 weight viewed as [N/16][K/64][576 bytes];
// a box is box_ntiles n-tiles x box_blocks blocks (default 8 x 8: 128 rows x 512 K, 36 KB).
nvfp4_status encode_tmap_wprep(CUtensorMap* map, const void* wprep, int64_t N, int64_t K, uint32_t box_blocks = 8,
                               uint32_t box_ntiles = 8);
// bf16 activations [M][K] viewed as [K/64 blocks][M tokens][64]: box = box_blocks x
// box_rows tokens x 64, 128-byte swizzled; tokens past M read as zero.
nvfp4_status encode_tmap_x_blocks(CUtensorMap* map, const void* x, int64_t M, int64_t K, uint32_t box_rows,
                                  uint32_t box_blocks);

// Per-translation-unit device error words (see ptx.cuh): returns the recorded
// status (0 if none) or NVFP4_ERR_CUDA, optionally clearing it.
int read_device_error_gemm(bool clear);
// Test-only fault injection for the stream-K schedule (see nvfp4_test_streamk_fault).
nvfp4_status gemm_test_streamk_fault(int skip_publish, unsigned long long flag_wait_ns);
int read_device_error_w4a16(bool clear);

// Kernel launchers (defined next to their kernels).
// packed = false: sf is [rows x K/16] row-major; true: sf is the packed 128x4-atom
// buffer of nvfp4_packed_scales_bytes(rows, K) bytes, padding written as zero.
nvfp4_status launch_quantize(const void* x, int64_t rows, int64_t K, float g, uint8_t* codes,
                             uint8_t* sf, bool packed, cudaStream_t stream, const DeviceInfo& dev);
nvfp4_status launch_pack_scales(const uint8_t* sf, int64_t rows, int64_t K, uint8_t* out,
                                cudaStream_t stream, const DeviceInfo& dev);
// Two-pass quantisation: codes [rows x K] bytes (2K codes, value and residual
// K-blocks of 256 interleaved), scales packed for a [rows x 2K] operand; K % 256 == 0.
nvfp4_status launch_quantize_two_pass(const void* x, int64_t rows, int64_t K, float g, uint8_t* codes,
                                      uint8_t* sf_packed, cudaStream_t stream, const DeviceInfo& dev);

int gemm_num_configs();
const char* gemm_config_name(int config);
int gemm_choose_config(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);
// b_shift = 1: B (and SFB) hold K >> 1 elements per row, and A's K-block kb meets
// B's K-block kb >> 1 (the two-pass activation layout); 0 for a plain GEMM.
nvfp4_status launch_gemm(int config, const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
                         const uint8_t* SFB, float alpha, void* D, int64_t M, int64_t N, int64_t K,
                         cudaStream_t stream, const DeviceInfo& dev, int b_shift = 0);
// Two-pass W4A4 GEMM: A2/SFA2 hold the value and residual codes of a [M x K]
// activation interleaved per 256-element K-block (2K codes per row); B is [N x K].
nvfp4_status launch_gemm_two_pass(const uint8_t* A2, const uint8_t* SFA2, const uint8_t* B, const uint8_t* SFB,
                                  float alpha, void* D, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                                  const DeviceInfo& dev);

// Stream-K GEMM: workspace bytes for the current device, and the launch (falls back
// to launch_gemm's automatic configuration for shapes the CTA-pair kernel does not take).
size_t gemm_streamk_workspace_bytes(const DeviceInfo& dev);
nvfp4_status launch_gemm_streamk(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                                 float alpha, void* D, int64_t M, int64_t N, int64_t K, void* ws,
                                 cudaStream_t stream, const DeviceInfo& dev);

nvfp4_status launch_w4a16_prepare(const uint8_t* W, const uint8_t* SW, int64_t N, int64_t K, void* Wprep,
                                  cudaStream_t stream, const DeviceInfo& dev);
// alpha_col: NULL for the global scale alpha, else N per-output-column FP32 scales.
nvfp4_status launch_w4a16_linear(const void* x, const void* Wprep, float alpha, const float* alpha_col, void* y,
                                 int64_t M, int64_t N, int64_t K, cudaStream_t stream, const DeviceInfo& dev);
// Balanced (stream-K) W4A16 linear: workspace bytes for the current device, and the
// launch (more than 32 tokens go to launch_w4a16_linear's tensor-core kernel).
size_t w4a16_streamk_workspace_bytes(const DeviceInfo& dev);
nvfp4_status launch_w4a16_linear_streamk(const void* x, const void* Wprep, float alpha, const float* alpha_col,
                                         void* y, int64_t M, int64_t N, int64_t K, void* ws, cudaStream_t stream,
                                         const DeviceInfo& dev);

// Diagnostic: tcgen05 instruction ceiling for kind 0 (block-scaled FP4), 1 (BF16) or
// 2 (E4M3); see nvfp4_mma_ceiling.
nvfp4_status mma_ceiling(int kind, int iters, double* tflops, double* cycles_per_mma, cudaStream_t stream,
                         const DeviceInfo& dev);

}  // namespace nvfp4

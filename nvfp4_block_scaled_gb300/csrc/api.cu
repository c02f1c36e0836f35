// api.cu -- the extern "C" entry points declared in include/nvfp4.h: argument
// checks, device checks, tensor-map encoding and dispatch to the kernel launchers.

#include <cstdio>
#include <mutex>

#include "internal.h"

namespace nvfp4 {

namespace {

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

nvfp4_status current_device(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::call_once(g_dev_once[dev], [dev]() {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) d.num_sms = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess) d.cc_major = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess) d.cc_minor = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess)
      d.max_smem_optin = static_cast<size_t>(v);
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess)
      d.smem_per_sm = static_cast<size_t>(v);
    d.ok = d.cc_major == 10 && d.cc_minor == 3 && d.num_sms > 0;
    g_devices[dev] = d;
  });
  *out = g_devices[dev];
  if (out->num_sms <= 0) return NVFP4_ERR_CUDA;
  return out->ok ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED_DEVICE;
}

nvfp4_status encode_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                               uint64_t row_pitch, uint32_t box_inner, uint32_t box_outer,
                               CUtensorMapSwizzle swizzle) {
  return encode_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, inner, outer, row_pitch, box_inner, box_outer,
                        swizzle);
}

nvfp4_status encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                            uint64_t outer, uint64_t row_pitch, uint32_t box_inner, uint32_t box_outer,
                            CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return NVFP4_ERR_CUDA;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_pitch};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status encode_tmap_u8_3d_chunks(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t box_rows,
                                      uint32_t box_chunks) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || K % 256 != 0) return NVFP4_ERR_CUDA;
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K / 256)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K / 2), 128};
  const cuuint32_t box[3] = {128, box_rows, box_chunks};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status encode_tmap_sf_3d(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t box_atoms,
                               uint32_t box_bands) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || K % 64 != 0) return NVFP4_ERR_CUDA;
  const int64_t bands = (rows + 127) / 128, atoms = K / 64;
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(atoms), static_cast<cuuint64_t>(bands)};
  const cuuint64_t strides[2] = {512, static_cast<cuuint64_t>(atoms * 512)};
  const cuuint32_t box[3] = {128, box_atoms, box_bands};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status encode_tmap_wprep(CUtensorMap* map, const void* wprep, int64_t N, int64_t K, uint32_t box_blocks,
                               uint32_t box_ntiles) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return NVFP4_ERR_CUDA;
  const cuuint64_t dims[3] = {72, static_cast<cuuint64_t>(K / 64), static_cast<cuuint64_t>(N / 16)};
  const cuuint64_t strides[2] = {576, static_cast<cuuint64_t>(K / 64) * 576};
  const cuuint32_t box[3] = {72, box_blocks, box_ntiles};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void*>(wprep), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status encode_tmap_x_blocks(CUtensorMap* map, const void* x, int64_t M, int64_t K, uint32_t box_rows,
                                  uint32_t box_blocks) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || K % 64 != 0) return NVFP4_ERR_CUDA;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, box_blocks};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4

using namespace nvfp4;

namespace {

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

inline cudaStream_t as_stream(nvfp4_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* nvfp4_status_string(nvfp4_status status) {
  switch (static_cast<int>(status)) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "NVFP4_ERR_UNSUPPORTED_SHAPE";
    case NVFP4_ERR_MISALIGNED: return "NVFP4_ERR_MISALIGNED";
    case NVFP4_ERR_UNSUPPORTED_DEVICE: return "NVFP4_ERR_UNSUPPORTED_DEVICE";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
    case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
    default: return "NVFP4_ERR_UNKNOWN";
  }
}

int nvfp4_version(void) { return 10000; }

static nvfp4_status quantize_checks(const void* x_bf16, int64_t rows, int64_t K, float global_scale,
                                    const uint8_t* codes, const uint8_t* sf) {
  if (x_bf16 == nullptr || codes == nullptr || sf == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (rows < 1 || K < 16 || rows > kMaxDim || K > kMaxDim) return NVFP4_ERR_INVALID_ARG;
  if (!(global_scale > 0.0f) || !(global_scale <= 3.4028234663852886e38f)) return NVFP4_ERR_INVALID_ARG;
  if (K % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x_bf16, 16) || !aligned(codes, 8)) return NVFP4_ERR_MISALIGNED;
  return NVFP4_OK;
}

nvfp4_status nvfp4_quantize(const void* x_bf16, int64_t rows, int64_t K, float global_scale, uint8_t* codes,
                            uint8_t* sf_rowmajor, nvfp4_stream_t stream) {
  nvfp4_status st = quantize_checks(x_bf16, rows, K, global_scale, codes, sf_rowmajor);
  if (st != NVFP4_OK) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return launch_quantize(x_bf16, rows, K, global_scale, codes, sf_rowmajor, false, as_stream(stream), dev);
}

nvfp4_status nvfp4_quantize_packed(const void* x_bf16, int64_t rows, int64_t K, float global_scale,
                                   uint8_t* codes, uint8_t* sf_packed, nvfp4_stream_t stream) {
  nvfp4_status st = quantize_checks(x_bf16, rows, K, global_scale, codes, sf_packed);
  if (st != NVFP4_OK) return st;
  if (!aligned(sf_packed, 16)) return NVFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return launch_quantize(x_bf16, rows, K, global_scale, codes, sf_packed, true, as_stream(stream), dev);
}

nvfp4_status nvfp4_quantize_two_pass(const void* x_bf16, int64_t rows, int64_t K, float global_scale,
                                     uint8_t* codes2, uint8_t* sf2_packed, nvfp4_stream_t stream) {
  nvfp4_status st = quantize_checks(x_bf16, rows, K, global_scale, codes2, sf2_packed);
  if (st != NVFP4_OK) return st;
  if (K % 256 != 0 || 2 * K > kMaxDim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(sf2_packed, 16)) return NVFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return launch_quantize_two_pass(x_bf16, rows, K, global_scale, codes2, sf2_packed, as_stream(stream), dev);
}

size_t nvfp4_packed_scales_bytes(int64_t rows, int64_t K) {
  if (rows < 1 || K < 16 || K % 16 != 0 || rows > kMaxDim || K > kMaxDim) return 0;
  return static_cast<size_t>((rows + 127) / 128) * 128 * static_cast<size_t>((K + 63) / 64) * 4;
}

nvfp4_status nvfp4_pack_scales(const uint8_t* sf_rowmajor, int64_t rows, int64_t K, uint8_t* sf_packed,
                               nvfp4_stream_t stream) {
  if (sf_rowmajor == nullptr || sf_packed == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (rows < 1 || K < 16 || rows > kMaxDim || K > kMaxDim) return NVFP4_ERR_INVALID_ARG;
  if (K % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(sf_packed, 16)) return NVFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return launch_pack_scales(sf_rowmajor, rows, K, sf_packed, as_stream(stream), dev);
}

static nvfp4_status gemm_checks(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                                float alpha, void* D, int64_t M, int64_t N, int64_t K) {
  if (A == nullptr || SFA == nullptr || B == nullptr || SFB == nullptr || D == nullptr)
    return NVFP4_ERR_INVALID_ARG;
  if (M < 1 || N < 8 || K < 64 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return NVFP4_ERR_INVALID_ARG;
  if (!(alpha == alpha) || alpha > 3.4028234663852886e38f || alpha < -3.4028234663852886e38f)
    return NVFP4_ERR_INVALID_ARG;
  if (K % 64 != 0 || N % 8 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(SFA, 16) || !aligned(SFB, 16) || !aligned(D, 16))
    return NVFP4_ERR_MISALIGNED;
  return NVFP4_OK;
}

nvfp4_status nvfp4_gemm_config(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                               float alpha, void* D_bf16, int64_t M, int64_t N, int64_t K, int config,
                               nvfp4_stream_t stream) {
  nvfp4_status st = gemm_checks(A, SFA, B, SFB, alpha, D_bf16, M, N, K);
  if (st != NVFP4_OK) return st;
  if (config < 0 || config > gemm_num_configs()) return NVFP4_ERR_INVALID_ARG;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  if (config == 0) config = gemm_choose_config(M, N, K, dev);
  return launch_gemm(config, A, SFA, B, SFB, alpha, D_bf16, M, N, K, as_stream(stream), dev);
}

nvfp4_status nvfp4_gemm(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB, float alpha,
                        void* D_bf16, int64_t M, int64_t N, int64_t K, nvfp4_stream_t stream) {
  return nvfp4_gemm_config(A, SFA, B, SFB, alpha, D_bf16, M, N, K, 0, stream);
}

size_t nvfp4_gemm_streamk_workspace_bytes(void) {
  DeviceInfo dev;
  if (current_device(&dev) != NVFP4_OK) return 0;
  return gemm_streamk_workspace_bytes(dev);
}

nvfp4_status nvfp4_gemm_streamk(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                                float alpha, void* D_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                                size_t workspace_bytes, nvfp4_stream_t stream) {
  nvfp4_status st = gemm_checks(A, SFA, B, SFB, alpha, D_bf16, M, N, K);
  if (st != NVFP4_OK) return st;
  if (workspace == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return NVFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const size_t need = gemm_streamk_workspace_bytes(dev);
  if (need == 0) return NVFP4_ERR_CUDA;
  if (workspace_bytes < need) return NVFP4_ERR_INVALID_ARG;
  return launch_gemm_streamk(A, SFA, B, SFB, alpha, D_bf16, M, N, K, workspace, as_stream(stream), dev);
}

nvfp4_status nvfp4_gemm_two_pass(const uint8_t* A2, const uint8_t* SFA2, const uint8_t* B, const uint8_t* SFB,
                                 float alpha, void* D_bf16, int64_t M, int64_t N, int64_t K, nvfp4_stream_t stream) {
  nvfp4_status st = gemm_checks(A2, SFA2, B, SFB, alpha, D_bf16, M, N, K);
  if (st != NVFP4_OK) return st;
  if (K % 256 != 0 || 2 * K > kMaxDim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return launch_gemm_two_pass(A2, SFA2, B, SFB, alpha, D_bf16, M, N, K, as_stream(stream), dev);
}

const char* nvfp4_gemm_config_name(int config) { return gemm_config_name(config); }

int nvfp4_gemm_choose_config(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 8 || K < 64) return NVFP4_ERR_INVALID_ARG;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return gemm_choose_config(M, N, K, dev);
}

size_t nvfp4_w4a16_prepared_bytes(int64_t N, int64_t K) {
  if (N < 16 || K < 64 || N % 16 != 0 || K % 64 != 0 || N > kMaxDim || K > kMaxDim) return 0;
  return static_cast<size_t>(N) * static_cast<size_t>(K) / 2 + static_cast<size_t>(N) * static_cast<size_t>(K) / 16;
}

nvfp4_status nvfp4_w4a16_prepare(const uint8_t* W_codes, const uint8_t* W_sf_rowmajor, int64_t N, int64_t K,
                                 void* Wprep, nvfp4_stream_t stream) {
  if (W_codes == nullptr || W_sf_rowmajor == nullptr || Wprep == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (N < 16 || K < 64 || N > kMaxDim || K > kMaxDim) return NVFP4_ERR_INVALID_ARG;
  if (N % 16 != 0 || K % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(Wprep, 16) || !aligned(W_codes, 16)) return NVFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return launch_w4a16_prepare(W_codes, W_sf_rowmajor, N, K, Wprep, as_stream(stream), dev);
}

static nvfp4_status w4a16_checks(const void* x_bf16, const void* Wprep, void* y_bf16, int64_t M, int64_t N,
                                 int64_t K) {
  if (x_bf16 == nullptr || Wprep == nullptr || y_bf16 == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (M < 1 || N < 128 || K < 256 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return NVFP4_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 256 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x_bf16, 16) || !aligned(Wprep, 16) || !aligned(y_bf16, 16)) return NVFP4_ERR_MISALIGNED;
  return NVFP4_OK;
}

nvfp4_status nvfp4_w4a16_linear(const void* x_bf16, const void* Wprep, float alpha, void* y_bf16, int64_t M,
                                int64_t N, int64_t K, nvfp4_stream_t stream) {
  nvfp4_status st = w4a16_checks(x_bf16, Wprep, y_bf16, M, N, K);
  if (st != NVFP4_OK) return st;
  if (!(alpha == alpha) || alpha > 3.4028234663852886e38f || alpha < -3.4028234663852886e38f)
    return NVFP4_ERR_INVALID_ARG;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return launch_w4a16_linear(x_bf16, Wprep, alpha, nullptr, y_bf16, M, N, K, as_stream(stream), dev);
}

nvfp4_status nvfp4_w4a16_linear_colscale(const void* x_bf16, const void* Wprep, const float* alpha_col,
                                         void* y_bf16, int64_t M, int64_t N, int64_t K, nvfp4_stream_t stream) {
  nvfp4_status st = w4a16_checks(x_bf16, Wprep, y_bf16, M, N, K);
  if (st != NVFP4_OK) return st;
  if (alpha_col == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(alpha_col, 16)) return NVFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return launch_w4a16_linear(x_bf16, Wprep, 1.0f, alpha_col, y_bf16, M, N, K, as_stream(stream), dev);
}

size_t nvfp4_w4a16_streamk_workspace_bytes(void) {
  DeviceInfo dev;
  if (current_device(&dev) != NVFP4_OK) return 0;
  return w4a16_streamk_workspace_bytes(dev);
}

nvfp4_status nvfp4_w4a16_linear_streamk(const void* x_bf16, const void* Wprep, float alpha, const float* alpha_col,
                                        void* y_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                                        size_t workspace_bytes, nvfp4_stream_t stream) {
  nvfp4_status st = w4a16_checks(x_bf16, Wprep, y_bf16, M, N, K);
  if (st != NVFP4_OK) return st;
  if (alpha_col == nullptr &&
      (!(alpha == alpha) || alpha > 3.4028234663852886e38f || alpha < -3.4028234663852886e38f))
    return NVFP4_ERR_INVALID_ARG;
  if (alpha_col != nullptr && !aligned(alpha_col, 16)) return NVFP4_ERR_MISALIGNED;
  if (workspace == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return NVFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  if (workspace_bytes < w4a16_streamk_workspace_bytes(dev)) return NVFP4_ERR_INVALID_ARG;
  return launch_w4a16_linear_streamk(x_bf16, Wprep, alpha_col != nullptr ? 1.0f : alpha, alpha_col, y_bf16, M, N,
                                     K, workspace, as_stream(stream), dev);
}

nvfp4_status nvfp4_mma_ceiling(int kind, int iters, double* tflops, double* cycles_per_mma,
                               nvfp4_stream_t stream) {
  if (kind < 0 || kind > 2 || iters < 4 || iters % 4 != 0 || iters > (1 << 24)) return NVFP4_ERR_INVALID_ARG;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return mma_ceiling(kind, iters, tflops, cycles_per_mma, as_stream(stream), dev);
}

nvfp4_status nvfp4_device_error(nvfp4_stream_t stream, int clear) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return NVFP4_ERR_CUDA;
  const int a = read_device_error_gemm(clear != 0);
  const int b = read_device_error_w4a16(clear != 0);
  if (a == NVFP4_ERR_CUDA || b == NVFP4_ERR_CUDA) return NVFP4_ERR_CUDA;
  if (a != 0) return static_cast<nvfp4_status>(a);
  if (b != 0) return static_cast<nvfp4_status>(b);
  return NVFP4_OK;
}

nvfp4_status nvfp4_test_streamk_fault(int skip_publish, uint64_t flag_wait_ns) {
  DeviceInfo dev;
  const nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  return gemm_test_streamk_fault(skip_publish, static_cast<unsigned long long>(flag_wait_ns));
}

}  // extern "C"

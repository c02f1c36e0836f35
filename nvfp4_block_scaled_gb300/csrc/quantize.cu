// quantize.cu -- NVFP4 operand producers: BF16 -> E2M1 codes + E4M3 block scales,
// and the row-major -> 128x4-atom scale-factor permutation.
//
// Both kernels are HBM-bound elementwise/permutation kernels: one 16-element block
// per thread (coalesced 32-byte loads, 8-byte code stores), grid sized to a
// multiple of the SM count with a grid-stride loop.

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

// Exact value of a non-negative E4M3 byte (1..0x7E or 0) as float: normal
// (1 + m/8) 2^(e-7), subnormal m 2^-9.
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xF;
  const uint32_t m = b & 7;
  if (e == 0) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9, exact
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Eight floats -> eight E2M1 codes (round to nearest even, saturating), packed
// little-endian: v[0] in the low nibble of byte 0, v[7] in the high nibble of byte 3.
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4, float v5,
                                           float v6, float v7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

__global__ void __launch_bounds__(256) quantize_kernel(const uint4* __restrict__ x, int64_t nblocks,
                                                       float g, uint2* __restrict__ codes,
                                                       uint8_t* __restrict__ sf) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
    const uint4 v0 = __ldcs(x + 2 * b);
    const uint4 v1 = __ldcs(x + 2 * b + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    const float s = __fdiv_rn(__fdiv_rn(amax, 6.0f), g);
    const uint32_t sbyte = __nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3);
    uint32_t c0 = 0, c1 = 0;
    if (sbyte != 0) {
      const float denom = __fmul_rn(e4m3_to_float(sbyte), g);
      float q[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(f[i], denom);
      c0 = e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
      c1 = e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
      // A code whose magnitude rounded to zero is written as +0 (clear its sign bit).
      const uint32_t nz0 = ((c0 & 0x77777777u) + 0x77777777u) & 0x88888888u;
      const uint32_t nz1 = ((c1 & 0x77777777u) + 0x77777777u) & 0x88888888u;
      c0 &= 0x77777777u | nz0;
      c1 &= 0x77777777u | nz1;
    }
    __stcs(codes + b, make_uint2(c0, c1));
    sf[b] = static_cast<uint8_t>(sbyte);
  }
}

// One thread per 32-bit word of the packed output: word w of atom a holds the
// scales of row m = 32*(w%4) + w/4 of the atom's 128-row band, micro-blocks
// 4*(a % groups) .. +3.  Out-of-range rows / blocks are written as zero.
__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t* __restrict__ sf, int64_t rows,
                                                          int64_t C, int64_t groups, int64_t nwords,
                                                          uint32_t* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nwords; i += stride) {
    const int64_t atom = i >> 7;
    const int w = static_cast<int>(i & 127);
    const int64_t band = atom / groups;
    const int64_t grp = atom - band * groups;
    const int64_t r = band * 128 + 32 * (w & 3) + (w >> 2);
    uint32_t v = 0;
    if (r < rows) {
      const uint8_t* src = sf + r * C + grp * 4;
      const int64_t c0 = grp * 4;
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (c0 + b < C) v |= static_cast<uint32_t>(src[b]) << (8 * b);
    }
    out[i] = v;
  }
}

int grid_for(int64_t work_items, int threads, const DeviceInfo& dev, int per_sm) {
  const int64_t need = (work_items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(dev.num_sms) * per_sm;
  return static_cast<int>(need < cap ? (need < 1 ? 1 : need) : cap);
}

}  // namespace

nvfp4_status launch_quantize(const void* x, int64_t rows, int64_t K, float g, uint8_t* codes, uint8_t* sf,
                             cudaStream_t stream, const DeviceInfo& dev) {
  const int64_t nblocks = rows * (K / 16);
  const int grid = grid_for(nblocks, 256, dev, 8);
  quantize_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(x), nblocks, g,
                                            reinterpret_cast<uint2*>(codes), sf);
  return from_cuda(cudaGetLastError());
}

nvfp4_status launch_pack_scales(const uint8_t* sf, int64_t rows, int64_t K, uint8_t* out, cudaStream_t stream,
                                const DeviceInfo& dev) {
  const int64_t C = K / 16;
  const int64_t groups = (C + 3) / 4;
  const int64_t bands = (rows + 127) / 128;
  const int64_t nwords = bands * groups * 128;
  const int grid = grid_for(nwords, 256, dev, 8);
  pack_scales_kernel<<<grid, 256, 0, stream>>>(sf, rows, C, groups, nwords, reinterpret_cast<uint32_t*>(out));
  return from_cuda(cudaGetLastError());
}

}  // namespace nvfp4

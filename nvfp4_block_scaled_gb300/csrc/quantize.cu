// quantize.cu -- NVFP4 operand producers: BF16 -> E2M1 codes + E4M3 block scales,
// and the row-major -> 128x4-atom scale-factor permutation.
//
// The kernels are HBM-bound.  Every quantiser takes one 16-element block per thread
// (coalesced 32-byte loads, 8-byte code stores) over a grid-stride loop sized to a
// multiple of the SM count; the fused and two-pass forms store each scale byte
// straight at its place in the packed layout.  pack_scales is a permutation of
// 32-bit words (each packed word is four consecutive scales of one row), done with
// one load and one coalesced store per word.

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

// The 16 floats of one block of bf16: v0, v1 = its 32 bytes.
__device__ __forceinline__ void unpack_bf16x16(uint4 v0, uint4 v1, float (&f)[16]) {
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// E2M1 codes of the IEEE quotients fl(f[o+i] / denom), i = 0..7, computed without a
// division per element.  r = 1/denom rounded once (IEEE), so q = fl(f * r) is within
// a relative 2^-23 of f / denom and fl(f / denom) within 2^-24 of it: the correctly
// rounded quotient lies strictly between fl(q * (1 - 2^-20)) and fl(q * (1 + 2^-20)).
// The E2M1 conversion is monotonic, so when both ends of that bracket give the same
// eight codes those are the codes of the quotients.  Otherwise (some element within a
// few ulp of a rounding midpoint) the word is recomputed from the IEEE divisions.
// Quotients too small to be normal floats lie far below the first midpoint (0.25) and
// give code 0 at both ends, as they do exactly.
__device__ __forceinline__ uint32_t codes_word(const float (&f)[16], int o, float r, float denom) {
  constexpr float kLo = 1.0f - 0x1p-20f, kHi = 1.0f + 0x1p-20f;
  float lo[8], hi[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float q = __fmul_rn(f[o + i], r);
    lo[i] = __fmul_rn(q, kLo);
    hi[i] = __fmul_rn(q, kHi);
  }
  const uint32_t a = e2m1x8(lo[0], lo[1], lo[2], lo[3], lo[4], lo[5], lo[6], lo[7]);
  const uint32_t b = e2m1x8(hi[0], hi[1], hi[2], hi[3], hi[4], hi[5], hi[6], hi[7]);
  if (a == b) return a;
  float e[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) e[i] = __fdiv_rn(f[o + i], denom);
  return e2m1x8(e[0], e[1], e[2], e[3], e[4], e[5], e[6], e[7]);
}

// Quantise one 16-element block of floats.  Returns the E4M3 scale byte and writes
// the 16 codes (little-endian nibbles) to *c0, *c1.
__device__ __forceinline__ uint32_t quantize_floats(const float (&f)[16], float g, uint32_t* c0_out,
                                                    uint32_t* c1_out) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const float s = __fdiv_rn(__fdiv_rn(amax, 6.0f), g);
  const uint32_t sbyte = __nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3);
  uint32_t c0 = 0, c1 = 0;
  if (sbyte != 0) {
    const float denom = __fmul_rn(e4m3_to_float(sbyte), g);
    const float r = __frcp_rn(denom);
    if (r <= 3.0e38f) {  // a finite reciprocal: products and a bracket (codes_word)
      c0 = codes_word(f, 0, r, denom);
      c1 = codes_word(f, 8, r, denom);
    } else {             // denom so small that 1/denom overflows: divide
      float q[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(f[i], denom);
      c0 = e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
      c1 = e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
    }
    // A code whose magnitude rounded to zero is written as +0 (clear its sign bit).
    const uint32_t nz0 = ((c0 & 0x77777777u) + 0x77777777u) & 0x88888888u;
    const uint32_t nz1 = ((c1 & 0x77777777u) + 0x77777777u) & 0x88888888u;
    c0 &= 0x77777777u | nz0;
    c1 &= 0x77777777u | nz1;
  }
  *c0_out = c0;
  *c1_out = c1;
  return sbyte;
}

// Quantise one 16-element block of bf16 (v0, v1 = its 32 bytes).
__device__ __forceinline__ uint32_t quantize_block(uint4 v0, uint4 v1, float g, uint32_t* c0_out,
                                                   uint32_t* c1_out) {
  float f[16];
  unpack_bf16x16(v0, v1, f);
  return quantize_floats(f, g, c0_out, c1_out);
}

// Residual of a quantised block: r_i = f_i - (value(code_i) * scale) * g, the product
// exact (at most 5 significant bits), the multiply by g and the subtraction each one
// IEEE float32 operation (no contraction).  value(code) * scale is formed without a
// per-code branch: the code's magnitude bits placed at float bits 22..24 and its sign
// at bit 31 give the float value(code) * 2^-126 (a subnormal for exponent field 0, as
// E2M1's own subnormal), which two exact multiplies (by 2^100, then by scale * 2^26)
// bring to value(code) * scale.
__device__ __forceinline__ void residual_block(const float (&f)[16], uint32_t c0, uint32_t c1, uint32_t sbyte,
                                               float g, float (&r)[16]) {
  const float sc26 = __fmul_rn(e4m3_to_float(sbyte), 67108864.0f);  // scale * 2^26, exact
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t nib = ((i < 8 ? c0 : c1) >> (4 * (i & 7))) & 0xFu;
    const float v126 = __uint_as_float(((nib & 7u) << 22) | ((nib & 8u) << 28));  // value * 2^-126
    const float vs = __fmul_rn(__fmul_rn(v126, 1.2676506002282294e30f), sc26);     // value * scale
    r[i] = __fsub_rn(f[i], __fmul_rn(vs, g));
  }
}

__global__ void __launch_bounds__(256) quantize_kernel(const uint4* __restrict__ x, int64_t nblocks,
                                                       float g, uint2* __restrict__ codes,
                                                       uint8_t* __restrict__ sf) {
  // x may be produced by the previous grid in the stream.  No early launch_dependents:
  // a following GEMM or W4A16 call reads its weights before waiting for this grid, so
  // this grid (which may be writing them) signals its dependents only by completing.
  griddep_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
    uint32_t c0, c1;
    const uint32_t sbyte = quantize_block(__ldcs(x + 2 * b), __ldcs(x + 2 * b + 1), g, &c0, &c1);
    __stcs(codes + b, make_uint2(c0, c1));
    sf[b] = static_cast<uint8_t>(sbyte);
  }
}

// ------------------------------------------------------------------ flat producers
//
// One 16-element block per thread over a grid-stride loop (the layout of
// quantize_kernel: a warp reads 1 KB of contiguous x), each scale byte stored straight
// at its place in the packed 128x4-atom layout.  The loop runs over the padded
// [bands * 128 rows] x [4 * groups columns] scale grid, so padding positions (rows
// past `rows`, columns past C) receive zero bytes and every byte of the packed buffer
// is written exactly once.  Byte b of the packed buffer for (row r, scale column c):
// ((r / 128 * groups + c / 4) * 128 + 4 * (r % 32) + (r % 128) / 32) * 4 + c % 4.
template <typename I>
__device__ __forceinline__ I packed_byte(I r, I c, I groups) {
  return (((r >> 7) * groups + (c >> 2)) * 128 + 4 * (r & 31) + ((r >> 5) & 3)) * 4 + (c & 3);
}

// I: the index type (uint32_t when the padded grid, and so the packed buffer, has
// fewer than 2^32 - 2^24 entries, so that no index passes 2^32 on the last stride).  The grid-stride loop advances (row, column) without a
// division per step.
template <typename I>
__global__ void __launch_bounds__(256) quantize_packed_flat_kernel(const uint4* __restrict__ x, int64_t rows,
                                                                   int64_t C, int64_t groups, int64_t total,
                                                                   float g, uint2* __restrict__ codes,
                                                                   uint8_t* __restrict__ sf_packed) {
  griddep_wait();  // x from the previous grid; dependents are signalled at completion (see quantize_kernel)
  const I Cp = static_cast<I>(4 * groups), Ci = static_cast<I>(C), Rows = static_cast<I>(rows);
  const I stride = static_cast<I>(gridDim.x) * blockDim.x;
  const I stride_r = stride / Cp, stride_c = stride - stride_r * Cp;
  const I v0 = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x;
  I r = v0 / Cp, c = v0 - r * Cp;
  for (I v = v0; v < static_cast<I>(total); v += stride) {
    uint32_t sbyte = 0;
    if (r < Rows && c < Ci) {
      const int64_t b = static_cast<int64_t>(r) * Ci + c;
      uint32_t c0, c1;
      sbyte = quantize_block(__ldcs(x + 2 * b), __ldcs(x + 2 * b + 1), g, &c0, &c1);
      __stcs(codes + b, make_uint2(c0, c1));
    }
    sf_packed[packed_byte<I>(r, c, static_cast<I>(groups))] = static_cast<uint8_t>(sbyte);
    r += stride_r;
    c += stride_c;
    if (c >= Cp) {
      c -= Cp;
      ++r;
    }
  }
}

// Two-pass quantisation, one source block per thread: block (r, c = 16 j + u) of x
// gives value codes at code block 32 j + u of row r's 2K codes and residual codes at
// 32 j + 16 + u, and its two scales at those columns of the packed [rows x 2K]
// operand (K % 256 == 0, so the scale columns need no padding; rows are padded to 128).
template <typename I>
__global__ void __launch_bounds__(256) quantize_two_pass_flat_kernel(const uint4* __restrict__ x, int64_t rows,
                                                                     int64_t C, int64_t total, float g,
                                                                     uint2* __restrict__ codes,
                                                                     uint8_t* __restrict__ sf_packed) {
  griddep_wait();  // x from the previous grid; dependents are signalled at completion (see quantize_kernel)
  const I Ci = static_cast<I>(C), Rows = static_cast<I>(rows), groups2 = static_cast<I>((2 * C) / 4);
  const I stride = static_cast<I>(gridDim.x) * blockDim.x;
  const I stride_r = stride / Ci, stride_c = stride - stride_r * Ci;
  const I v0 = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x;
  I r = v0 / Ci, c = v0 - r * Ci;
  for (I v = v0; v < static_cast<I>(total); v += stride) {
    const I cv = 2 * c - (c & 15);  // 32 j + u
    uint32_t s1 = 0, s2 = 0;
    if (r < Rows) {
      const int64_t b = static_cast<int64_t>(r) * Ci + c;
      float f[16];
      unpack_bf16x16(__ldcs(x + 2 * b), __ldcs(x + 2 * b + 1), f);
      uint32_t c0, c1, d0, d1;
      s1 = quantize_floats(f, g, &c0, &c1);
      float rf[16];
      residual_block(f, c0, c1, s1, g, rf);
      s2 = quantize_floats(rf, g, &d0, &d1);
      uint2* crow = codes + static_cast<int64_t>(r) * 2 * C;
      __stcs(crow + cv, make_uint2(c0, c1));
      __stcs(crow + cv + 16, make_uint2(d0, d1));
    }
    sf_packed[packed_byte<I>(r, cv, groups2)] = static_cast<uint8_t>(s1);
    sf_packed[packed_byte<I>(r, cv + 16, groups2)] = static_cast<uint8_t>(s2);
    r += stride_r;
    c += stride_c;
    if (c >= Ci) {
      c -= Ci;
      ++r;
    }
  }
}

// One thread block per (128-row band, 32 atoms): the band's 128 rows x 128 scale
// bytes are read row-major (coalesced 32-bit words) into shared memory, then
// written out atom by atom, each atom's 128 words contiguous.  Word w of an atom
// holds the four scales of row 32*(w%4) + w/4 of the band.  Rows past `rows` and
// scales past C are written as zero.  The tile is XOR-swizzled on the word column
// (by 8 * (row / 32)) so both the row-wise writes and the atom-wise reads of
// shared memory are free of bank conflicts.
constexpr int kPackAtoms = 32;
constexpr int kPackPitch = kPackAtoms + 1;  // words per tile row

__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t* __restrict__ sf, int64_t rows,
                                                          int64_t C, int64_t groups, int64_t tiles_per_band,
                                                          int64_t num_tiles, bool word_loads,
                                                          uint32_t* __restrict__ out) {
  __shared__ uint32_t tile[128 * kPackPitch];
  griddep_wait();  // x from the previous grid; dependents are signalled at completion (see quantize_kernel)
  for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
    const int64_t band = t / tiles_per_band;
    const int64_t g0 = (t - band * tiles_per_band) * kPackAtoms;
    const int ng = static_cast<int>(groups - g0 < kPackAtoms ? groups - g0 : kPackAtoms);
    // Thread (row0 = tid / 32, gw = tid % 32) loads rows row0 + 8k, k = 0..15, of
    // word column gw: sixteen independent loads in flight per thread.
    const int gw = threadIdx.x % kPackAtoms;
    const int row0 = threadIdx.x / kPackAtoms;
    const int64_t c0 = 4 * (g0 + gw);
    const bool col_ok = gw < ng;
    if (word_loads && col_ok && c0 + 4 <= C && band * 128 + 128 <= rows) {
      const uint8_t* src = sf + (band * 128 + row0) * C + c0;
      uint32_t v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = __ldg(reinterpret_cast<const uint32_t*>(src + 8 * k * C));
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int row = row0 + 8 * k;
        tile[row * kPackPitch + (gw ^ (8 * (row >> 5)))] = v[k];
      }
    } else {
#pragma unroll 1
      for (int k = 0; k < 16; ++k) {
        const int row = row0 + 8 * k;
        const int64_t r = band * 128 + row;
        uint32_t w = 0;
        if (col_ok && r < rows) {
          const uint8_t* src = sf + r * C + c0;
          for (int b = 0; b < 4; ++b)
            if (c0 + b < C) w |= static_cast<uint32_t>(src[b]) << (8 * b);
        }
        tile[row * kPackPitch + (gw ^ (8 * (row >> 5)))] = w;
      }
    }
    __syncthreads();
    uint32_t* dst = out + (band * groups + g0) * 128;
    for (int i = threadIdx.x; i < ng * 128; i += blockDim.x) {
      const int a = i >> 7, w = i & 127;
      const int row = 32 * (w & 3) + (w >> 2);
      dst[i] = tile[row * kPackPitch + (a ^ (8 * (row >> 5)))];
    }
    __syncthreads();
  }
}

// Launch configuration with programmatic dependent launch allowed (the kernels wait
// for the previous grid in the stream before touching memory).
cudaLaunchConfig_t programmatic_config(int grid, int threads, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  return cfg;
}

void set_programmatic(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[1]) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

int grid_for(int64_t work_items, int threads, const DeviceInfo& dev, int per_sm) {
  const int64_t need = (work_items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(dev.num_sms) * per_sm;
  return static_cast<int>(need < cap ? (need < 1 ? 1 : need) : cap);
}

}  // namespace

nvfp4_status launch_quantize(const void* x, int64_t rows, int64_t K, float g, uint8_t* codes, uint8_t* sf,
                             bool packed, cudaStream_t stream, const DeviceInfo& dev) {
  const int64_t C = K / 16;
  cudaLaunchAttribute attr[1];
  if (!packed) {
    const int64_t nblocks = rows * C;
    cudaLaunchConfig_t cfg = programmatic_config(grid_for(nblocks, 256, dev, 8), 256, stream);
    set_programmatic(cfg, attr);
    return from_cuda(cudaLaunchKernelEx(&cfg, quantize_kernel, static_cast<const uint4*>(x), nblocks, g,
                                        reinterpret_cast<uint2*>(codes), sf));
  }
  const int64_t groups = (C + 3) / 4;
  const int64_t total = ((rows + 127) / 128) * 128 * (4 * groups);  // padded scale grid
  cudaLaunchConfig_t cfg = programmatic_config(grid_for(total, 256, dev, 8), 256, stream);
  set_programmatic(cfg, attr);
  if (total < (int64_t(1) << 32) - (int64_t(1) << 24))
    return from_cuda(cudaLaunchKernelEx(&cfg, quantize_packed_flat_kernel<uint32_t>, static_cast<const uint4*>(x),
                                        rows, C, groups, total, g, reinterpret_cast<uint2*>(codes), sf));
  return from_cuda(cudaLaunchKernelEx(&cfg, quantize_packed_flat_kernel<int64_t>, static_cast<const uint4*>(x), rows,
                                      C, groups, total, g, reinterpret_cast<uint2*>(codes), sf));
}

nvfp4_status launch_quantize_two_pass(const void* x, int64_t rows, int64_t K, float g, uint8_t* codes,
                                      uint8_t* sf_packed, cudaStream_t stream, const DeviceInfo& dev) {
  const int64_t C = K / 16;
  const int64_t total = ((rows + 127) / 128) * 128 * C;  // rows padded to whole bands
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = programmatic_config(grid_for(total, 256, dev, 8), 256, stream);
  set_programmatic(cfg, attr);
  if (total < (int64_t(1) << 32) - (int64_t(1) << 24))
    return from_cuda(cudaLaunchKernelEx(&cfg, quantize_two_pass_flat_kernel<uint32_t>, static_cast<const uint4*>(x),
                                        rows, C, total, g, reinterpret_cast<uint2*>(codes), sf_packed));
  return from_cuda(cudaLaunchKernelEx(&cfg, quantize_two_pass_flat_kernel<int64_t>, static_cast<const uint4*>(x),
                                      rows, C, total, g, reinterpret_cast<uint2*>(codes), sf_packed));
}

nvfp4_status launch_pack_scales(const uint8_t* sf, int64_t rows, int64_t K, uint8_t* out, cudaStream_t stream,
                                const DeviceInfo& dev) {
  const int64_t C = K / 16;
  const int64_t groups = (C + 3) / 4;
  const int64_t bands = (rows + 127) / 128;
  const bool word_loads = (C % 4 == 0) && aligned(sf, 4);
  const int64_t tiles_per_band = (groups + kPackAtoms - 1) / kPackAtoms;
  const int64_t num_tiles = bands * tiles_per_band;
  const int grid = grid_for(num_tiles * 256, 256, dev, 8);
  cudaLaunchConfig_t cfg = programmatic_config(grid, 256, stream);
  cudaLaunchAttribute attr[1];
  set_programmatic(cfg, attr);
  return from_cuda(cudaLaunchKernelEx(&cfg, pack_scales_kernel, sf, rows, C, groups, tiles_per_band, num_tiles,
                                      word_loads, reinterpret_cast<uint32_t*>(out)));
}

}  // namespace nvfp4

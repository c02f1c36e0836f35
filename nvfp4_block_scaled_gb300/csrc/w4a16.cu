// w4a16.cu -- BF16 activations x NVFP4 weights (TileLang PR #3290, "SM120 W4A16
// NVFP4 GEMM example for decode-sized batches": Summary and Design), for sm_103a.
//
// prepare: re-lays out codes + E4M3 scales once into 576-byte blocks (16 weight
//   rows x 64 K) in the fragment order of mma.m16n8k16 with the WEIGHT as the
//   A operand (16 rows of N); codes are bit-placed so that one AND (and a shift)
//   yields bf16x2 values fp4 * 2^-126, scales re-encoded as b with
//   bf16(0x7000 | b<<4) = |scale| * 2^119; zero scales zero their codes, negative
//   scales flip the code signs.  One bf16x2 multiply then gives w * 2^-7 exactly.
// linear (decode, M <= 64 per pass): a thread block cluster of S CTAs splits K;
//   each CTA stages its slice of x in shared memory, its 8 warps stream one
//   16-row weight tile each straight from HBM into registers (16-byte loads,
//   several blocks in flight), dequantise, and issue mma.sync with FP32
//   accumulation; partial sums are reduced across the cluster through
//   distributed shared memory in a fixed order (deterministic, no workspace),
//   then y = bf16(acc * alpha * 2^7).

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kBlockBytes = 576;  // 16 rows x 64 K: 512 bytes of codes + 64 scale bytes

// ------------------------------------------------------------------ prepare

__device__ __forceinline__ uint32_t reencode_scale(uint32_t mag) {
  if (mag == 0) return 0;
  const uint32_t e = mag >> 3, m = mag & 7;
  if (e != 0) return ((e + 15u) << 3) | m;
  const uint32_t p = 31u - __clz(m);  // floor(log2 m), m in 1..7
  return ((p + 13u) << 3) | ((m << (3u - p)) & 7u);
}

// code nibble of element (row, k) after folding the block scale's sign / zero
__device__ __forceinline__ uint32_t folded_code(const uint8_t* W, const uint8_t* SW, int64_t row, int64_t k,
                                                int64_t K) {
  const uint32_t byte = W[row * (K / 2) + (k >> 1)];
  uint32_t c = (k & 1) ? (byte >> 4) : (byte & 0xF);
  const uint32_t s = SW[row * (K / 16) + (k >> 4)];
  if ((s & 0x7F) == 0) return 0;
  if (s & 0x80) c ^= 8;
  return c;
}

__global__ void __launch_bounds__(256) w4a16_prepare_kernel(const uint8_t* __restrict__ W,
                                                            const uint8_t* __restrict__ SW, int64_t N, int64_t K,
                                                            uint8_t* __restrict__ out) {
  const int64_t KC = K / 64;
  const int64_t total = (N / 16) * KC * 32;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int lane = static_cast<int>(i & 31);
    const int64_t blk = i >> 5;
    const int64_t nt = blk / KC, kc = blk - (blk / KC) * KC;
    const int g = lane >> 2, t = lane & 3;
    const int64_t r0 = nt * 16 + g, r1 = r0 + 8;
    uint32_t words[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t k0 = kc * 64 + 16 * j + 2 * t;
      const uint32_t a0 = folded_code(W, SW, r0, k0, K), a1 = folded_code(W, SW, r0, k0 + 1, K);
      const uint32_t a2 = folded_code(W, SW, r1, k0, K), a3 = folded_code(W, SW, r1, k0 + 1, K);
      const uint32_t a4 = folded_code(W, SW, r0, k0 + 8, K), a5 = folded_code(W, SW, r0, k0 + 9, K);
      const uint32_t a6 = folded_code(W, SW, r1, k0 + 8, K), a7 = folded_code(W, SW, r1, k0 + 9, K);
      uint32_t w = 0;
      w |= ((a0 & 7u) << 6) | ((a0 >> 3) << 15);
      w |= ((a1 & 7u) << 22) | ((a1 >> 3) << 31);
      w |= ((a2 & 7u) << 3) | ((a2 >> 3) << 12);
      w |= ((a3 & 7u) << 19) | ((a3 >> 3) << 28);
      w |= (a4 & 7u) | ((a4 >> 3) << 9);
      w |= ((a5 & 7u) << 16) | ((a5 >> 3) << 25);
      w |= ((a6 & 3u) << 10) | (((a6 >> 2) & 1u) << 13) | ((a6 >> 3) << 14);
      w |= ((a7 & 3u) << 26) | (((a7 >> 2) & 1u) << 29) | ((a7 >> 3) << 30);
      words[j] = w;
    }
    uint8_t* dst = out + blk * kBlockBytes;
    *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(words[0], words[1], words[2], words[3]);
    if (t == 0) {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t sa = SW[r0 * (K / 16) + kc * 4 + j] & 0x7F;
        const uint32_t sb = SW[r1 * (K / 16) + kc * 4 + j] & 0x7F;
        const uint32_t pair = reencode_scale(sa) | (reencode_scale(sb) << 8);
        if (j < 2) lo |= pair << (16 * j); else hi |= pair << (16 * (j - 2));
      }
      *reinterpret_cast<uint2*>(dst + 512 + 8 * g) = make_uint2(lo, hi);
    }
  }
}

// ------------------------------------------------------------------ linear (decode)

__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Dequantise one word (8 codes) into the 4 A-fragment registers, times the
// row scales (s_lo for rows g, s_hi for rows g+8, both bf16x2 {s, s}).
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s_lo, uint32_t s_hi, uint32_t (&a)[4]) {
  constexpr uint32_t kMask = 0x81C081C0u;
  const uint32_t r0 = w & kMask;
  const uint32_t r1 = (w << 3) & kMask;
  const uint32_t r2 = (w << 6) & kMask;
  const uint32_t r3 = ((w >> 4) & 0x00C000C0u) | ((w >> 5) & 0x01000100u) | ((w << 1) & 0x80008000u);
  a[0] = hmul2_bf16(r0, s_lo);
  a[1] = hmul2_bf16(r1, s_hi);
  a[2] = hmul2_bf16(r2, s_lo);
  a[3] = hmul2_bf16(r3, s_hi);
}

// bf16x2 {S, S} with S = 0x7000 | b << 4 for the scale byte b at byte index `idx` of `word`.
__device__ __forceinline__ uint32_t scale_pair(uint32_t word, int idx) {
  const uint32_t b = (word >> (8 * idx)) & 0xFFu;
  return b * 0x00100010u + 0x70007000u;
}

constexpr int kDecodeWarps = 8;
constexpr int kPF = 4;  // weight blocks in flight per warp

template <int MT>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    w4a16_decode_kernel(const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ wprep, float alpha128,
                        __nv_bfloat16* __restrict__ y, int M, int N, int K, int S) {
  constexpr int Mpad = 8 * MT;
  extern __shared__ __align__(16) uint8_t smem[];
  const int rank = blockIdx.x;  // position in the cluster = K split index
  const int ng = blockIdx.y;    // 128-row group of N
  const int KC = K / 64;
  const int kc_per = KC / S;
  const int kc0 = rank * kc_per;
  const int Kr = kc_per * 64;
  const int pitch = Kr + 8;  // elements; +16 bytes keeps fragment loads conflict-free
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);
  float* part = reinterpret_cast<float*>(smem + static_cast<size_t>(Mpad) * pitch * 2);  // [Mpad][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nt = ng * kDecodeWarps + warp;
  const uint8_t* wp = wprep + (static_cast<size_t>(nt) * KC + kc0) * kBlockBytes;

  // Start the weight stream before waiting for x.
  uint4 cw[kPF];
  uint2 sw[kPF];
#pragma unroll
  for (int p = 0; p < kPF; ++p) {
    if (p < kc_per) {
      cw[p] = ldg_stream(wp + p * kBlockBytes + 16 * lane);
      sw[p] = ldg_stream2(wp + p * kBlockBytes + 512 + 8 * g);
    }
  }

  // Stage x[0:Mpad, kc0*64 : kc0*64 + Kr] (rows >= M zero-filled).
  const int chunks_per_row = Kr / 8;
  const uint32_t xs_base = smem_u32(xs);
  for (int c = threadIdx.x; c < Mpad * chunks_per_row; c += blockDim.x) {
    const int r = c / chunks_per_row, q = c - r * chunks_per_row;
    const int rr = r < M ? r : 0;
    const __nv_bfloat16* src = x + static_cast<size_t>(rr) * K + static_cast<size_t>(kc0) * 64 + q * 8;
    cp_async16(xs_base + (r * pitch + q * 8) * 2, src, r < M ? 16u : 0u);
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  const uint32_t* xw = reinterpret_cast<const uint32_t*>(xs);
  const int pitch_w = pitch / 2;  // in 32-bit words

#pragma unroll 1
  for (int kc = 0; kc < kc_per; kc += kPF) {
#pragma unroll
    for (int p = 0; p < kPF; ++p) {
      if (kc + p < kc_per) {
        const uint4 c = cw[p];
        const uint2 s = sw[p];
        if (kc + p + kPF < kc_per) {
          cw[p] = ldg_stream(wp + (kc + p + kPF) * kBlockBytes + 16 * lane);
          sw[p] = ldg_stream2(wp + (kc + p + kPF) * kBlockBytes + 512 + 8 * g);
        }
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t sword = j < 2 ? s.x : s.y;
          const uint32_t s_lo = scale_pair(sword, (j & 1) * 2);
          const uint32_t s_hi = scale_pair(sword, (j & 1) * 2 + 1);
          uint32_t a[4];
          dequant_word(words[j], s_lo, s_hi, a);
          const int kw = ((kc + p) * 64 + 16 * j) / 2 + t;  // word column of k = 2t
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t* row = xw + (8 * mt + g) * pitch_w;
            mma_bf16_16816(acc[mt], a, row[kw], row[kw + 4]);
          }
        }
      }
    }
  }

  // Partial sums -> shared memory as part[token][row in group].
  const int rbase = warp * 16 + g;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int tok = 8 * mt + 2 * t;
    part[tok * 128 + rbase] = acc[mt][0];
    part[(tok + 1) * 128 + rbase] = acc[mt][1];
    part[tok * 128 + rbase + 8] = acc[mt][2];
    part[(tok + 1) * 128 + rbase + 8] = acc[mt][3];
  }
  cluster_sync_all();

  // Fixed-order reduction over the cluster: this CTA finalises rows
  // [rank*128/S, (rank+1)*128/S) of the group for every real token.
  const int rows_per = 128 / S;
  const uint32_t part_base = smem_u32(part);
  for (int idx = threadIdx.x; idx < rows_per * M; idx += blockDim.x) {
    const int tok = idx / rows_per;
    const int row = rank * rows_per + (idx - tok * rows_per);
    const uint32_t off = part_base + static_cast<uint32_t>(tok * 128 + row) * 4u;
    float sum = 0.f;
    for (int src = 0; src < S; ++src) sum += ld_dsmem_f32(off, static_cast<uint32_t>(src));
    y[static_cast<size_t>(tok) * N + static_cast<size_t>(ng) * 128 + row] = __float2bfloat16_rn(sum * alpha128);
  }
  cluster_sync_all();
}

size_t decode_smem_bytes(int MT, int K, int S) {
  const int Kr = K / S;
  return static_cast<size_t>(8 * MT) * (Kr + 8) * 2 + static_cast<size_t>(8 * MT) * 128 * 4;
}

template <int MT>
nvfp4_status launch_decode(const __nv_bfloat16* x, const uint8_t* wprep, float alpha128, __nv_bfloat16* y, int M,
                           int N, int K, int S, cudaStream_t stream) {
  auto kern = w4a16_decode_kernel<MT>;
  const size_t smem = decode_smem_bytes(MT, K, S);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return NVFP4_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, N / 128, 1);
  cfg.blockDim = dim3(kDecodeWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return from_cuda(cudaLaunchKernelEx(&cfg, kern, x, wprep, alpha128, y, M, N, K, S));
}

}  // namespace

int read_device_error_w4a16(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (clear && v != 0) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_device_error, &z, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  return v;
}

nvfp4_status launch_w4a16_prepare(const uint8_t* W, const uint8_t* SW, int64_t N, int64_t K, void* Wprep,
                                  cudaStream_t stream, const DeviceInfo& dev) {
  const int64_t total = (N / 16) * (K / 64) * 32;
  int64_t grid = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
  if (grid > cap) grid = cap;
  w4a16_prepare_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(W, SW, N, K, static_cast<uint8_t*>(Wprep));
  return from_cuda(cudaGetLastError());
}

nvfp4_status launch_w4a16_linear(const void* x, const void* Wprep, float alpha, void* y, int64_t M, int64_t N,
                                 int64_t K, cudaStream_t stream, const DeviceInfo& dev) {
  const float alpha128 = alpha * 128.0f;
  const int KC = static_cast<int>(K / 64);
  const int groups = static_cast<int>(N / 128);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* yb = static_cast<__nv_bfloat16*>(y);
  const auto* wp = static_cast<const uint8_t*>(Wprep);
  // Largest token chunk (64, 32, 16 or 8 rows) whose slice of x fits in shared
  // memory at the deepest K split.
  int chunk = 64;
  while (chunk > 8 && (KC % 8 != 0 || decode_smem_bytes(chunk / 8, static_cast<int>(K), 8) > dev.max_smem_optin))
    chunk /= 2;
  for (int64_t m0 = 0; m0 < M; m0 += chunk) {
    const int mc = static_cast<int>(M - m0 < chunk ? M - m0 : chunk);
    const int MT = mc <= 8 ? 1 : mc <= 16 ? 2 : mc <= 32 ? 4 : 8;
    // K split: enough CTAs for about two waves, a slice of x that fits in shared memory.
    int S = 1;
    while (S < 8 && KC % (2 * S) == 0 &&
           (static_cast<int64_t>(groups) * S < 2LL * dev.num_sms ||
            decode_smem_bytes(MT, static_cast<int>(K), S) > 100 * 1024))
      S *= 2;
    if (decode_smem_bytes(MT, static_cast<int>(K), S) > dev.max_smem_optin) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    const __nv_bfloat16* xc = xb + m0 * K;
    __nv_bfloat16* yc = yb + m0 * N;
    nvfp4_status st;
    switch (MT) {
      case 1: st = launch_decode<1>(xc, wp, alpha128, yc, mc, static_cast<int>(N), static_cast<int>(K), S, stream); break;
      case 2: st = launch_decode<2>(xc, wp, alpha128, yc, mc, static_cast<int>(N), static_cast<int>(K), S, stream); break;
      case 4: st = launch_decode<4>(xc, wp, alpha128, yc, mc, static_cast<int>(N), static_cast<int>(K), S, stream); break;
      default: st = launch_decode<8>(xc, wp, alpha128, yc, mc, static_cast<int>(N), static_cast<int>(K), S, stream); break;
    }
    if (st != NVFP4_OK) return st;
  }
  return NVFP4_OK;
}

}  // namespace nvfp4

// w4a16.cu -- BF16 activations x NVFP4 weights (TileLang PR #3290, "SM120 W4A16
// NVFP4 GEMM example for decode-sized batches": Summary and Design), for sm_103a.
//
// prepare: re-lays out codes + E4M3 scales once into 576-byte blocks (16 weight
//   rows x 64 K) in the fragment order of mma.m16n8k16 with the WEIGHT as the
//   A operand (16 rows of N); codes are bit-placed so that one AND (and a shift)
//   yields bf16x2 values fp4 * 2^-126, scales re-encoded as b with
//   bf16(0x7000 | b<<4) = |scale| * 2^119; zero scales zero their codes, negative
//   scales flip the code signs.  One bf16x2 multiply then gives w * 2^-7 exactly.
// linear, more than 32 tokens: weights dequantised into shared memory, tcgen05
//   kind::f16 MMAs with the tokens as the N dimension (see the tensor-core section).
// linear, up to 32 tokens (decode): a thread block cluster of S CTAs
//   splits K; each CTA owns 128 weight rows and a contiguous range of 512-wide K
//   chunks.  A producer warp streams each chunk (36 KB of weights: 8 n-tiles x
//   8 blocks, contiguous per n-tile) together with the matching x columns
//   (Mpad tokens x 512 K, 128-byte swizzled, zero rows past M) with 3-D TMA boxes
//   into a 2-deep ring -- large copies are what keep HBM busy; per-warp 16-byte
//   loads top out far below it.  Sixteen consumer warps (an n-tile and half of each
//   chunk's blocks each) dequantise from shared memory and issue mma.sync with
//   FP32 accumulation, x fragments from ldmatrix.  Partial sums (the drained ring
//   holds them) are reduced across the cluster through distributed shared memory in
//   a fixed order (deterministic, no workspace), then y = bf16(acc * alpha * 2^7).

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "sk_units.h"
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
      // (magnitude bits 0-2, sign) of a0..a5 at (p, p+1, p+2, q); a6 and a7 at
      // (4, 0, 1, 3) and (20, 16, 17, 19) -- the order dequant_word undoes.
      uint32_t w = 0;
      w |= ((a0 & 7u) << 6) | ((a0 >> 3) << 15);
      w |= ((a1 & 7u) << 22) | ((a1 >> 3) << 31);
      w |= ((a2 & 7u) << 28) | ((a2 >> 3) << 5);
      w |= ((a3 & 7u) << 12) | ((a3 >> 3) << 21);
      w |= ((a4 & 7u) << 25) | ((a4 >> 3) << 2);
      w |= ((a5 & 7u) << 9) | ((a5 >> 3) << 18);
      const uint32_t lo6 = ((a6 & 1u) << 4) | ((a6 >> 1) & 3u) | ((a6 >> 3) << 3);
      const uint32_t lo7 = ((a7 & 1u) << 4) | ((a7 >> 1) & 3u) | ((a7 >> 3) << 3);
      w |= lo6 | (lo7 << 16);
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

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Remote (distributed shared memory) load; ordered after the preceding cluster
// barrier by that barrier's own memory clobber.
__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
  return v;
}

// Multipliers of the register dequant, kept in constant memory so that the compiler
// issues them as integer multiplies (FMA pipe) rather than as shift-add sequences
// and LEAs, which share the ALU pipe with the masks, rotations and byte permutes.
__constant__ uint32_t c_deq_mul[2] = {0x1084u, 16u};

// a * {s.lo, s.lo} and a * {s.hi, s.hi} (bf16x2, round to nearest even)
__device__ __forceinline__ uint32_t hmul2_lo(uint32_t a, uint32_t s) {
  uint32_t d;
  asm("{.reg .b16 l, h; .reg .b32 t; mov.b32 {l, h}, %2; mov.b32 t, {l, l}; mul.rn.bf16x2 %0, %1, t;}"
      : "=r"(d) : "r"(a), "r"(s));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_hi(uint32_t a, uint32_t s) {
  uint32_t d;
  asm("{.reg .b16 l, h; .reg .b32 t; mov.b32 {l, h}, %2; mov.b32 t, {h, h}; mul.rn.bf16x2 %0, %1, t;}"
      : "=r"(d) : "r"(a), "r"(s));
  return d;
}

// Dequantise one word (8 codes) into the 4 A-fragment registers, times the row
// scales s2 = bf16x2 {S(row g), S(row g+8)}.  The mask keeps bits 6-8 and 15 of each
// half (mantissa MSB, the two low exponent bits, sign): a code lands as the bf16
// fp4 * 2^-126.  Registers 1 and 2 are rotations of w by 10 and 13; register 3
// multiplies the masked word by 2^2 + 2^7 + 2^12, three copies that share no bit, so
// the sum never carries.  8 integer operations per word.  (Rotations as widening
// multiplies measured slower: 17.6 against 15.8 us for a 17408 x 5120 decode.)
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s2, uint32_t (&a)[4]) {
  constexpr uint32_t kMask = 0x81C081C0u;
  const uint32_t r0 = w & kMask;
  const uint32_t r1 = __funnelshift_l(w, w, 10) & kMask;
  const uint32_t r2 = __funnelshift_l(w, w, 13) & kMask;
  const uint32_t r3 = ((w & 0x001B001Bu) * c_deq_mul[0]) & kMask;
  a[0] = hmul2_lo(r0, s2);
  a[1] = hmul2_hi(r1, s2);
  a[2] = hmul2_lo(r2, s2);
  a[3] = hmul2_hi(r3, s2);
}

// The scale pair of word j of a block: bf16x2 {S(g), S(g+8)} with S = 0x7000 | b << 4
// for the bytes b of rows g and g+8 at bytes 2 (j & 1) and 2 (j & 1) + 1 of `word`
// (the scale word of j < 2 or of j >= 2): one byte permute ({b_g, 0, b_g8, 0}) and
// one multiply-add.
__device__ __forceinline__ uint32_t scale_pair(uint32_t word, int j) {
  const uint32_t v = __byte_perm(word, 0u, static_cast<uint32_t>(j & 1) * 0x0202u + 0x4140u);
  return v * c_deq_mul[1] + 0x70007000u;
}

constexpr int kDecodeNT = 8;                    // 16-row n-tiles per CTA (128 rows)
constexpr int kDecodeWarps = 16;                // consumer warps: n-tile w % 8, chunk half w / 8
constexpr int kDecodeThreads = 32 * (kDecodeWarps + 1);  // + one producer warp
constexpr int kChunkKC = 8;                     // 64-wide K blocks per chunk (K = 512)
constexpr int kChunkBytes = kDecodeNT * kChunkKC * kBlockBytes;  // 36 KB: 128 rows x 512 K
constexpr int kRing = 2;                        // chunks in flight per CTA
constexpr int kDecodeMaxTokens = 32;            // tokens per launch

// One ring stage: the weight chunk, then x[Mpad tokens][512 K] as 8 K-blocks of
// [Mpad][128 B] (128-byte swizzled; tokens past M are zero-filled by the copy).
// After the main loop the ring is reused for the partial sums [2 halves][Mpad][128].
__host__ __device__ constexpr int decode_stage_bytes(int Mpad) { return kChunkBytes + Mpad * 1024; }
__host__ __device__ constexpr int decode_bar_off(int Mpad) { return kRing * decode_stage_bytes(Mpad); }
// + 1 KB so the kernel can align its base to the 1024 bytes the swizzle needs.
__host__ __device__ constexpr int decode_smem_bytes(int Mpad) { return decode_bar_off(Mpad) + 2 * kRing * 8 + 16 + 1024; }
static_assert(2 * kDecodeMaxTokens * 128 * 4 <= kRing * kChunkBytes, "partial sums fit in the ring");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Thread blocks per SM the register budget allows: two for up to 16 tokens.
template <int MT>
constexpr int decode_min_blocks() { return MT <= 2 ? 2 : 1; }

// Weight stream: the prepared weight viewed as a 3-D tensor
// [N/16 n-tiles][K/64 blocks][576 bytes]; one TMA box = 8 n-tiles x 8 blocks (36 KB),
// i.e. 128 rows x 512 K, landing in shared memory as [n-tile][block][576 B].
// Activation stream: x viewed as [K/64 blocks][M tokens][64 bf16]; one box =
// 8 blocks x Mpad tokens, so each stage carries the x columns its chunk needs.
template <int MT>
__global__ void __launch_bounds__(kDecodeThreads, decode_min_blocks<MT>())
    w4a16_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        float alpha128, const float* __restrict__ alpha_col, __nv_bfloat16* __restrict__ y, int M,
                        int N, int K, int S) {
  constexpr int Mpad = 8 * MT;
  constexpr int kStage = decode_stage_bytes(Mpad);
  constexpr int kStageTx = kStage;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));
  const int rank = blockIdx.x;  // position in the cluster = K split index
  const int grp = blockIdx.y;   // 128-row group of N
  const int KC = K / 64;
  const int C = (KC + kChunkKC - 1) / kChunkKC;
  const int c0 = rank * C / S, c1 = (rank + 1) * C / S;
  const int nch = c1 - c0;
  const uint32_t ring = sbase;
  float* part = reinterpret_cast<float*>(smem);  // [2][Mpad][128], valid after the main loop
  const uint32_t bar_full = sbase + decode_bar_off(Mpad);
  const uint32_t bar_empty = bar_full + 8 * kRing;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + decode_bar_off(Mpad) + 16 * kRing);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kDecodeWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The next call in the stream may start its weight stream now (see below).
  griddep_launch_dependents();

  if (warp == kDecodeWarps) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0) {
      prefetch_tensormap(&tmW);
      prefetch_tensormap(&tmX);
      auto load_w = [&](int i) {
        const int st = i % kRing;
        mbar_arrive_expect_tx(bar_full + 8 * st, kStageTx);
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(ring + st * kStage),
            "l"(&tmW), "r"(0), "r"((c0 + i) * kChunkKC), "r"(grp * kDecodeNT), "r"(bar_full + 8 * st)
            : "memory");
      };
      auto load_x = [&](int i) {
        const int st = i % kRing;
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(ring + st * kStage + kChunkBytes),
            "l"(&tmX), "r"(0), "r"(0), "r"((c0 + i) * kChunkKC), "r"(bar_full + 8 * st)
            : "memory");
      };
      // The weights never depend on an earlier kernel: the first ring stages' chunks
      // are requested before waiting for the previous grid in the stream, which may
      // be producing x (with programmatic launch this overlaps its tail).
      const int npre = nch < kRing ? nch : kRing;
      for (int i = 0; i < npre; ++i) load_w(i);
      griddep_wait();
      for (int i = 0; i < npre; ++i) load_x(i);
      for (int i = npre; i < nch; ++i) {
        const int st = i % kRing;
        if (!mbar_wait(bar_empty + 8 * st, ((i / kRing) - 1) & 1, abort_flag)) break;
        load_w(i);
        load_x(i);
      }
      // Let every issued copy land before the thread block can exit.
      for (int i = nch > kRing ? nch - kRing : 0; i < nch; ++i)
        mbar_wait_for(bar_full + 8 * (i % kRing), (i / kRing) & 1, 2000000000ull);
    }
  } else {
    // ------------------------------------------------------------ consumer warps
    // Start the (time-limited) barrier waits only once the previous grid is done.
    griddep_wait();
    const int nt = warp & (kDecodeNT - 1);  // n-tile within the group
    const int half = warp / kDecodeNT;      // which half of each chunk's blocks
    const int g = lane >> 2;
    // ldmatrix rows: lane l supplies token 8mt + l%8 of matrix l/8, i.e. the 16-byte
    // piece 4jj + l/8 of the token's 128-byte line, stored at piece ^ (token % 8).
    const uint32_t row_off = static_cast<uint32_t>(lane & 7) * 128u;
    const uint32_t sw = static_cast<uint32_t>(lane & 7);
    const uint32_t q = static_cast<uint32_t>(lane >> 3);

    float acc[2][MT][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) acc[a][mt][0] = acc[a][mt][1] = acc[a][mt][2] = acc[a][mt][3] = 0.f;

    for (int i = 0; i < nch; ++i) {
      const int st = i % kRing;
      // (vote wait: 1-2 % faster than lane 0 waiting with try_wait, measured)
      if (!warp_wait_vote(bar_full + 8 * st, (i / kRing) & 1, abort_flag)) break;
      const int kcc = min(kChunkKC, KC - (c0 + i) * kChunkKC);
      const int kb0 = half * (kChunkKC / 2);
      const int kb1 = min(kcc, kb0 + kChunkKC / 2);
      const uint32_t stage = ring + st * kStage;
      const uint32_t tile = stage + nt * (kChunkKC * kBlockBytes);
      const uint32_t xstage = stage + kChunkBytes + row_off;
      auto do_block = [&](int kc) {
        const uint32_t blk = tile + kc * kBlockBytes;
        uint4 c;
        uint2 sc;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(c.x), "=r"(c.y), "=r"(c.z), "=r"(c.w)
                     : "r"(blk + 16 * lane));
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(sc.x), "=r"(sc.y) : "r"(blk + 512 + 8 * g));
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
        const uint32_t xblk = xstage + static_cast<uint32_t>(kc * Mpad * 128);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {  // two pairs of 16-wide K steps
          uint32_t b[MT][4];
          const uint32_t piece = ((4u * jj + q) ^ sw) * 16u;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) ldsm_x4(xblk + mt * 1024 + piece, b[mt][0], b[mt][1], b[mt][2], b[mt][3]);
#pragma unroll
          for (int j2 = 0; j2 < 2; ++j2) {
            const int j = 2 * jj + j2;
            const uint32_t sword = j < 2 ? sc.x : sc.y;
            uint32_t a[4];
            dequant_word(words[j], scale_pair(sword, j), a);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) mma_bf16_16816(acc[j2][mt], a, b[mt][2 * j2], b[mt][2 * j2 + 1]);
          }
        }
      };
      if (kb1 - kb0 == kChunkKC / 2) {
        // a whole half chunk: unrolled (no loop branch, loads of the next block in flight)
#pragma unroll
        for (int u = 0; u < kChunkKC / 2; ++u) do_block(kb0 + u);
      } else {
#pragma unroll 1
        for (int kc = kb0; kc < kb1; ++kc) do_block(kc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }
    // All consumers are done with the ring (every copy they waited for has landed);
    // reuse it for the partial sums part[half][token][row in group].
    named_bar_sync(1, 32 * kDecodeWarps);
    float* ph = part + half * Mpad * 128;
    const int rbase = nt * 16 + g;
    const int t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int tok = 8 * mt + 2 * t;
      ph[tok * 128 + rbase] = acc[0][mt][0] + acc[1][mt][0];
      ph[(tok + 1) * 128 + rbase] = acc[0][mt][1] + acc[1][mt][1];
      ph[tok * 128 + rbase + 8] = acc[0][mt][2] + acc[1][mt][2];
      ph[(tok + 1) * 128 + rbase + 8] = acc[0][mt][3] + acc[1][mt][3];
    }
  }
  griddep_wait();  // y may still be written by the previous grid in the stream
  cluster_sync_all();

  // Fixed-order reduction over the cluster (and the two chunk halves): this CTA
  // finalises a 1/S share of the group's 128 rows for every real token.
  const int rows_lo = rank * 128 / S, rows_hi = (rank + 1) * 128 / S;
  const int rows_n = rows_hi - rows_lo;
  for (int idx = threadIdx.x; idx < rows_n * M; idx += kDecodeThreads) {
    const int tok = idx / rows_n;
    const int row = rows_lo + (idx - tok * rows_n);
    const uint32_t off = sbase + static_cast<uint32_t>(tok * 128 + row) * 4u;
    // Issue every remote load first, then add in the fixed order (rank, half).
    float v[2 * 8];
#pragma unroll
    for (int src = 0; src < 8; ++src) {
      if (src < S) {
        v[2 * src] = ld_dsmem_f32(off, static_cast<uint32_t>(src));
        v[2 * src + 1] = ld_dsmem_f32(off + Mpad * 128 * 4, static_cast<uint32_t>(src));
      }
    }
    float sum = 0.f;
#pragma unroll
    for (int src = 0; src < 8; ++src) {
      if (src < S) {
        sum += v[2 * src];
        sum += v[2 * src + 1];
      }
    }
    // alpha * 2^7 (the weights carry 2^-7); a per-column alpha times 128 is exact too
    const float sc = alpha_col != nullptr ? alpha_col[grp * 128 + row] * 128.0f : alpha128;
    y[static_cast<size_t>(tok) * N + static_cast<size_t>(grp) * 128 + row] = __float2bfloat16_rn(sum * sc);
  }
  cluster_sync_all();
}

// K split (cluster size S) for a shape: balanced chunk counts within a cluster and
// the thread blocks filling whole waves of the resident slots (SMs x blocks per SM).
int choose_split(int groups, int KC, int MT, const DeviceInfo& dev) {
  const int C = (KC + kChunkKC - 1) / kChunkKC;
  const size_t smem = decode_smem_bytes(8 * MT);
  int per_sm = MT <= 2 ? 2 : 1;
  if (dev.smem_per_sm > 0) per_sm = std::min<int>(per_sm, static_cast<int>(dev.smem_per_sm / (smem + 1024)));
  per_sm = std::max(per_sm, 1);
  const double slots = static_cast<double>(dev.num_sms) * per_sm;
  int best = 1;
  double best_score = -1.0;
  for (int S = 1; S <= 8 && S <= C; ++S) {
    const int maxc = (C + S - 1) / S;
    const double blocks = static_cast<double>(groups) * S;
    const double waves = std::ceil(blocks / slots);
    const double balance = (static_cast<double>(C) / S) / maxc;
    const double fill = blocks / (waves * slots);
    const double score = balance * fill;
    if (score > best_score + 1e-9) { best_score = score; best = S; }
  }
  return best;
}

template <int MT>
nvfp4_status launch_decode(const CUtensorMap& tmW, const CUtensorMap& tmX, float alpha128, const float* alpha_col,
                           __nv_bfloat16* y, int M, int N, int K, int S, cudaStream_t stream, const DeviceInfo& dev) {
  auto kern = w4a16_decode_kernel<MT>;
  const int smem = decode_smem_bytes(8 * MT);
  if (static_cast<size_t>(smem) > dev.max_smem_optin) return NVFP4_ERR_UNSUPPORTED_DEVICE;
  // The dynamic shared-memory limit is raised once per device (no per-call attribute
  // changes, so calls can be captured in CUDA graphs).
  static PerDeviceOnce smem_attr;
  if (!smem_attr.get(dev.device, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess;
      }))
    return NVFP4_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, N / 128, 1);
  cfg.blockDim = dim3(kDecodeThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Programmatic dependent launch: the kernel may start before the previous one in
  // the stream has finished; it waits for it (griddepcontrol.wait) before reading x
  // or writing y, and streams its weights meanwhile.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return from_cuda(cudaLaunchKernelEx(&cfg, kern, tmW, tmX, alpha128, alpha_col, y, M, N, K, S));
}

// ------------------------------------------------------------------ linear, stream-K decode
//
// The balanced form of the decode kernel (TileLang PR #3290, Design: the persistent
// stream-K kernel walking contiguous ranges of the (tile, k-tile) space, with a
// deterministic fix-up of split tiles).  The work is the sequence of units (group of
// 256 weight rows, 64-K block) in group-major order, and block i of G takes units
// [i U / G, (i + 1) U / G) -- equal shares to within one unit, whatever N and K.
//   warp 16     TMA producer: per stage one group's next <= 4 blocks (16 n-tiles x
//               4 blocks, 36 KB) and the matching x columns, into a ring
//   warps 0-15  n-tile w of every stage: register dequant + mma.sync (as the
//               cluster kernel), accumulating over the block's units of a group.
// A group wholly inside a block's range is written to y at once.  A block's first
// and last groups may be split with its neighbours: for those it stores its FP32
// partial in the caller's workspace as soon as the group's part ends, and at the end
// of its range takes one ticket per split group.  The block that takes a group's last
// ticket adds every part's partial in part order (so the result does not depend on
// which part finishes last), writes y and zeroes the ticket.  No block waits for
// another, and no warp stops in the middle of its range: a group's middle parts end
// with their blocks' ranges anyway, so the tickets lose nothing by waiting for it.
namespace skd {

constexpr int kNT = 16;                                  // n-tiles per group (256 rows)
constexpr int kWarps = 16;                               // consumer warps, one n-tile each
constexpr int kThreads = 32 * (kWarps + 1);              // + the producer warp
constexpr int kStageBlocks = 4;                          // 64-K blocks per full stage
constexpr int kWBytes = kNT * kStageBlocks * kBlockBytes;  // 36 KB
constexpr int kMaxTokens = 32;
constexpr int kSlotFloats = kMaxTokens * kNT * 16;       // workspace per slot and SM: [32 tokens][256 rows]
constexpr int kSmemLimit = 232448;                       // opt-in maximum per block
constexpr int kMaxParts = 512;                           // blocks per grid (<= 2 per SM)

// Up to 16 tokens two blocks share an SM (32 consumer warps per SM; the register
// budget allows it), each with a 2-stage ring; 32 tokens run one block per SM with
// as many stages (up to 5) as shared memory holds.
__host__ __device__ constexpr int per_sm(int Mpad) { return Mpad <= 16 ? 2 : 1; }
__host__ __device__ constexpr int stage_bytes(int Mpad) { return kWBytes + Mpad * kStageBlocks * 128; }
__host__ __device__ constexpr int ring(int Mpad) {
  return per_sm(Mpad) == 2 ? 2
         : (kSmemLimit - 4096) / stage_bytes(Mpad) < 5 ? (kSmemLimit - 4096) / stage_bytes(Mpad) : 5;
}
__host__ __device__ constexpr int bar_off(int Mpad) { return ring(Mpad) * stage_bytes(Mpad); }
// barriers (2 x 5 x 8 bytes), the abort flag and two last-ticket flags, the part list
// of a split group, alignment slack
__host__ __device__ constexpr int smem_bytes(int Mpad) { return bar_off(Mpad) + 96 + 4 * kMaxParts + 1024; }

// First unit of block i of G over U units (U < 2^31, checked by the host).
__host__ __device__ __forceinline__ int unit_start(int i, int G, int U) {
  return static_cast<int>(static_cast<int64_t>(i) * U / G);
}
// The block whose range holds unit u.
__device__ __forceinline__ int cta_of(int u, int G, int U) {
  int i = static_cast<int>((static_cast<int64_t>(u) * G) / U);
  while (i + 1 < G && unit_start(i + 1, G, U) <= u) ++i;
  while (i > 0 && unit_start(i, G, U) > u) --i;
  return i;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, per_sm(8 * MT))
    w4a16_decode_sk_kernel(const __grid_constant__ CUtensorMap tmW4, const __grid_constant__ CUtensorMap tmW1,
                           const __grid_constant__ CUtensorMap tmX, float alpha128, const float* __restrict__ alpha_col,
                           __nv_bfloat16* __restrict__ y, int M, int N, int K, float* __restrict__ partials,
                           int* __restrict__ tickets) {
  constexpr int Mpad = 8 * MT;
  constexpr int kStage = stage_bytes(Mpad);
  constexpr int R = ring(Mpad);
  constexpr int kXBytes = Mpad * kStageBlocks * 128;
  constexpr int kSlot = Mpad * 256;  // floats per partial slot: [Mpad tokens][256 rows]
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar_full = sbase + bar_off(Mpad);
  const uint32_t bar_empty = bar_full + 8 * 5;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + bar_off(Mpad) + 80);
  volatile int* last_flag = abort_flag + 1;  // [2]: first and last group of the range
  int* part_slot = reinterpret_cast<int*>(smem + bar_off(Mpad) + 96);  // [kMaxParts]

  const int G = gridDim.x;
  const int KB = K / 64;
  const int NG = (N + 255) / 256;
  const int U = NG * KB;
  const int u0 = unit_start(blockIdx.x, G, U), u1 = unit_start(blockIdx.x + 1, G, U);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < R; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmW4);
      prefetch_tensormap(&tmW1);
      prefetch_tensormap(&tmX);
      auto load_w = [&](int s, int u, int nblk) {
        const int st = s % R;
        const int g = u / KB, kb = u - g * KB;
        const uint32_t dst = sbase + st * kStage;
        mbar_arrive_expect_tx(bar_full + 8 * st, nblk * kNT * kBlockBytes + kXBytes);
        if (nblk == kStageBlocks) {
          asm volatile(
              "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
              " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
              "l"(&tmW4), "r"(0), "r"(kb), "r"(g * kNT), "r"(bar_full + 8 * st)
              : "memory");
        } else {
          // a segment's last 1-3 blocks: one box per block, [block][n-tile][576 B]
          for (int j = 0; j < nblk; ++j)
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst + j * kNT * kBlockBytes),
                "l"(&tmW1), "r"(0), "r"(kb + j), "r"(g * kNT), "r"(bar_full + 8 * st)
                : "memory");
        }
      };
      auto load_x = [&](int s, int u) {
        const int st = s % R;
        const int kb = u % KB;
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sbase + st * kStage + kWBytes),
            "l"(&tmX), "r"(0), "r"(0), "r"(kb), "r"(bar_full + 8 * st)
            : "memory");
      };
      auto stage_len = [&](int u) {
        const int seg_end = min(u1, (u / KB + 1) * KB);
        return min(kStageBlocks, seg_end - u);
      };
      // The weights never depend on an earlier kernel: the first R stages' weights are
      // requested before waiting for the previous grid in the stream (which may be
      // producing x); their x columns follow the wait.
      int s = 0;
      int u = u0;
      for (; s < R && u < u1; ++s) {
        const int n = stage_len(u);
        load_w(s, u, n);
        u += n;
      }
      griddep_wait();
      {
        int v = u0;
        for (int i = 0; i < s; ++i) {
          load_x(i, v);
          v += stage_len(v);
        }
      }
      for (; u < u1; ++s) {
        const int st = s % R;
        if (!mbar_wait(bar_empty + 8 * st, ((s / R) - 1) & 1, abort_flag)) break;
        const int n = stage_len(u);
        load_w(s, u, n);
        load_x(s, u);
        u += n;
      }
      // Let every issued copy land before the thread block can exit.
      for (int i = s > R ? s - R : 0; i < s; ++i)
        mbar_wait_for(bar_full + 8 * (i % R), (i / R) & 1, 2000000000ull);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  griddep_wait();  // x, y and the workspace may belong to the previous grid in the stream
  const int nt = warp;
  const int gq = lane >> 2, t = lane & 3;
  const uint32_t row_off = static_cast<uint32_t>(lane & 7) * 128u;
  const uint32_t sw = static_cast<uint32_t>(lane & 7);
  const uint32_t q = static_cast<uint32_t>(lane >> 3);

  float acc[2][MT][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) acc[a][mt][0] = acc[a][mt][1] = acc[a][mt][2] = acc[a][mt][3] = 0.f;

  auto do_block = [&](uint32_t blk, uint32_t xblk) {
    uint4 c;
    uint2 sc;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(c.x), "=r"(c.y), "=r"(c.z), "=r"(c.w)
                 : "r"(blk + 16 * lane));
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(sc.x), "=r"(sc.y) : "r"(blk + 512 + 8 * gq));
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      uint32_t bf[MT][4];
      const uint32_t piece = ((4u * jj + q) ^ sw) * 16u;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) ldsm_x4(xblk + mt * 1024 + piece, bf[mt][0], bf[mt][1], bf[mt][2], bf[mt][3]);
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        const int j = 2 * jj + j2;
        const uint32_t sword = j < 2 ? sc.x : sc.y;
        uint32_t a[4];
        dequant_word(words[j], scale_pair(sword, j), a);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma_bf16_16816(acc[j2][mt], a, bf[mt][2 * j2], bf[mt][2 * j2 + 1]);
      }
    }
  };

  // y = bf16(sum * scale) for 4 rows of one token, rows row..row+3 of the output.
  auto store4 = [&](float4 sum, int tok, int row) {
    float4 scl = make_float4(alpha128, alpha128, alpha128, alpha128);
    if (alpha_col != nullptr) {
      const float4 a = *reinterpret_cast<const float4*>(alpha_col + row);
      scl = make_float4(a.x * 128.0f, a.y * 128.0f, a.z * 128.0f, a.w * 128.0f);
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(sum.x * scl.x, sum.y * scl.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(sum.z * scl.z, sum.w * scl.w);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&lo);
    packed.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(y + static_cast<size_t>(tok) * N + row) = packed;
  };

  // After a timed-out wait (ok false) a warp still walks every stage and segment end
  // without touching the data, so that the named barriers and the tickets stay
  // consistent across the block's warps and across blocks.
  int s = 0;
  bool ok = true;
  int seg_start = u0;
  int g = u0 / KB;  // the group of the current segment, advanced without dividing
  int gbeg = g * KB, gend = gbeg + KB;
  int seg_end = min(u1, gend);
  int split_group[2] = {-1, -1};  // split groups whose partial is in slot 2i (first) / 2i + 1 (last)
  for (int u = u0; u < u1;) {
    const int nblk = min(kStageBlocks, seg_end - u);
    const int st = s % R;
    if (ok) ok = warp_wait_vote(bar_full + 8 * st, (s / R) & 1, abort_flag);
    const uint32_t stage = sbase + st * kStage;
    const uint32_t xstage = stage + kWBytes + row_off;
    if (ok) {
      if (nblk == kStageBlocks) {
        // [n-tile][block][576 B]
        const uint32_t tile = stage + nt * (kStageBlocks * kBlockBytes);
#pragma unroll
        for (int b = 0; b < kStageBlocks; ++b) do_block(tile + b * kBlockBytes, xstage + b * Mpad * 128);
      } else {
        // a segment's last 1-3 blocks: [block][n-tile][576 B]
        const uint32_t tile = stage + nt * kBlockBytes;
#pragma unroll 1
        for (int b = 0; b < nblk; ++b) do_block(tile + b * (kNT * kBlockBytes), xstage + b * Mpad * 128);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    ++s;
    u += nblk;
    if (u != seg_end) continue;

    // ---------------------------------------------------------- end of a group segment
    const int row_lo = g * 256 + nt * 16 + gq;  // and row_lo + 8
    float v[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[mt][e] = acc[0][mt][e] + acc[1][mt][e];
        acc[0][mt][e] = acc[1][mt][e] = 0.f;
      }
    if (seg_start == gbeg && seg_end == gend) {
      // the whole group in this block
      if (row_lo < N) {
        const float s_lo = alpha_col != nullptr ? alpha_col[row_lo] * 128.0f : alpha128;
        const float s_hi = alpha_col != nullptr ? alpha_col[row_lo + 8] * 128.0f : alpha128;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int tok = 8 * mt + 2 * t;
          if (tok < M) {
            y[static_cast<size_t>(tok) * N + row_lo] = __float2bfloat16_rn(v[mt][0] * s_lo);
            y[static_cast<size_t>(tok) * N + row_lo + 8] = __float2bfloat16_rn(v[mt][2] * s_hi);
          }
          if (tok + 1 < M) {
            y[static_cast<size_t>(tok + 1) * N + row_lo] = __float2bfloat16_rn(v[mt][1] * s_lo);
            y[static_cast<size_t>(tok + 1) * N + row_lo + 8] = __float2bfloat16_rn(v[mt][3] * s_hi);
          }
        }
      }
    } else {
      // a part of a split group: its partial goes to the workspace now, its ticket
      // at the end of the range
      const int which = seg_start == u0 ? 0 : 1;
      split_group[which] = g;
      float* dst = partials + static_cast<size_t>(2 * blockIdx.x + which) * kSlot;
      const int r = nt * 16 + gq;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int tok = 8 * mt + 2 * t;
        if (tok < M) {
          dst[tok * 256 + r] = v[mt][0];
          dst[tok * 256 + r + 8] = v[mt][2];
        }
        if (tok + 1 < M) {
          dst[(tok + 1) * 256 + r] = v[mt][1];
          dst[(tok + 1) * 256 + r + 8] = v[mt][3];
        }
      }
    }
    seg_start = seg_end;
    ++g;
    gbeg = gend;
    gend += KB;
    seg_end = min(u1, gend);
  }

  // ------------------------------------------------------------ tickets of split groups
  if (split_group[0] < 0 && split_group[1] < 0) return;
  named_bar_sync(1, 32 * kWarps);  // every consumer's partial stores are issued
  if (lane == 0 && warp < 2 && split_group[warp] >= 0) {
    // warp 0 takes the first group's ticket, warp 1 the last group's.  The barrier
    // orders the other threads' partial stores before this release; its acquire
    // half orders the partial loads below (after the next barrier) after it.
    const int gg = split_group[warp];
    const int first = cta_of(gg * KB, G, U), last = cta_of(gg * KB + KB - 1, G, U);
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(old) : "l"(tickets + first) : "memory");
    const int is_last = old == last - first;
    if (is_last) tickets[first] = 0;
    last_flag[warp] = is_last;
  }
  named_bar_sync(1, 32 * kWarps);
  // The ring is free now (every stage was consumed): it holds the chunk sums below.
  float4* chunk = reinterpret_cast<float4*>(smem);
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const int gg = split_group[which];
    if (gg < 0 || last_flag[which] == 0) continue;
    // This block took the group's last ticket: add the parts in part order.  With few
    // outputs (64 x M float4 of 4 rows) each output's parts are split into tpo
    // contiguous chunks, one per thread, and the chunk sums added in chunk order.
    const int first = cta_of(gg * KB, G, U), last = cta_of(gg * KB + KB - 1, G, U);
    const int P = last - first + 1;
    for (int p = threadIdx.x; p < P; p += 32 * kWarps)
      part_slot[p] = 2 * (first + p) + (unit_start(first + p, G, U) >= gg * KB ? 0 : 1);
    named_bar_sync(1, 32 * kWarps);
    const int O = 64 * M;
    const int tpo = O >= 32 * kWarps ? 1 : (32 * kWarps) / O;  // 1, 2, 4 or 8 (M = 1 .. 8)
    for (int idx = threadIdx.x; idx < O * tpo; idx += 32 * kWarps) {
      const int o = idx / tpo, j = idx - o * tpo;
      const int tok = o >> 6, r4 = 4 * (o & 63);
      const int p0 = j * P / tpo, p1 = (j + 1) * P / tpo;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
      for (int p = p0; p < p1; ++p) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(
            partials + static_cast<size_t>(part_slot[p]) * kSlot + tok * 256 + r4));
        sum.x += v.x;
        sum.y += v.y;
        sum.z += v.z;
        sum.w += v.w;
      }
      if (tpo == 1) {
        if (gg * 256 + r4 < N) store4(sum, tok, gg * 256 + r4);
      } else {
        chunk[idx] = sum;
      }
    }
    named_bar_sync(1, 32 * kWarps);
    if (tpo > 1) {
      for (int o = threadIdx.x; o < O; o += 32 * kWarps) {
        const int tok = o >> 6, r4 = 4 * (o & 63);
        float4 sum = chunk[o * tpo];
        for (int j = 1; j < tpo; ++j) {
          const float4 v = chunk[o * tpo + j];
          sum.x += v.x;
          sum.y += v.y;
          sum.z += v.z;
          sum.w += v.w;
        }
        if (gg * 256 + r4 < N) store4(sum, tok, gg * 256 + r4);
      }
      named_bar_sync(1, 32 * kWarps);  // chunk and part_slot are reused for the other group
    }
  }
}

}  // namespace skd

// Two partial slots per block: [Mpad tokens][256 rows] floats, at most 2 x SMs blocks
// of up to 16 tokens or SMs blocks of 32; then one ticket per block.
// Decode region (up to 32 tokens): two partial slots of 32 tokens x 256 rows and two
// tickets per SM.  Tensor-core region after it (more than 32 tokens): two slots of
// 128 rows x 256 tokens and one ticket per SM.
constexpr int kTcSkSlotFloats = 128 * 256;  // tensor-core stream-K partial: 128 rows x up to 256 tokens
size_t w4a16_sk_decode_bytes(int num_sms) {
  return static_cast<size_t>(2) * num_sms * skd::kSlotFloats * sizeof(float) + static_cast<size_t>(num_sms) * 8 + 256;
}
size_t w4a16_sk_tc_slot_bytes(int num_sms) {
  return static_cast<size_t>(2) * num_sms * kTcSkSlotFloats * sizeof(float);
}
size_t w4a16_streamk_workspace_bytes_for(int num_sms) {
  return w4a16_sk_decode_bytes(num_sms) + w4a16_sk_tc_slot_bytes(num_sms) + static_cast<size_t>(num_sms) * 4 + 256;
}

template <int MT>
nvfp4_status launch_decode_sk(const CUtensorMap& tmW4, const CUtensorMap& tmW1, const CUtensorMap& tmX,
                              float alpha128, const float* alpha_col, __nv_bfloat16* y, int M, int N, int K,
                              void* ws, cudaStream_t stream, const DeviceInfo& dev) {
  auto kern = skd::w4a16_decode_sk_kernel<MT>;
  const int smem = skd::smem_bytes(8 * MT);
  if (static_cast<size_t>(smem) > dev.max_smem_optin) return NVFP4_ERR_UNSUPPORTED_DEVICE;
  static PerDeviceOnce smem_attr;
  if (!smem_attr.get(dev.device, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess;
      }))
    return NVFP4_ERR_CUDA;
  // At most one block per unit, so that every block's range is non-empty: the parts
  // of a split group are then exactly the blocks from the one holding its first unit
  // to the one holding its last, and each of them takes one ticket.
  const int64_t U = static_cast<int64_t>((N + 255) / 256) * (K / 64);
  if (U > (int64_t(1) << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  const int slots = dev.num_sms * skd::per_sm(8 * MT);
  const int G = static_cast<int>(U < slots ? U : slots);
  if (G > skd::kMaxParts) return NVFP4_ERR_UNSUPPORTED_DEVICE;
  float* partials = static_cast<float*>(ws);
  int* tickets = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) +
                                        static_cast<size_t>(2) * dev.num_sms * skd::kSlotFloats * sizeof(float));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G, 1, 1);
  cfg.blockDim = dim3(skd::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // as in launch_decode
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return from_cuda(
      cudaLaunchKernelEx(&cfg, kern, tmW4, tmW1, tmX, alpha128, alpha_col, y, M, N, K, partials, tickets));
}

// ------------------------------------------------------------------ linear (tensor cores)
//
// For more than 32 tokens the weights are dequantised into shared memory and the
// products run on the tcgen05 tensor cores (kind::f16: BF16 x BF16 -> FP32 in TMEM):
// the 128 weight rows of a group are the MMA's M dimension, the tokens (up to 256
// per tile) its N dimension, so every dequantised weight feeds all tokens at once.
//   warp 0      TMA: 36 KB prepared-weight chunks (128 rows x 512 K) into a 2-deep ring
//   warp 1      TMA: x tiles (tokens x 64 K, 128-byte swizzled, zero rows past M)
//   warp 2      TMEM allocation; lane 0 issues the MMAs (4 x K=16 per 64-K block)
//   warps 3-18  dequantise: warp (p, w) turns n-tile w's 576-byte block of each
//               64-K step i with i % 2 == p into rows 16w..16w+15 of a 128 x 64 BF16
//               A tile (128-byte swizzle, the layout the MMA's K-major descriptor
//               reads)
//   warps 3-6   epilogue: TMEM -> registers -> y (or, when a cluster splits K, ->
//               shared memory, fixed-order reduction across the cluster through
//               distributed shared memory -> y)
namespace tcw {

constexpr int kMaxRawStages = 4;
constexpr int kMaxAStages = 4;
constexpr int kMaxXStages = 16;
constexpr int kABytes = 128 * 128;                // 128 rows x 64 K bf16
constexpr int kDeqWarps = 16;                     // two groups of 8: even and odd 64-K steps
constexpr int kFirstDeqWarp = 3;
constexpr int kThreads = 32 * (kFirstDeqWarp + kDeqWarps);
constexpr int kMaxTokens = 256;
constexpr int kNumBars = 2 * kMaxRawStages + 2 * kMaxAStages + 2 * kMaxXStages + 1;

// Shared memory: a ring of 36 KB weight chunks, dequantised A tiles and x tiles.
// The weight ring is what keeps HBM busy (a chunk takes several microseconds to
// arrive under load), the A ring decouples dequantisation from the MMAs, and an x
// slot refills only after the MMA that read it has completed.  Two chunks (16 steps
// of weights) are ahead enough; an x slot is refilled only after the MMA that read
// it has completed and a copy takes about 1.4 us to land, so x slots get what is
// left (up to 16), and a fourth A tile when x has 8 slots or more.
struct Layout {
  int rs, as, xs;
  int off_a, off_x, off_bar, total;
};

__host__ __device__ inline Layout layout(int nt) {
  Layout L;
  const int xbytes = nt * 128;
  const int budget = 232448 - 1024 - 8 * kNumBars - 16;
  L.rs = 2;
  L.as = 3;
  L.xs = (budget - L.as * kABytes - L.rs * kChunkBytes) / xbytes;
  if (L.xs > kMaxXStages) L.xs = kMaxXStages;
  if (L.xs >= 8 && budget - (L.as + 1) * kABytes - L.rs * kChunkBytes >= L.xs * xbytes) L.as = 4;
  L.off_a = L.rs * kChunkBytes;
  L.off_x = L.off_a + L.as * kABytes;
  L.off_bar = L.off_x + L.xs * xbytes;
  L.total = L.off_bar + 8 * kNumBars + 16 + 1024;
  return L;
}

__host__ __device__ inline uint32_t tmem_cols_for(int nt) {
  return nt <= 32 ? 32u : nt <= 64 ? 64u : nt <= 128 ? 128u : 256u;
}

// kind::f16 instruction descriptor: FP32 accumulator (bits 4-5 = 1), A and B BF16
// (bits 7-9 and 10-12 = 1), both K-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__global__ void __launch_bounds__(kThreads, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    float alpha128, const float* __restrict__ alpha_col, __nv_bfloat16* __restrict__ y, int M,
                    int N, int K, int S, int nt_tok) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));
  const Layout L = layout(nt_tok);
  const int rank = blockIdx.x;  // K split index (position in the cluster)
  const int grp = blockIdx.y;   // 128-row group of N
  const int m0 = blockIdx.z * nt_tok;
  const int KC = K / 64;
  const int C = (KC + kChunkKC - 1) / kChunkKC;
  const int c0 = rank * C / S, c1 = (rank + 1) * C / S;
  const int ks0 = c0 * kChunkKC, ks1 = min(c1 * kChunkKC, KC);  // 64-K steps of this rank
  const int xbytes = nt_tok * 128;

  const uint32_t raw_full = sbase + L.off_bar;
  const uint32_t raw_empty = raw_full + 8 * kMaxRawStages;
  const uint32_t a_full = raw_empty + 8 * kMaxRawStages;
  const uint32_t a_empty = a_full + 8 * kMaxAStages;
  const uint32_t x_full = a_empty + 8 * kMaxAStages;
  const uint32_t x_empty = x_full + 8 * kMaxXStages;
  const uint32_t acc_full = x_empty + 8 * kMaxXStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.off_bar + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.off_bar + 8 * kNumBars + 4);
  const int AS = L.as;
  const int RS = L.rs;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ncols = tmem_cols_for(nt_tok);
  if (threadIdx.x == 0) {
    for (int i = 0; i < RS; ++i) {
      mbar_init(raw_full + 8 * i, 1);
      mbar_init(raw_empty + 8 * i, kDeqWarps);
    }
    for (int i = 0; i < AS; ++i) {
      mbar_init(a_full + 8 * i, kDeqWarps / 2);
      mbar_init(a_empty + 8 * i, 1);
    }
    for (int i = 0; i < L.xs; ++i) {
      mbar_init(x_full + 8 * i, 1);
      mbar_init(x_empty + 8 * i, 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ weight chunks
    // The first ring's chunks are requested before waiting for the previous grid in
    // the stream (the weights never depend on it); every time-limited wait comes after.
    if (lane == 0) {
      prefetch_tensormap(&tmW);
      const int nch = c1 - c0;
      for (int i = 0; i < nch; ++i) {
        const int st = i % RS;
        if (i == RS) griddep_wait();
        if (i >= RS && !mbar_wait(raw_empty + 8 * st, ((i / RS) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(raw_full + 8 * st, kChunkBytes);
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sbase + st * kChunkBytes),
            "l"(&tmW), "r"(0), "r"((c0 + i) * kChunkKC), "r"(grp * kDecodeNT), "r"(raw_full + 8 * st)
            : "memory");
      }
      for (int i = nch > RS ? nch - RS : 0; i < nch; ++i)
        mbar_wait_for(raw_full + 8 * (i % RS), (i / RS) & 1, 2000000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ x tiles
    if (lane == 0) {
      prefetch_tensormap(&tmX);
      griddep_wait();  // x may be produced by the previous grid in the stream
      const int n = ks1 - ks0;
      for (int i = 0; i < n; ++i) {
        const int st = i % L.xs;
        if (i >= L.xs && !mbar_wait(x_empty + 8 * st, ((i / L.xs) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(x_full + 8 * st, xbytes);
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sbase + L.off_x + st * xbytes),
            "l"(&tmX), "r"(0), "r"(m0), "r"(ks0 + i), "r"(x_full + 8 * st)
            : "memory");
      }
      for (int i = n > L.xs ? n - L.xs : 0; i < n; ++i)
        mbar_wait_for(x_full + 8 * (i % L.xs), (i / L.xs) & 1, 2000000000ull);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop on warp-uniform values (barrier waits by vote) and
    // lane 0, elected in each instruction, issues: 4-6 % faster than a lone lane
    // waiting with try_wait (measured at 72, 144 and 1024 tokens).
    {
      griddep_wait();
      const uint32_t tm = warp_uniform(tmem);
      const uint32_t sb = warp_uniform(sbase);
      const uint32_t idesc = idesc_bf16(128, nt_tok);
      const int n = ks1 - ks0;
      const uint32_t u_af = sb + (a_full - sbase), u_ae = sb + (a_empty - sbase);
      const uint32_t u_xf = sb + (x_full - sbase), u_xe = sb + (x_empty - sbase), u_acc = sb + (acc_full - sbase);
      const uint64_t a_desc0 = make_sdesc(sb + L.off_a, 16, 1024, 2);
      const uint64_t x_desc0 = make_sdesc(sb + L.off_x, 16, 1024, 2);
      int as = 0, xs = 0;
      uint32_t a_ph = 0, x_ph = 0;
      for (int i = 0; i < n; ++i) {
        if (!warp_wait_vote(u_af + 8 * as, a_ph, abort_flag)) break;
        if (!warp_wait_vote(u_xf + 8 * xs, x_ph, abort_flag)) break;
        tc_fence_after();
        const uint64_t ad = a_desc0 + static_cast<uint64_t>(as * (kABytes >> 4));
        const uint64_t xd = x_desc0 + static_cast<uint64_t>(xs * (xbytes >> 4));
        tc_mma_f16_elect(tm, ad, xd, idesc, i != 0 ? 1u : 0u);
        tc_mma_f16_elect(tm, ad + 2, xd + 2, idesc, 1u);
        tc_mma_f16_elect(tm, ad + 4, xd + 4, idesc, 1u);
        tc_mma_f16_elect(tm, ad + 6, xd + 6, idesc, 1u);
        tc_commit_elect(u_ae + 8 * as);
        tc_commit_elect(u_xe + 8 * xs);
        if (++as == AS) { as = 0; a_ph ^= 1; }
        if (++xs == L.xs) { xs = 0; x_ph ^= 1; }
      }
      tc_commit_elect(u_acc);
    }
  } else {
    // ------------------------------------------------------------ dequantise
    // Warp (p, w): n-tile w of every step i with i % 2 == p -- two steps in flight,
    // since one block per warp is a short dependent chain that latency, not issue,
    // bounds.
    griddep_wait();
    const int w = (warp - kFirstDeqWarp) & 7;     // n-tile within the group
    const int par = (warp - kFirstDeqWarp) >> 3;  // step parity handled by this warp
    const int g = lane >> 2, t = lane & 3;
    const int n = ks1 - ks0;
    for (int i = par; i < n; i += 2) {
      const int kb = i % kChunkKC;        // block within the chunk
      const int ci = i / kChunkKC;        // chunk index (relative)
      const int rs = ci % RS;
      const int as = i % AS;
      if (kb == par && !warp_wait(raw_full + 8 * rs, (ci / RS) & 1, abort_flag)) break;
      if (i >= AS && !warp_wait(a_empty + 8 * as, ((i / AS) - 1) & 1, abort_flag)) break;
      const uint32_t blk = sbase + rs * kChunkBytes + (w * kChunkKC + kb) * kBlockBytes;
      uint4 c;
      uint2 sc;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(c.x), "=r"(c.y), "=r"(c.z), "=r"(c.w)
                   : "r"(blk + 16 * lane));
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(sc.x), "=r"(sc.y) : "r"(blk + 512 + 8 * g));
      const uint32_t words[4] = {c.x, c.y, c.z, c.w};
      // Rows 16w + g and 16w + g + 8 of the A tile; row r's 16-byte piece p sits at
      // r * 128 + ((p ^ (r % 8)) * 16) (128-byte swizzle), and r % 8 == g here.
      const uint32_t a_lo = sbase + L.off_a + as * kABytes + (16 * w + g) * 128 + 4 * t;
      const uint32_t a_hi = a_lo + 8 * 128;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t sword = j < 2 ? sc.x : sc.y;
        uint32_t a[4];
        dequant_word(words[j], scale_pair(sword, j), a);
        const uint32_t p0 = static_cast<uint32_t>(((2 * j) ^ g) * 16);
        const uint32_t p1 = static_cast<uint32_t>(((2 * j + 1) ^ g) * 16);
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(a_lo + p0), "r"(a[0]) : "memory");
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(a_hi + p0), "r"(a[1]) : "memory");
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(a_lo + p1), "r"(a[2]) : "memory");
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(a_hi + p1), "r"(a[3]) : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(a_full + 8 * as);
        // Last step of this parity in the chunk: the chunk's blocks of this warp are
        // consumed.  (A warp with no step in a partial last chunk never arrives for
        // it; nothing waits for that phase.)
        if (kb + 2 >= kChunkKC || i + 2 >= n) mbar_arrive(raw_empty + 8 * rs);
      }
    }

    // ------------------------------------------------------------ epilogue (warps 3-6)
    if (warp - kFirstDeqWarp < 4) {
      const int q = warp & 3;  // TMEM lane quarter this warp may access
      const int row = 32 * q + lane;
      const int mv = min(nt_tok, M - m0);
      const float sc = alpha_col != nullptr ? alpha_col[grp * 128 + row] * 128.0f : alpha128;
      if (warp_wait(acc_full, 0, abort_flag)) {
        tc_fence_after();
        float* part = reinterpret_cast<float*>(smem);  // [tokens][128 rows], after the loop
#pragma unroll 1
        for (int c32 = 0; c32 < nt_tok; c32 += 32) {
          uint32_t v[32];
          tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + c32, v);
          tc_wait_ld();
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int tok = c32 + jj;
            if (tok < mv) {
              if (S == 1)
                y[static_cast<size_t>(m0 + tok) * N + static_cast<size_t>(grp) * 128 + row] =
                    __float2bfloat16_rn(__uint_as_float(v[jj]) * sc);
              else
                part[tok * 128 + row] = __uint_as_float(v[jj]);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();

  if (S > 1) {
    // Fixed-order reduction over the cluster: this CTA finalises a 1/S share of the
    // group's 128 rows (in units of 4 rows: one 16-byte remote load per source) for
    // every token of the tile.
    griddep_wait();
    cluster_sync_all();
    const int mv = min(nt_tok, M - m0);
    const int q_lo = rank * 32 / S, q_hi = (rank + 1) * 32 / S;
    const int q_n = q_hi - q_lo;
    for (int idx = threadIdx.x; idx < q_n * mv; idx += kThreads) {
      const int tok = idx / q_n;
      const int row = 4 * (q_lo + (idx - tok * q_n));
      const uint32_t off = sbase + static_cast<uint32_t>(tok * 128 + row) * 4u;
      float4 v[8];
#pragma unroll
      for (int src = 0; src < 8; ++src)
        if (src < S) v[src] = ld_dsmem_f32x4(off, static_cast<uint32_t>(src));
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int src = 0; src < 8; ++src) {
        if (src < S) {
          sum.x += v[src].x;
          sum.y += v[src].y;
          sum.z += v[src].z;
          sum.w += v[src].w;
        }
      }
      float4 sc = make_float4(alpha128, alpha128, alpha128, alpha128);
      if (alpha_col != nullptr) {
        const float4 a = *reinterpret_cast<const float4*>(alpha_col + grp * 128 + row);
        sc = make_float4(a.x * 128.0f, a.y * 128.0f, a.z * 128.0f, a.w * 128.0f);
      }
      __nv_bfloat162 lo = __floats2bfloat162_rn(sum.x * sc.x, sum.y * sc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(sum.z * sc.z, sum.w * sc.w);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(y + static_cast<size_t>(m0 + tok) * N + static_cast<size_t>(grp) * 128 + row) = packed;
    }
    cluster_sync_all();
  }
  if (warp == 2) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}


// ------------------------------------------------------------------ tensor-core stream-K
//
// More than 32 tokens with a caller workspace (TileLang PR #3290, Design: the persistent stream-K
// kernel over contiguous (tile, k-tile) ranges).  The units are (token tile, 128-row
// group, 64-K step), group-major; block b of G takes units [b U / G, (b+1) U / G).  A
// block walks its range as segments, one per (token tile, group) it touches: the same
// weight-chunk, x-tile, A-tile and MMA pipeline as w4a16_tc_kernel, with the rings
// counted across segments, the accumulator drained by four epilogue warps of their
// own after each segment.  A segment that covers its whole group goes to y; a part of
// a split group goes to the workspace (slot 2b for the block's first segment, 2b + 1
// for its last), and the block takes the group's ticket at the end of its range.  The
// block taking a group's last ticket adds the parts in part order, writes y and
// zeroes the ticket.  No block waits for another.
constexpr int kSkEpiWarp = kFirstDeqWarp + kDeqWarps;  // 19..22: epilogue, one per TMEM lane quarter
constexpr int kSkThreads = 32 * (kSkEpiWarp + 4);
constexpr int kSkSlotFloats = kTcSkSlotFloats;          // partial of one group: 128 rows x up to 256 tokens
static_assert(kSkSlotFloats >= 128 * kMaxTokens, "stream-K slot");

// (unit ranges: csrc/sk_units.h, shared with a host-side test)

__global__ void __launch_bounds__(kSkThreads, 1)
    w4a16_tc_sk_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       float alpha128, const float* __restrict__ alpha_col, __nv_bfloat16* __restrict__ y, int M,
                       int N, int K, int nt_tok, int mt, float* __restrict__ partials, int* __restrict__ tickets) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - smem_u32(smem_raw));
  const Layout L = layout(nt_tok);
  const int G = gridDim.x;
  const int KS = K / 64;
  const int groups = N / 128;
  const int64_t U = static_cast<int64_t>(mt) * groups * KS;
  const int64_t u0 = sku::unit_start(blockIdx.x, G, U), u1 = sku::unit_start(blockIdx.x + 1, G, U);
  const int xbytes = nt_tok * 128;

  const uint32_t raw_full = sbase + L.off_bar;
  const uint32_t raw_empty = raw_full + 8 * kMaxRawStages;
  const uint32_t a_full = raw_empty + 8 * kMaxRawStages;
  const uint32_t a_empty = a_full + 8 * kMaxAStages;
  const uint32_t x_full = a_empty + 8 * kMaxAStages;
  const uint32_t x_empty = x_full + 8 * kMaxXStages;
  const uint32_t acc_full = x_empty + 8 * kMaxXStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.off_bar + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.off_bar + 8 * kNumBars + 4);
  // (the weight ring uses RS = 2 of its kMaxRawStages barrier slots: the last one is free)
  const uint32_t acc_empty = raw_full + 8 * (kMaxRawStages - 1);
  const int AS = L.as;
  const int RS = L.rs;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ncols = tmem_cols_for(nt_tok);
  if (threadIdx.x == 0) {
    for (int i = 0; i < RS; ++i) {
      mbar_init(raw_full + 8 * i, 1);
      mbar_init(raw_empty + 8 * i, kDeqWarps);
    }
    for (int i = 0; i < AS; ++i) {
      mbar_init(a_full + 8 * i, kDeqWarps / 2);
      mbar_init(a_empty + 8 * i, 1);
    }
    for (int i = 0; i < L.xs; ++i) {
      mbar_init(x_full + 8 * i, 1);
      mbar_init(x_empty + 8 * i, 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  // Segment s of this block: units [su, su + n) = steps [s0, s0 + n) of (token tile, group) pg.
  auto segment = [&](int64_t su, int64_t& pg, int& s0, int& n) {
    pg = su / KS;
    s0 = static_cast<int>(su - pg * KS);
    n = static_cast<int>(min(static_cast<int64_t>(KS - s0), u1 - su));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ weight chunks (boxes of 8 steps from s0)
    if (lane == 0) {
      prefetch_tensormap(&tmW);
      int gc = 0;  // chunks issued
      int st = 0;  // ring slot of chunk gc, and the parity of its round
      uint32_t ph = 0;
      bool ok = true;
      for (int64_t su = u0; su < u1 && ok;) {
        int64_t pg;
        int s0, n;
        segment(su, pg, s0, n);
        const int g = static_cast<int>(pg % groups);
        for (int ci = 0; ci * kChunkKC < n; ++ci, ++gc) {
          if (gc == RS) griddep_wait();
          if (gc >= RS && !mbar_wait(raw_empty + 8 * st, ph ^ 1, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(raw_full + 8 * st, kChunkBytes);
          asm volatile(
              "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
              " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sbase + st * kChunkBytes),
              "l"(&tmW), "r"(0), "r"(s0 + ci * kChunkKC), "r"(g * kDecodeNT), "r"(raw_full + 8 * st)
              : "memory");
          if (++st == RS) { st = 0; ph ^= 1; }
        }
        su += n;
      }
      if (gc <= RS) griddep_wait();
      for (int i = gc > RS ? gc - RS : 0; i < gc; ++i)
        mbar_wait_for(raw_full + 8 * (i % RS), (i / RS) & 1, 2000000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ x tiles
    if (lane == 0) {
      prefetch_tensormap(&tmX);
      griddep_wait();
      int gs = 0;  // steps issued
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int64_t su = u0; su < u1 && ok;) {
        int64_t pg;
        int s0, n;
        segment(su, pg, s0, n);
        const int m0 = static_cast<int>(pg / groups) * nt_tok;
        for (int i = 0; i < n; ++i, ++gs) {
          if (gs >= L.xs && !mbar_wait(x_empty + 8 * st, ph ^ 1, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(x_full + 8 * st, xbytes);
          asm volatile(
              "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
              " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sbase + L.off_x + st * xbytes),
              "l"(&tmX), "r"(0), "r"(m0), "r"(s0 + i), "r"(x_full + 8 * st)
              : "memory");
          if (++st == L.xs) { st = 0; ph ^= 1; }
        }
        su += n;
      }
      for (int i = gs > L.xs ? gs - L.xs : 0; i < gs; ++i)
        mbar_wait_for(x_full + 8 * (i % L.xs), (i / L.xs) & 1, 2000000000ull);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer (whole warp, elected issue)
    griddep_wait();
    const uint32_t tm = warp_uniform(tmem);
    const uint32_t sb = warp_uniform(sbase);
    const uint32_t idesc = idesc_bf16(128, nt_tok);
    const uint32_t u_af = sb + (a_full - sbase), u_ae = sb + (a_empty - sbase);
    const uint32_t u_xf = sb + (x_full - sbase), u_xe = sb + (x_empty - sbase);
    const uint32_t u_accf = sb + (acc_full - sbase), u_acce = sb + (acc_empty - sbase);
    const uint64_t a_desc0 = make_sdesc(sb + L.off_a, 16, 1024, 2);
    const uint64_t x_desc0 = make_sdesc(sb + L.off_x, 16, 1024, 2);
    // ring slots and phases advance by one per step (no division on this warp's path)
    int as = 0, xs = 0, seg = 0;
    uint32_t a_ph = 0, x_ph = 0;
    bool ok = true;
    for (int64_t su = u0; su < u1 && ok; ++seg) {
      int64_t pg;
      int s0, n;
      segment(su, pg, s0, n);
      // the epilogue has drained the previous segment's accumulator
      if (seg > 0 && !warp_wait_vote(u_acce, (seg - 1) & 1, abort_flag)) break;
      tc_fence_after();
      for (int i = 0; i < n; ++i) {
        if (!warp_wait_vote(u_af + 8 * as, a_ph, abort_flag)) { ok = false; break; }
        if (!warp_wait_vote(u_xf + 8 * xs, x_ph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t ad = a_desc0 + static_cast<uint64_t>(as * (kABytes >> 4));
        const uint64_t xd = x_desc0 + static_cast<uint64_t>(xs * (xbytes >> 4));
        tc_mma_f16_elect(tm, ad, xd, idesc, i != 0 ? 1u : 0u);
        tc_mma_f16_elect(tm, ad + 2, xd + 2, idesc, 1u);
        tc_mma_f16_elect(tm, ad + 4, xd + 4, idesc, 1u);
        tc_mma_f16_elect(tm, ad + 6, xd + 6, idesc, 1u);
        tc_commit_elect(u_ae + 8 * as);
        tc_commit_elect(u_xe + 8 * xs);
        if (++as == AS) { as = 0; a_ph ^= 1; }
        if (++xs == L.xs) { xs = 0; x_ph ^= 1; }
      }
      tc_commit_elect(u_accf);  // also after a timed-out wait: lets the epilogue proceed
      su += n;
    }
  } else if (warp < kSkEpiWarp) {
    // ------------------------------------------------------------ dequantise
    // Warp (p, w): n-tile w of the steps of parity p within each chunk.  Every warp
    // waits for every chunk and releases it once, also a chunk with no step of its
    // parity (a one-step chunk at a segment's end): the ring slot is refilled only
    // after all sixteen warps are past the chunk.
    griddep_wait();
    const int w = (warp - kFirstDeqWarp) & 7;
    const int par = (warp - kFirstDeqWarp) >> 3;
    const int g8 = lane >> 2, t = lane & 3;
    int rs = 0;  // chunk ring slot and the parity of its round
    uint32_t rph = 0;
    int gs0 = 0;  // steps before the current segment
    // A ring position of global step `cur`, advanced by small steps (no division)
    int cur = 0, as = 0;
    uint32_t aph = 0;
    auto a_slot_of = [&](int ig) {
      while (cur < ig) {
        ++cur;
        if (++as == AS) { as = 0; aph ^= 1; }
      }
    };
    bool ok = true;
    for (int64_t su = u0; su < u1 && ok;) {
      int64_t pg;
      int s0, n;
      segment(su, pg, s0, n);
      for (int ci = 0; ci * kChunkKC < n && ok; ++ci) {
        if (!warp_wait(raw_full + 8 * rs, rph, abort_flag)) { ok = false; break; }
        const int kcn = min(kChunkKC, n - ci * kChunkKC);
        for (int kb = par; kb < kcn; kb += 2) {
          const int ig = gs0 + ci * kChunkKC + kb;  // global step
          a_slot_of(ig);
          if (ig >= AS && !warp_wait(a_empty + 8 * as, aph ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t blk = sbase + rs * kChunkBytes + (w * kChunkKC + kb) * kBlockBytes;
          uint4 c;
          uint2 sc;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(c.x), "=r"(c.y), "=r"(c.z), "=r"(c.w)
                       : "r"(blk + 16 * lane));
          asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(sc.x), "=r"(sc.y) : "r"(blk + 512 + 8 * g8));
          const uint32_t words[4] = {c.x, c.y, c.z, c.w};
          const uint32_t a_lo = sbase + L.off_a + as * kABytes + (16 * w + g8) * 128 + 4 * t;
          const uint32_t a_hi = a_lo + 8 * 128;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t sword = j < 2 ? sc.x : sc.y;
            uint32_t a[4];
            dequant_word(words[j], scale_pair(sword, j), a);
            const uint32_t p0 = static_cast<uint32_t>(((2 * j) ^ g8) * 16);
            const uint32_t p1 = static_cast<uint32_t>(((2 * j + 1) ^ g8) * 16);
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(a_lo + p0), "r"(a[0]) : "memory");
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(a_hi + p0), "r"(a[1]) : "memory");
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(a_lo + p1), "r"(a[2]) : "memory");
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(a_hi + p1), "r"(a[3]) : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(a_full + 8 * as);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_empty + 8 * rs);
        if (++rs == RS) { rs = 0; rph ^= 1; }
      }
      gs0 += n;
      su += n;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 19-22)
    griddep_wait();
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = 32 * q + lane;
    const int nchunks = (nt_tok + 31) / 32;
    int seg = 0;
    for (int64_t su = u0; su < u1; ++seg) {
      int64_t pg;
      int s0, n;
      segment(su, pg, s0, n);
      if (!warp_wait(acc_full, seg & 1, abort_flag)) break;
      tc_fence_after();
      const int g = static_cast<int>(pg % groups);
      const int m0 = static_cast<int>(pg / groups) * nt_tok;
      const int mv = min(nt_tok, M - m0);
      const bool whole = s0 == 0 && n == KS;
      const float sc = alpha_col != nullptr ? alpha_col[g * 128 + row] * 128.0f : alpha128;
      // slot of a split part: this block's first segment or its last
      float4* dst = reinterpret_cast<float4*>(partials) +
                    (static_cast<size_t>(2 * blockIdx.x + (su == u0 ? 0 : 1)) * kSkSlotFloats) / 4;
#pragma unroll 1
      for (int c = 0; c < nchunks; ++c) {
        uint32_t v[32];
        tc_ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * q) << 16) + 32 * c, v);
        tc_wait_ld(v);
        if (whole) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int tok = 32 * c + jj;
            if (tok < mv)
              y[static_cast<size_t>(m0 + tok) * N + static_cast<size_t>(g) * 128 + row] =
                  __float2bfloat16_rn(__uint_as_float(v[jj]) * sc);
          }
        } else {
          // [lane quarter][32-token chunk][float4 i][lane]: whole 512-byte warp stores
#pragma unroll
          for (int i = 0; i < 8; ++i)
            __stcg(dst + ((q * nchunks + c) * 8 + i) * 32 + lane,
                   make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                               __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
        }
      }
      if (!whole) __threadfence();  // the part is visible at GPU scope before the block's ticket
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      su += n;
    }
  }

  // ------------------------------------------------------------ tickets of split groups
  tc_fence_before();
  __syncthreads();
  griddep_wait();  // every thread writes y below
  // Every role is done and no copy is in flight: the ring's first bytes hold the flags
  // and then the slot of every part of the group being summed.
  int* last_flag = reinterpret_cast<int*>(smem);  // [2]
  int* part_slot = last_flag + 4;                 // [parts], at most one per block
  if (threadIdx.x < 2) {
    last_flag[threadIdx.x] = 0;
    // part 0: the group of the range's first unit, part 1: that of its last unit
    const int64_t su = threadIdx.x == 0 ? u0 : u1 - 1;
    const int64_t pg = su / KS;
    const int64_t gu0 = pg * KS, gu1 = gu0 + KS;
    const bool split = u0 > gu0 || u1 < gu1;
    const bool distinct = threadIdx.x == 0 || (u0 / KS) != pg;
    if (u1 > u0 && split && distinct && !*abort_flag) {
      const int first = sku::cta_of(gu0, G, U), last = sku::cta_of(gu1 - 1, G, U);
      int old;
      asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(old) : "l"(tickets + first) : "memory");
      if (old == last - first) {
        tickets[first] = 0;
        last_flag[threadIdx.x] = 1;
      }
    }
  }
  __syncthreads();
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    if (!last_flag[which]) continue;
    // This block took the group's last ticket: add the parts in part order.
    const int64_t pg = (which == 0 ? u0 : u1 - 1) / KS;
    const int64_t gu0 = pg * KS;
    const int first = sku::cta_of(gu0, G, U), last = sku::cta_of(gu0 + KS - 1, G, U);
    const int g = static_cast<int>(pg % groups);
    const int m0 = static_cast<int>(pg / groups) * nt_tok;
    const int mv = min(nt_tok, M - m0);
    const int nchunks = (nt_tok + 31) / 32;
    for (int p = first + static_cast<int>(threadIdx.x); p <= last; p += kSkThreads)
      part_slot[p - first] = sku::part_slot(p, G, U, gu0);
    __syncthreads();
    // One float4 of the slot layout per thread and pass ([lane quarter][32-token
    // chunk][float4 i][lane]).  The sum is bound by L2 latency: every thread of the
    // block takes part, each with up to eight loads in flight (one load at a time
    // measured ~12 us for five parts of 48 KB).
    const int nf4 = 4 * nchunks * 8 * 32;
    const int P = last - first + 1;
    const float4* part4 = reinterpret_cast<const float4*>(partials);
#pragma unroll 2
    for (int e = threadIdx.x; e < nf4; e += kSkThreads) {
      const int ln = e & 31, i = (e >> 5) & 7, qc = e >> 8;
      const int q = qc / nchunks, c = qc - q * nchunks;
      const int tok0 = 32 * c + 4 * i;
      if (tok0 >= mv) continue;
      const int row = 32 * q + ln;
      // up to eight parts' loads in flight at once, then added in part order
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p0 = 0; p0 < P; p0 += 8) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (p0 + k < P) v[k] = __ldcg(part4 + static_cast<size_t>(part_slot[p0 + k]) * (kSkSlotFloats / 4) + e);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (p0 + k < P) {
            sum.x += v[k].x;
            sum.y += v[k].y;
            sum.z += v[k].z;
            sum.w += v[k].w;
          }
        }
      }
      const float sc = alpha_col != nullptr ? alpha_col[g * 128 + row] * 128.0f : alpha128;
      const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (tok0 + k < mv)
          y[static_cast<size_t>(m0 + tok0 + k) * N + static_cast<size_t>(g) * 128 + row] =
              __float2bfloat16_rn(vals[k] * sc);
    }
    __syncthreads();  // part_slot is rewritten for the next group
  }
  if (warp == 2) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

}  // namespace tcw

// Split count S (cluster size) and token-tile width for the tensor-core path.  A
// unit (128 weight rows x one token tile) runs as a cluster of S CTAs that split K;
// active[S] clusters of that size fit on the GPU at once (queried: clusters live
// inside a GPC, so this is not the SM count / S).  Cost model: waves x (64-K steps
// per CTA + 8), the 8 standing for a CTA's fixed cost (pipeline fill, drain and
// the cluster reduction; a globaltimer trace put it near 8 steps).  An earlier
// wave-fill score that ignored both chose S = 5 for M = 1024 x N = 17408: 2720
// CTAs of 16 steps each, 2.5x slower than S = 1.
void choose_tc(int groups, int KC, int M, const int (&active)[9], int* S_out, int* nt_out, int* ttiles_out) {
  const int mt = (M + tcw::kMaxTokens - 1) / tcw::kMaxTokens;     // token tiles
  const int per = (M + mt - 1) / mt;
  const int nt = ((per + 15) / 16) * 16;                          // tokens per tile (multiple of 16)
  const int C = (KC + kChunkKC - 1) / kChunkKC;
  const int64_t units = static_cast<int64_t>(groups) * mt;
  int best = 1;
  int64_t best_cost = -1;
  for (int S = 1; S <= 8 && S <= C; ++S) {
    const int64_t act = active[S] > 0 ? active[S] : 1;
    const int64_t waves = (units + act - 1) / act;
    const int64_t steps = (static_cast<int64_t>((C + S - 1) / S)) * kChunkKC;
    const int64_t cost = waves * (steps + 8);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = S; }
  }
  *S_out = best;
  *nt_out = nt;
  *ttiles_out = mt;
}

nvfp4_status launch_tc(const CUtensorMap& tmW, const void* x, float alpha128, const float* alpha_col, __nv_bfloat16* y,
                       int M, int N, int K, cudaStream_t stream, const DeviceInfo& dev) {
  auto kern = tcw::w4a16_tc_kernel;
  static PerDeviceOnce setup;
  static int active[64][9] = {};  // co-resident clusters of S CTAs (one CTA per SM), per device
  const int d = dev.device < 64 ? dev.device : 63;
  const int ok = setup.get(d, [&] {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(dev.max_smem_optin)) != cudaSuccess)
      return 0;
    for (int s = 1; s <= 8; ++s) {
      cudaLaunchConfig_t qc = {};
      qc.gridDim = dim3(s, 1, 1);
      qc.blockDim = dim3(tcw::kThreads, 1, 1);
      qc.dynamicSmemBytes = static_cast<size_t>(tcw::layout(tcw::kMaxTokens).total);
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
  int S, nt, mt;
  choose_tc(N / 128, K / 64, M, active[d], &S, &nt, &mt);
  const tcw::Layout L = tcw::layout(nt);
  if (L.rs < 2 || L.xs < 3 || static_cast<size_t>(L.total) > dev.max_smem_optin) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (S > 1 && nt * 128 * 4 > L.off_bar) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap tmX;
  nvfp4_status st = encode_tmap_x_blocks(&tmX, x, M, K, static_cast<uint32_t>(nt), 1);
  if (st != NVFP4_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, N / 128, mt);
  cfg.blockDim = dim3(tcw::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // as in launch_decode
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return from_cuda(cudaLaunchKernelEx(&cfg, kern, tmW, tmX, alpha128, alpha_col, y, M, N, K, S, nt));
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

nvfp4_status launch_w4a16_linear(const void* x, const void* Wprep, float alpha, const float* alpha_col, void* y,
                                 int64_t M, int64_t N, int64_t K, cudaStream_t stream, const DeviceInfo& dev) {
  const float alpha128 = alpha * 128.0f;
  const int KC = static_cast<int>(K / 64);
  const int groups = static_cast<int>(N / 128);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* yb = static_cast<__nv_bfloat16*>(y);
  // The prepared weight as [N/16][K/64][576 B] (UINT64 elements: 72 per block).
  CUtensorMap tmW;
  {
    nvfp4_status st = encode_tmap_wprep(&tmW, Wprep, N, K);
    if (st != NVFP4_OK) return st;
  }
  // More than 32 tokens: tensor cores (dequantise once into shared memory, every
  // weight feeding all tokens).  Up to 32 tokens: the register-dequant decode kernel,
  // which streams at a higher rate there -- the tensor-core path recycles each A
  // tile through an MMA commit (about a microsecond), and shared memory holds too
  // few tiles to hide that at decode-sized MMAs.
  if (M > 32) return launch_tc(tmW, xb, alpha128, alpha_col, yb, static_cast<int>(M), static_cast<int>(N),
                               static_cast<int>(K), stream, dev);
  // Token chunks of up to 32 rows per launch.
  for (int64_t m0 = 0; m0 < M; m0 += kDecodeMaxTokens) {
    const int mc = static_cast<int>(M - m0 < kDecodeMaxTokens ? M - m0 : kDecodeMaxTokens);
    const int MT = mc <= 8 ? 1 : mc <= 16 ? 2 : 4;
    const int S = choose_split(groups, KC, MT, dev);
    CUtensorMap tmX;
    nvfp4_status st = encode_tmap_x_blocks(&tmX, xb + m0 * K, mc, K, 8 * MT, kChunkKC);
    if (st != NVFP4_OK) return st;
    __nv_bfloat16* yc = yb + m0 * N;
    switch (MT) {
      case 1: st = launch_decode<1>(tmW, tmX, alpha128, alpha_col, yc, mc, static_cast<int>(N), static_cast<int>(K), S, stream, dev); break;
      case 2: st = launch_decode<2>(tmW, tmX, alpha128, alpha_col, yc, mc, static_cast<int>(N), static_cast<int>(K), S, stream, dev); break;
      default: st = launch_decode<4>(tmW, tmX, alpha128, alpha_col, yc, mc, static_cast<int>(N), static_cast<int>(K), S, stream, dev); break;
    }
    if (st != NVFP4_OK) return st;
  }
  return NVFP4_OK;
}

size_t w4a16_streamk_workspace_bytes(const DeviceInfo& dev) { return w4a16_streamk_workspace_bytes_for(dev.num_sms); }

// More than 32 tokens with the workspace: tensor-core stream-K over (token tile,
// 128-row group, 64-K step) units, one block per SM (or per unit, if fewer).
nvfp4_status launch_tc_sk(const void* x, const void* Wprep, float alpha128, const float* alpha_col, void* y,
                          int64_t M, int64_t N, int64_t K, void* ws, cudaStream_t stream, const DeviceInfo& dev) {
  auto kern = tcw::w4a16_tc_sk_kernel;
  static PerDeviceOnce setup;
  const int d = dev.device < 64 ? dev.device : 63;
  if (!setup.get(d, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(dev.max_smem_optin)) == cudaSuccess
                   ? 1
                   : 0;
      }))
    return NVFP4_ERR_CUDA;
  const int mt = static_cast<int>((M + tcw::kMaxTokens - 1) / tcw::kMaxTokens);  // token tiles
  const int per = static_cast<int>((M + mt - 1) / mt);
  const int nt = ((per + 15) / 16) * 16;
  const tcw::Layout L = tcw::layout(nt);
  if (L.rs < 2 || L.rs >= tcw::kMaxRawStages || L.xs < 3 || static_cast<size_t>(L.total) > dev.max_smem_optin)
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  const int64_t U = static_cast<int64_t>(mt) * (N / 128) * (K / 64);
  const int G = static_cast<int>(U < dev.num_sms ? U : dev.num_sms);
  CUtensorMap tmW, tmX;
  nvfp4_status st = encode_tmap_wprep(&tmW, Wprep, N, K);
  if (st == NVFP4_OK) st = encode_tmap_x_blocks(&tmX, x, M, K, static_cast<uint32_t>(nt), 1);
  if (st != NVFP4_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(ws) + w4a16_sk_decode_bytes(dev.num_sms);
  float* partials = reinterpret_cast<float*>(base);
  int* tickets = reinterpret_cast<int*>(base + w4a16_sk_tc_slot_bytes(dev.num_sms));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G, 1, 1);
  cfg.blockDim = dim3(tcw::kSkThreads, 1, 1);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return from_cuda(cudaLaunchKernelEx(&cfg, kern, tmW, tmX, alpha128, alpha_col, static_cast<__nv_bfloat16*>(y),
                                      static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), nt, mt, partials,
                                      tickets));
}

nvfp4_status launch_w4a16_linear_streamk(const void* x, const void* Wprep, float alpha, const float* alpha_col,
                                         void* y, int64_t M, int64_t N, int64_t K, void* ws, cudaStream_t stream,
                                         const DeviceInfo& dev) {
  // More than 32 tokens: the tensor-core kernels.  Stream-K pays where the tile grid
  // of the cluster-split kernel (token tiles x 128-row groups) leaves most of a wave
  // empty; elsewhere its fix-up (one block adding a split group's partials at the end,
  // ~5 us per group at 72 tokens) costs more than the balance gains.  Measured (graph
  // replay): 5120 x 17408, 1024 tokens 195.8 -> 153.8 us; 5120 x 5120, 1024 tokens
  // 68.7 -> 67.3 us; 17408 x 5120, 1024 tokens 164.7 -> 185.3 us; up to 256 tokens
  // stream-K measured 0.49-0.94 of the cluster-split kernel.
  if (M > skd::kMaxTokens) {
    const int64_t tiles = ((M + tcw::kMaxTokens - 1) / tcw::kMaxTokens) * (N / 128);
    if (M > tcw::kMaxTokens && 4 * tiles < 5 * static_cast<int64_t>(dev.num_sms))
      return launch_tc_sk(x, Wprep, alpha * 128.0f, alpha_col, y, M, N, K, ws, stream, dev);
    return launch_w4a16_linear(x, Wprep, alpha, alpha_col, y, M, N, K, stream, dev);
  }
  const float alpha128 = alpha * 128.0f;
  CUtensorMap tmW4, tmW1, tmX;
  nvfp4_status st = encode_tmap_wprep(&tmW4, Wprep, N, K, skd::kStageBlocks, skd::kNT);
  if (st == NVFP4_OK) st = encode_tmap_wprep(&tmW1, Wprep, N, K, 1, skd::kNT);
  const int MT = M <= 8 ? 1 : M <= 16 ? 2 : 4;
  if (st == NVFP4_OK) st = encode_tmap_x_blocks(&tmX, x, M, K, 8 * MT, skd::kStageBlocks);
  if (st != NVFP4_OK) return st;
  auto* yb = static_cast<__nv_bfloat16*>(y);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  switch (MT) {
    case 1: return launch_decode_sk<1>(tmW4, tmW1, tmX, alpha128, alpha_col, yb, m, n, k, ws, stream, dev);
    case 2: return launch_decode_sk<2>(tmW4, tmW1, tmX, alpha128, alpha_col, yb, m, n, k, ws, stream, dev);
    default: return launch_decode_sk<4>(tmW4, tmW1, tmX, alpha128, alpha_col, yb, m, n, k, ws, stream, dev);
  }
}

}  // namespace nvfp4

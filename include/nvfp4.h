/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 block-scaled library.
 *
 * The library computes the NVFP4 block-scaled GEMM
 *
 *     D[m,n] = bf16( alpha * sum_k (A[m,k] * SFA[m,k/16]) * (B[n,k] * SFB[n,k/16]) )
 *
 * with E2M1 element codes, one unsigned E4M3 scale per 16 consecutive K elements,
 * an FP32 per-tensor alpha, FP32 accumulation and BF16 output, plus the producers
 * of its operands (quantisation, scale-factor packing) and a decode-shaped W4A16
 * variant (BF16 activations times NVFP4 weights dequantised in registers).
 *
 * Sources (cited by page title and section):
 *   [P1] Colfax Research, "Optimizing an NVFP4 Blockscaled GEMM on RTX PRO 6000
 *        Blackwell GPU (SM120)".
 *   [P2] TileLang PR #3290, "[CUDA] Add an SM120 W4A16 NVFP4 GEMM example for
 *        decode-sized batches".
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller; the library
 *     allocates no device memory and keeps no per-call state on the device, except
 *     for the static workspace array of nvfp4_gemm_streamk_noalloc.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and never synchronises the host.  Calls on different streams may run
 *     concurrently.
 *   - Every kernel is launched with programmatic dependent launch allowed: a call
 *     may start while the previous kernel in the stream is still running, and waits
 *     for that kernel to complete before it reads activations or writes its output.
 *     The WEIGHT operands of nvfp4_gemm* (B, SFB) and of nvfp4_w4a16_linear* (Wprep)
 *     are read without that wait, so that a layer's weights stream in while the
 *     previous kernel finishes.  Weights must therefore not be written by a kernel
 *     in the same stream that is still running when the call starts: a kernel that
 *     signals programmatic completion early (griddepcontrol.launch_dependents).
 *     Every kernel that does not, and every producer of this library (quantize,
 *     pack_scales, w4a16_prepare and their variants signal their dependents only by
 *     completing), may write the weights right before the call.  A caller's own
 *     kernel launched after one of these calls with programmatic stream
 *     serialization must wait (griddepcontrol.wait / cudaGridDependencySynchronize)
 *     before reading the output.
 *   - Errors are returned as nvfp4_status; nothing aborts or throws.  Arguments are
 *     checked on the host; device data (codes, scales) is NOT validated: a NaN
 *     (0x7F/0xFF) or negative scale byte given to nvfp4_gemm gives undefined
 *     output values (never a fault).
 *   - All sizes are 64-bit and all device offsets are computed in 64 bits.
 *   - The device must be compute capability 10.3 (GB300); otherwise every compute
 *     entry point returns NVFP4_ERR_UNSUPPORTED_DEVICE.
 *   - Packed E2M1 codes: two 4-bit codes per byte, the LOW nibble holds the even k.
 *     Code bits: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa; values
 *     +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   - E4M3 scale byte: bit 7 sign (must be 0 for GEMM inputs), bits 6..3 exponent
 *     (bias 7), bits 2..0 mantissa; subnormals m*2^-9 and zero are valid scales.
 */
#ifndef NVFP4_GB300_H_
#define NVFP4_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* nvfp4_stream_t;

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = -1,       /* null pointer, non-positive size, bad scale value */
  NVFP4_ERR_UNSUPPORTED_SHAPE = -2, /* a size violates a documented divisibility rule */
  NVFP4_ERR_MISALIGNED = -3,        /* a pointer violates a documented alignment rule */
  NVFP4_ERR_UNSUPPORTED_DEVICE = -4,/* current device is not compute capability 10.3 */
  NVFP4_ERR_CUDA = -5,              /* a CUDA runtime/driver call or a launch failed */
  NVFP4_ERR_TIMEOUT = -6            /* a kernel gave up a bounded wait (see nvfp4_device_error) */
} nvfp4_status;

/* Static, human-readable name of a status code (never NULL; values outside the enum
   give "NVFP4_ERR_UNKNOWN"). */
const char* nvfp4_status_string(nvfp4_status status);

/* ABI version of this header: major * 10000 + minor * 100 + patch. */
int nvfp4_version(void);

/*
 * nvfp4_quantize -- BF16 activations/weights -> NVFP4 codes + row-major E4M3 scales.
 *
 * The pages name the format ([P2] Design: E2M1 codes packed two per byte, unsigned
 * E4M3 block scales, a per-tensor or per-column scale) but print no quantiser; this is the two-level
 * NVFP4 recipe, with every step in IEEE float32, round to nearest even, unfused:
 *   s      = E4M3_satfinite( (amax_block / 6) / global_scale )
 *   code_k = E2M1_satfinite( x_k / (dec(s) * global_scale) )
 *   a block whose scale is 0 gets all-zero codes; no -0 code is produced.
 * The caller chooses global_scale (the usual choice is amax(|x|) / (6 * 448)).
 *
 *   x_bf16       [rows x K] bf16, row-major, contiguous, 16-byte aligned.
 *   rows, K      rows >= 1, K >= 16, K % 16 == 0.
 *   global_scale finite and > 0.
 *   codes        [rows x K/2] bytes out, 8-byte aligned.
 *   sf_rowmajor  [rows x K/16] bytes out (one E4M3 per 16-element block).
 * Bit-exact (same bytes) as the IEEE reading above on every input without NaN;
 * NaN inputs give unspecified codes.
 */
nvfp4_status nvfp4_quantize(const void* x_bf16, int64_t rows, int64_t K, float global_scale,
                            uint8_t* codes, uint8_t* sf_rowmajor, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_packed -- nvfp4_quantize with the scales written straight into the
 * packed 128x4-atom layout the GEMM reads (the result of nvfp4_pack_scales on
 * nvfp4_quantize's row-major scales, byte for byte, padding included), so that an
 * activation goes quantize -> GEMM with no separate packing pass.
 *
 *   x_bf16, rows, K, global_scale, codes   as nvfp4_quantize.
 *   sf_packed   nvfp4_packed_scales_bytes(rows, K) bytes out, 16-byte aligned;
 *               padding rows and padding micro-blocks are written as zero.
 * Errors as nvfp4_quantize, plus NVFP4_ERR_MISALIGNED for a misaligned sf_packed.
 */
nvfp4_status nvfp4_quantize_packed(const void* x_bf16, int64_t rows, int64_t K, float global_scale,
                                   uint8_t* codes, uint8_t* sf_packed, nvfp4_stream_t stream);

/*
 * nvfp4_quantize_two_pass -- BF16 activations -> a two-pass (value + residual) NVFP4
 * operand for nvfp4_gemm_two_pass.
 *
 * [P2] follow-ups: activations quantised in two NVFP4 passes, value and residual,
 * both consumed by the block-scaled FP4 MMA.  The page gives no formula; this
 * library reads it as
 *   q1 = nvfp4_quantize(x, global_scale)
 *   r  = x - (value(q1 code) * q1 scale) * global_scale     (IEEE float32 steps:
 *        the product is exact, the multiply and the subtraction each round)
 *   q2 = the same quantiser applied to r, with the same global_scale,
 * so that x ~ (dq1 + dq2) * global_scale and one GEMM alpha serves both passes.
 *
 *   x_bf16, rows, global_scale   as nvfp4_quantize.
 *   K           K >= 256 and K % 256 == 0 (else NVFP4_ERR_UNSUPPORTED_SHAPE).
 *   codes2      [rows x K] bytes out (2K codes per row), 8-byte aligned: for each
 *               256-element K-block j of x, bytes [256j, 256j + 128) hold q1's codes of
 *               that block and bytes [256j + 128, 256j + 256) q2's codes of the same
 *               elements (low nibble = even k, as everywhere).
 *   sf2_packed  nvfp4_packed_scales_bytes(rows, 2 * K) bytes out, 16-byte aligned:
 *               the packed layout of a [rows x 2K] operand whose scale column 32j + u
 *               is q1's scale u of K-block j (u < 16) and 32j + 16 + u is q2's.
 * Bytes equal the IEEE reading above on every input without NaN.
 */
nvfp4_status nvfp4_quantize_two_pass(const void* x_bf16, int64_t rows, int64_t K, float global_scale,
                                     uint8_t* codes2, uint8_t* sf2_packed, nvfp4_stream_t stream);

/*
 * Size in bytes of the packed scale-factor buffer of a [rows x K] operand:
 * ceil(rows/128)*128 * ceil(K/64)*4.  Returns 0 for rows < 1 or K < 16 or K % 16 != 0.
 */
size_t nvfp4_packed_scales_bytes(int64_t rows, int64_t K);

/*
 * nvfp4_pack_scales -- row-major scales -> the 128x4-atom layout the GEMM reads.
 *
 * [P1] Version 5: within a 512-byte atom covering 128 rows x 64 K elements, the
 * scale of row m and micro-block b (0..3) sits at byte 16*(m%32) + 4*((m/32)%4) + b;
 * atoms are ordered K-fastest inside a 128-row band.  Padding rows and padding
 * micro-blocks are written as zero.
 *
 *   sf_rowmajor  [rows x K/16] bytes.
 *   rows, K      rows >= 1, K >= 16, K % 16 == 0.
 *   sf_packed    nvfp4_packed_scales_bytes(rows, K) bytes out, 16-byte aligned.
 */
nvfp4_status nvfp4_pack_scales(const uint8_t* sf_rowmajor, int64_t rows, int64_t K,
                               uint8_t* sf_packed, nvfp4_stream_t stream);

/*
 * nvfp4_gemm -- D = bf16(alpha * sum_k (A*SFA)(B*SFB)), FP32 accumulation.
 *
 * [P1] Version 1 (the block-scaled GEMM, K-major operands, BF16 output) and
 * Version 3 (alpha multiplies the FP32 accumulator before the conversion).
 * Runs on the tcgen05 tensor cores (kind::mxf4nvf4, scale_vec::4X).
 *
 *   A      [M x K/2] packed codes, K-major (row m holds k = 0..K-1), 16-byte aligned.
 *   SFA    nvfp4_packed_scales_bytes(M, K) bytes in the packed layout, 16-byte aligned.
 *   B      [N x K/2] packed codes, K-major, 16-byte aligned.
 *   SFB    nvfp4_packed_scales_bytes(N, K) bytes, packed layout, 16-byte aligned.
 *   alpha  finite FP32.
 *   D_bf16 [M x N] bf16 out, row-major, 16-byte aligned.
 *   M, N, K  M >= 1, N >= 8 and N % 8 == 0, K >= 64 and K % 64 == 0.
 * Accuracy: |D - exact| <= 2^-8 |exact| + 1e-6 |alpha| sum_k |a_k b_k| per element.
 * Deterministic: repeated calls give bit-identical D.
 */
nvfp4_status nvfp4_gemm(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                        float alpha, void* D_bf16, int64_t M, int64_t N, int64_t K,
                        nvfp4_stream_t stream);

/*
 * nvfp4_gemm_config -- nvfp4_gemm with an explicit kernel configuration (for tests
 * and tuning).  config 0 is the automatic choice of nvfp4_gemm; the other values
 * are listed by nvfp4_gemm_config_name.  Returns NVFP4_ERR_INVALID_ARG for an
 * unknown config.
 */
nvfp4_status nvfp4_gemm_config(const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
                               const uint8_t* SFB, float alpha, void* D_bf16, int64_t M,
                               int64_t N, int64_t K, int config, nvfp4_stream_t stream);

/*
 * nvfp4_gemm_streamk -- nvfp4_gemm with a stream-K schedule for the CTA-pair kernel.
 *
 * When the 256x256 output tiles are not a whole number of waves of CTA pairs, the
 * last one or two waves' (tile, K-block) units are split evenly over the pairs, each
 * pair taking one contiguous run of them ([P2] Design section, stream-K); a tile
 * shared by two pairs is finished by the second, which adds the first one's FP32
 * partial (written to the workspace) in a fixed order, so repeated calls are
 * bit-identical (not bit-identical to nvfp4_gemm, whose summation order differs).
 * The split is taken only where a cost model in K-blocks per pair, charging the
 * fix-up as 16 K-blocks, predicts a gain over the data-parallel waves (measured:
 * 1024x5120x17408 58 us against 85 us, 1024x5120x5120 31 against 35); otherwise, and
 * for shapes the pair kernel does not take, the call runs as nvfp4_gemm.
 *
 *   A, SFA, B, SFB, alpha, D_bf16, M, N, K   as nvfp4_gemm.
 *   workspace        DEVICE buffer owned by the caller, at least
 *                    nvfp4_gemm_streamk_workspace_bytes() bytes, 16-byte aligned, and
 *                    zero-filled before its first use.  A call that completes without
 *                    a device error leaves it ready for the next one (its flag words
 *                    are back to zero).  Calls that share a workspace must not overlap
 *                    on the device (calls on one stream never do).
 *   workspace_bytes  its size.
 * Errors as nvfp4_gemm, plus NVFP4_ERR_INVALID_ARG for a NULL or too small workspace
 * and NVFP4_ERR_MISALIGNED for a misaligned one.  After NVFP4_ERR_TIMEOUT the
 * workspace must be zero-filled again.
 */
nvfp4_status nvfp4_gemm_streamk(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                                float alpha, void* D_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                                size_t workspace_bytes, nvfp4_stream_t stream);

/* Workspace bytes nvfp4_gemm_streamk needs on the current device (any shape), 0 on error. */
size_t nvfp4_gemm_streamk_workspace_bytes(void);

/*
 * nvfp4_gemm_streamk_noalloc -- nvfp4_gemm_streamk with the workspace held inside the
 * library: a static device array of 20 MiB + 4 KiB per device (flag words plus one
 * 128 KB FP32 partial per CTA of up to 80 CTA pairs).  Neither cited page has a
 * counterpart; it is a library convenience, not part of the method.
 *
 * It is for callers that cannot hand over a device buffer: code with no allocator
 * of its own (a plugin or callback inside a host framework that owns the memory
 * pools), and paths that must not call cudaMalloc/cudaFree because those
 * synchronise the device or because device memory is fully committed.  The call
 * allocates nothing: the array's address is looked up once per device
 * (cudaGetSymbolAddress), and the array comes with the library's module.
 *
 *   A, SFA, B, SFB, alpha, D_bf16, M, N, K, stream   as nvfp4_gemm_streamk, whose
 *                    argument checks, schedule and results (bit for bit) it shares.
 *   reset_scratch    nonzero: zero the array on `stream` before the launch.  The
 *                    first call on each device does this by itself; pass it after a
 *                    call that ended in NVFP4_ERR_TIMEOUT (nvfp4_device_error), which
 *                    can leave flag words raised.
 *
 * There is one array per device, shared by every call on it: calls that overlap on
 * the GPU (other streams, other host threads) race on it and give wrong results or
 * time out.  Calls on one stream never overlap.  The array's address and the
 * "already cleared" state are cached per device for the life of the process, so the
 * entry point is not valid across cudaDeviceReset (or any other teardown of the
 * device's primary context): after one, the cached address may be stale.
 * Errors as nvfp4_gemm_streamk, plus NVFP4_ERR_UNSUPPORTED_DEVICE, before anything is
 * enqueued, when the device's CTA-pair grid needs more workspace than the array holds,
 * and NVFP4_ERR_CUDA when the array's address cannot be looked up.
 */
nvfp4_status nvfp4_gemm_streamk_noalloc(const uint8_t* A, const uint8_t* SFA, const uint8_t* B,
                                        const uint8_t* SFB, float alpha, void* D_bf16, int64_t M, int64_t N,
                                        int64_t K, int reset_scratch, nvfp4_stream_t stream);

/*
 * nvfp4_gemm_two_pass -- D = bf16(alpha * sum_k (dq1[m,k] + dq2[m,k]) * (B*SFB)[n,k]),
 * FP32 accumulation, for a two-pass activation from nvfp4_quantize_two_pass
 * ([P2] follow-ups, value + residual on the block-scaled FP4 MMA).
 *
 * Both passes run on the same tcgen05 kernels as nvfp4_gemm, into one accumulator:
 * the kernels walk the activation's 2K codes and use each 256-element K-block of
 * the weight twice (once for the value block, once for the residual block), so
 * the weight is read from memory once per output tile, as in nvfp4_gemm.
 *
 *   A2, SFA2   codes2 and sf2_packed of nvfp4_quantize_two_pass for [M x K].
 *   B, SFB     the weight as for nvfp4_gemm: [N x K/2] codes, packed scales of [N x K].
 *   alpha      finite FP32 (global scale of the activation x that of the weight).
 *   D_bf16, M, N   as nvfp4_gemm.
 *   K          the weight's K: K >= 256 and K % 256 == 0.
 * Accuracy: |D - exact| <= 2^-8 |exact| + 1e-6 |alpha| sum_k (|dq1_k| + |dq2_k|) |b_k|.
 * Deterministic.  Errors as nvfp4_gemm, plus NVFP4_ERR_UNSUPPORTED_SHAPE for K % 256.
 */
nvfp4_status nvfp4_gemm_two_pass(const uint8_t* A2, const uint8_t* SFA2, const uint8_t* B, const uint8_t* SFB,
                                 float alpha, void* D_bf16, int64_t M, int64_t N, int64_t K, nvfp4_stream_t stream);

/* Name of a GEMM kernel configuration, or NULL past the last one (config >= 1). */
const char* nvfp4_gemm_config_name(int config);

/* Configuration nvfp4_gemm picks for (M, N, K) on the current device (>= 1), or a negative status. */
int nvfp4_gemm_choose_config(int64_t M, int64_t N, int64_t K);

/*
 * Size in bytes of a prepared W4A16 weight: N*K/2 + N*K/16, the size of the
 * checkpoint tensors ([P2] Design, weight-layout paragraph).  0 for invalid N, K.
 */
size_t nvfp4_w4a16_prepared_bytes(int64_t N, int64_t K);

/*
 * nvfp4_w4a16_prepare -- re-lay out an NVFP4 weight once for nvfp4_w4a16_linear.
 *
 * [P2] Design, weight-layout paragraph: codes are moved into the fragment order of the
 * decode kernel, each E4M3 scale is re-encoded as a byte b with
 * bf16(0x7000 | b<<4) == |scale| * 2^119 (exact for every finite E4M3, subnormals
 * included), zero scales zero their codes and negative scales flip their codes'
 * signs.  The byte order is this library's own (specified with the oracle).
 *
 *   W_codes        [N x K/2] packed codes, K-major.
 *   W_sf_rowmajor  [N x K/16] E4M3 scale bytes, row-major (sign allowed; NaN bytes
 *                  give unspecified weights).
 *   N, K           N % 16 == 0, K % 64 == 0, both >= their modulus.
 *   Wprep          nvfp4_w4a16_prepared_bytes(N, K) bytes out, 16-byte aligned.
 */
nvfp4_status nvfp4_w4a16_prepare(const uint8_t* W_codes, const uint8_t* W_sf_rowmajor, int64_t N,
                                 int64_t K, void* Wprep, nvfp4_stream_t stream);

/*
 * nvfp4_w4a16_linear -- y = bf16(alpha * x * dequant(W)^T), FP32 accumulation.
 *
 * [P2] Summary and Design: BF16 activations, NVFP4 weights dequantised in
 * registers, deterministic split-K (here a fixed-order reduction inside a thread
 * block cluster, so no workspace is needed), BF16 output.
 *
 *   x_bf16  [M x K] bf16 row-major, 16-byte aligned.
 *   Wprep   output of nvfp4_w4a16_prepare for (N, K).
 *   alpha   the weight's FP32 global scale.
 *   y_bf16  [M x N] bf16 out, row-major, 16-byte aligned.
 *   M, N, K M >= 1; N % 128 == 0; K % 256 == 0.
 * Accuracy: |y - exact| <= 2^-8 |exact| + 1e-6 |alpha| sum_k |x_k w_k|.
 * Deterministic: repeated calls give bit-identical y.
 */
nvfp4_status nvfp4_w4a16_linear(const void* x_bf16, const void* Wprep, float alpha, void* y_bf16,
                                int64_t M, int64_t N, int64_t K, nvfp4_stream_t stream);

/*
 * Size in bytes of the workspace nvfp4_w4a16_linear_streamk needs on the current
 * device: for up to 32 tokens two FP32 partial slots of 32 tokens x 256 rows and two
 * tickets per SM, then for more tokens two slots of 128 rows x 256 tokens and one
 * ticket per SM (about 320 KB per SM in all); 0 if no device can be queried.
 */
size_t nvfp4_w4a16_streamk_workspace_bytes(void);

/*
 * nvfp4_w4a16_linear_streamk -- nvfp4_w4a16_linear (or its per-column form) with the
 * work split evenly over the SMs.
 *
 * [P2] Design, the persistent stream-K kernel: for up to 32 tokens one thread block
 * per SM takes an equal contiguous share of the units (256 weight rows x 64 K) in
 * row-group-major order, whatever N and K.  A row group split between blocks is
 * summed through the workspace: each part stores its FP32 partial and takes a ticket,
 * and the part that takes the last ticket adds all partials in part order (so the
 * result does not depend on which part finishes last), writes y and zeroes the
 * ticket.  No block waits for another.  More than 32 tokens run the same scheme on
 * the tensor-core kernel: units of (token tile of up to 256 tokens, 128 weight rows,
 * 64 K) over one block per SM, each block dequantising its weights into shared
 * memory for tcgen05 BF16 MMAs, with the partials and tickets in the workspace's
 * second region.
 *
 *   x_bf16, Wprep, y_bf16, M, N, K   as nvfp4_w4a16_linear.
 *   alpha        the global scale, used when alpha_col is NULL (then finite).
 *   alpha_col    NULL, or N FP32 per-output-column scales (16-byte aligned), as in
 *                nvfp4_w4a16_linear_colscale; alpha is then ignored.
 *   workspace    DEVICE buffer owned by the caller, at least
 *                nvfp4_w4a16_streamk_workspace_bytes() bytes, 16-byte aligned,
 *                zero-filled before its first use.  Every completed call leaves its
 *                tickets at zero again, so the buffer needs no clearing between
 *                calls (or CUDA-graph replays).  Calls that share a workspace must
 *                not overlap in time; give concurrent streams their own.
 *   workspace_bytes  its size.
 * Errors as nvfp4_w4a16_linear, plus NVFP4_ERR_INVALID_ARG for a NULL or too small
 * workspace.  After a call that reported a device error (nvfp4_device_error) the
 * workspace must be zero-filled again.
 * Accuracy as nvfp4_w4a16_linear.  Deterministic: repeated calls with the same
 * shapes on the same device give bit-identical y (the split depends on the SM count).
 */
nvfp4_status nvfp4_w4a16_linear_streamk(const void* x_bf16, const void* Wprep, float alpha, const float* alpha_col,
                                        void* y_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                                        size_t workspace_bytes, nvfp4_stream_t stream);

/*
 * nvfp4_w4a16_linear_colscale -- nvfp4_w4a16_linear with one FP32 weight scale per
 * output column instead of the global alpha:
 *
 *     y[m, n] = bf16(alpha_col[n] * sum_k x[m, k] * dequant(W)[n, k]),  FP32 accumulation.
 *
 * [P2] Design: the weight scale may be global or per output column.  Same kernels,
 * arguments and rules as nvfp4_w4a16_linear, except:
 *   alpha_col  [N] FP32, DEVICE pointer owned by the caller, 16-byte aligned; read
 *              once per output element (finite values assumed, not checked).
 * Accuracy: |y - exact| <= 2^-8 |exact| + 1e-6 |alpha_col[n]| sum_k |x_k w_k|.
 * Errors: NVFP4_ERR_INVALID_ARG for a NULL alpha_col, NVFP4_ERR_MISALIGNED if it is
 * not 16-byte aligned, otherwise as nvfp4_w4a16_linear.
 */
nvfp4_status nvfp4_w4a16_linear_colscale(const void* x_bf16, const void* Wprep, const float* alpha_col,
                                         void* y_bf16, int64_t M, int64_t N, int64_t K, nvfp4_stream_t stream);

/*
 * nvfp4_device_error -- synchronise `stream`, then read the device-side error word
 * of the current device.  Kernels never trap: a kernel that gives up one of its
 * bounded waits (a pipeline barrier that did not complete within its time limit)
 * records NVFP4_ERR_TIMEOUT there and returns early.  Returns NVFP4_OK if the word
 * is clear, the recorded status otherwise, NVFP4_ERR_CUDA if the synchronisation
 * failed.  clear != 0 resets the word.
 */
nvfp4_status nvfp4_device_error(nvfp4_stream_t stream, int clear);

/*
 * nvfp4_mma_ceiling -- diagnostic: the tensor-core instruction ceiling of the device.
 *
 * Every CTA pair issues `iters` tcgen05.mma.cta_group::2 instructions (M = 256, N = 256,
 * operands resident in shared memory, FP32 accumulator in TMEM) of one kind back to
 * back: kind 0 = block-scaled E2M1 (kind::mxf4nvf4, scale_vec::4X, the GEMM's
 * instruction), 1 = BF16 (kind::f16), 2 = E4M3 (kind::f8f6f4).  Writes the achieved
 * TFLOP/s over the slowest pair and the median clock cycles per instruction.  It is
 * synchronous on `stream` and independent of any operand data.
 *   kind     0, 1 or 2.
 *   iters    instructions per pair, a multiple of 4 in [4, 2^24].
 *   tflops, cycles_per_mma   HOST pointers (either may be NULL).
 * Errors: NVFP4_ERR_INVALID_ARG for a bad kind or iters, NVFP4_ERR_TIMEOUT if the
 * instructions did not complete within 2 s, NVFP4_ERR_CUDA, NVFP4_ERR_UNSUPPORTED_DEVICE.
 */
nvfp4_status nvfp4_mma_ceiling(int kind, int iters, double* tflops, double* cycles_per_mma,
                               nvfp4_stream_t stream);

/*
 * nvfp4_test_streamk_fault -- FOR TESTS ONLY: fault injection into the stream-K
 * schedule of nvfp4_gemm_streamk / nvfp4_gemm_streamk_noalloc on the current device.
 * No counterpart on the cited pages; it exists to exercise the timeout path without
 * faulting, trapping or hanging the GPU.
 *
 *   skip_publish   nonzero: the pairs that start a shared tile (stream-K "heads")
 *                  do not publish their partial, so the pairs that finish it wait on
 *                  a flag that nothing sets; 0: normal operation.
 *   flag_wait_ns   limit of those flag waits in nanoseconds (0 = the default 2 s).
 *
 * With skip_publish set, a launch that splits tiles ends (no hang) with
 * nvfp4_device_error reporting NVFP4_ERR_TIMEOUT; its output is undefined.  Call
 * again with (0, 0) to restore normal operation, then re-zero the stream-K workspace
 * (or pass reset_scratch to nvfp4_gemm_streamk_noalloc) before the next stream-K call.
 * Synchronous (device-global settings); not for use while stream-K launches run.
 * Errors: NVFP4_ERR_UNSUPPORTED_DEVICE, NVFP4_ERR_CUDA.
 */
nvfp4_status nvfp4_test_streamk_fault(int skip_publish, uint64_t flag_wait_ns);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H_ */

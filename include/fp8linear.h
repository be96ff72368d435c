/*
 * fp8linear.h - C ABI of the FP8 E4M3 quantized linear layer for one NVIDIA
 * GB300 GPU (sm_103a).
 *
 * The layer (page titles and the parts of the pages that define it):
 *  - "[Kernel][FP8] Initial support with dynamic per-tensor scaling",
 *    Algorithm: weights are quantized once with a per-tensor scale; the
 *    activation scale is computed in every forward pass; the forward pass is
 *    a cast to float8_e4m3fn followed by a scaled matrix product
 *    (torch._scaled_mm in the microbenchmark list).
 *  - "RFC: FP8 Quantization Schema in vLLM", Scope and Interface Content:
 *    OCP FP8_E4M3 numbers; static input scales; an output scale that lets a
 *    GEMM emit FP8_E4M3 directly (the output_scale discussion).
 *  - "Marlin fp8", kernel argument checks: a weight-only FP8 product for
 *    16-bit activations whose weight scale is one value per output channel
 *    (b_scales of shape [1, N]).
 *  - "RFC: FP8 Quantization Schema in vLLM", the gate_proj question: FP8 GEMM
 *    shapes must be divisible by 16.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library never allocates, frees or keeps device memory between calls.
 *  - Tensors are dense and row-major: X / A are [M, K], W is [N, K] (the
 *    nn.Linear layout; both product operands have K contiguous), Y is [M, N].
 *  - E4M3 tensors are arrays of uint8 codes (OCP float8_e4m3fn bit patterns).
 *  - Scales are float32 values in DEVICE memory, so a dynamic scale written
 *    by one call is consumed by the next without a host round trip.
 *  - Tensor pointers must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    only enqueue work: they return before the GPU finishes, never
 *    synchronize, and a return of FP8L_OK means the work was launched.
 *  - Errors found on the host (FP8L_EINVAL, FP8L_ESHAPE, FP8L_EALIGN,
 *    FP8L_EUNSUPPORTED) are returned before anything is launched and leave
 *    every output untouched.  FP8L_ECUDA reports a failed CUDA call or
 *    launch.  Device-side wait time-outs are recorded in the workspace (or,
 *    for fp8_w8a16_mm, in a status word of the library) and reported by
 *    fp8l_read_status().
 *  - Inputs must be finite.  NaN or Inf input is outside the contract.
 */
#ifndef FP8LINEAR_H
#define FP8LINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI version (fp8l_abi_version): 1, the first release; 2 adds
 * fp8_pack_w8a16_weights, fp8_packed_weight_bytes and FP8L_WEIGHTS_PACKED;
 * 3 adds fp8l_debug_waits, the per-token activation scales
 * (FP8L_A_PER_TOKEN), fp8_rmsnorm_quant and fp8_grouped_mm.  Each change is additive: a caller written for an
 * earlier version runs unchanged. */
#define FP8L_ABI_VERSION 7

/* Only the entry points below are exported from the shared library. */
#if defined(__GNUC__)
#define FP8L_API __attribute__((visibility("default")))
#else
#define FP8L_API
#endif

/* Status codes returned by every entry point. */
enum fp8l_status {
    FP8L_OK = 0,
    FP8L_EINVAL = 1,      /* null pointer, unknown dtype or flag value      */
    FP8L_ESHAPE = 2,      /* a size is negative, too large, or breaks a
                             multiple-of-16 rule                            */
    FP8L_EALIGN = 3,      /* a tensor pointer is not 16-byte aligned        */
    FP8L_ECUDA = 4,       /* a CUDA call or kernel launch failed            */
    FP8L_ETIMEOUT = 5,    /* a device-side wait gave up (fp8l_read_status)  */
    FP8L_EUNSUPPORTED = 6 /* the current device is not compute capability
                             10.3, or the dtype combination is unsupported  */
};

/* Flags of the product entry points.
 *
 * FP8L_WEIGHTS_STABLE: the caller guarantees that no work still in flight on
 * `stream` writes the weights `w` or the weight scales (the usual case of an
 * inference loop, where weights are written once at load time).  The
 * product's kernel is then launched as a programmatic dependent of the
 * preceding kernel on the stream, so it is resident before that kernel
 * ends; the weight-streaming kernel also issues its first weight loads
 * before waiting for it, so consecutive products overlap.  Activations,
 * scales and outputs are only accessed after the wait. */
#define FP8L_WEIGHTS_STABLE 1u

/* FP8L_WEIGHTS_PACKED (fp8_w8a16_mm only): `w` holds the weights in the
 * packed layout written by fp8_pack_w8a16_weights, not as [N, K] rows. */
#define FP8L_WEIGHTS_PACKED 2u

/* FP8L_A_PER_TOKEN (fp8_scaled_mm only): a_scale holds M values, one per
 * row of `a` (per-token activation scales, as fp8_quant_per_row computes
 * them for activations), instead of one. */
#define FP8L_A_PER_TOKEN 4u

/* FP8L_SINGLE_SM_TILES (fp8_scaled_mm only): run a tensor-core product
 * with one SM per 128 x 256 tile even where it would pair two SMs on a
 * 256 x 256 tile (a tuning and testing option; both kernels accumulate in
 * fp32 over k in the same blocks, and their results agree within the
 * layer's tolerance). */
#define FP8L_SINGLE_SM_TILES 8u

/* Kernel choice of fp8_scaled_mm (a tuning and testing option; every
 * kernel accumulates in fp32 and their results agree within the layer's
 * tolerance).  FP8L_KERNEL_AUTO (0) picks by M as fp8_scaled_mm describes.
 *   FP8L_KERNEL_STREAM   weight streaming on the CUDA cores (mma.sync),
 *                        any M, in groups of 16 rows;
 *   FP8L_KERNEL_SWAPPED  tcgen05 product with the operands swapped (128
 *                        weight rows by M tokens per tile), 1 <= M <= 128
 *                        (FP8L_ESHAPE otherwise);
 *   FP8L_KERNEL_TILED    tcgen05 product on token x channel tiles, any M. */
#define FP8L_KERNEL_AUTO 0u
#define FP8L_KERNEL_STREAM 16u
#define FP8L_KERNEL_SWAPPED 32u
#define FP8L_KERNEL_TILED 48u
#define FP8L_KERNEL_MASK 48u

/* Element types. */
enum fp8l_dtype {
    FP8L_F16 = 0,   /* IEEE binary16                                         */
    FP8L_BF16 = 1,  /* bfloat16                                              */
    FP8L_E4M3 = 2,  /* OCP float8_e4m3fn code (uint8)                        */
    FP8L_F32 = 3    /* IEEE binary32 (quantizer input only)                  */
};

/* Size in bytes of the workspace that fp8_quant_per_tensor (dynamic mode)
 * and fp8_scaled_mm need.  The caller allocates it once (device memory,
 * 16-byte aligned), fills it with zeros once, and may reuse it for every
 * later call on streams that do not run those calls concurrently.  It holds
 * a device status word and the dynamic quantizer's grid-barrier words (a call
 * counter, two arrival counts and two maximum words used by alternate calls,
 * and per-block partial maxima); the library keeps nothing else in it between
 * calls.  A call whose device-side wait gave up may leave the barrier words
 * mid-call; fp8l_read_status, when it reports FP8L_ETIMEOUT, zeroes them
 * (bytes [0, 32)) before it returns, so the workspace is ready again. */
FP8L_API size_t fp8l_workspace_bytes(void);

/* Per-tensor quantization of a [rows, cols] activation or weight tensor
 * to E4M3 ("[Kernel][FP8] Initial support with dynamic per-tensor scaling",
 * Algorithm; static scales: "RFC: FP8 Quantization Schema in vLLM", Scope).
 *
 *   dynamic != 0:  amax  = max_i |x_i|                       (exact)
 *                  s     = amax / 448  (one fp32 IEEE division; s = 1 when
 *                          that quotient is 0, i.e. for an all-zero tensor)
 *                  *scale = s is written to device memory
 *   dynamic == 0:  s = *scale is read from device memory (a static,
 *                  calibrated input_scale); it must be positive and finite
 *   every element: q_i = E4M3(fp32(x_i / s)), the quotient being one fp32
 *                  IEEE division and E4M3() the saturating
 *                  round-to-nearest-even cast (|v| >= 448 gives +-448; the
 *                  sign is kept, so negatives that round to 0 give 0x80).
 *
 * x:         [rows, cols] of x_dtype (FP8L_F16, FP8L_BF16 or FP8L_F32).
 * q:         [rows, cols] uint8 codes (output).
 * scale:     one float (output when dynamic, input otherwise).
 * workspace: fp8l_workspace_bytes() bytes; may be NULL when dynamic == 0.
 * rows*cols may be 0 (then only the dynamic scale, 1.0f, is written) and
 * at most 2^40.  The result is bit-for-bit deterministic. */
FP8L_API int fp8_quant_per_tensor(const void *x, int x_dtype, int64_t rows, int64_t cols,
                         uint8_t *q, float *scale, int dynamic,
                         void *workspace, void *stream);

/* Per-row quantization, one dynamic scale per row: the per-output-channel
 * weight scale of "Marlin fp8" (b_scales [1, N]).  Row r is quantized
 * exactly as fp8_quant_per_tensor(dynamic=1) would quantize it alone, and
 * its scale is written to row_scale[r].  Used once after weights are loaded
 * ("[Kernel][FP8] Initial support ...", Algorithm).
 *
 * x: [rows, cols] of x_dtype (FP8L_F16, FP8L_BF16 or FP8L_F32);
 * q: [rows, cols] uint8; row_scale: [rows] float.  cols must be a multiple
 * of 16 and at most 2^20; rows at most 2^31 - 1. */
FP8L_API int fp8_quant_per_row(const void *x, int x_dtype, int64_t rows, int64_t cols,
                      uint8_t *q, float *row_scale, void *stream);

/* W8A8 scaled matrix product ("[Kernel][FP8] Initial support ...",
 * torch._scaled_mm; per-channel weight scales: "Marlin fp8"; E4M3 output
 * through output_scale: "RFC: FP8 Quantization Schema in vLLM").
 *
 *   acc[m,n] = sum_k dec(a[m,k]) * dec(w[n,k])      (fp32 accumulation)
 *   v[m,n]   = acc[m,n] * as(m) * ws(n)             ws(n) = w_scale[n] when
 *                                                   w_per_channel, else w_scale[0];
 *                                                   as(m) = a_scale[m] with
 *                                                   FP8L_A_PER_TOKEN, else a_scale[0]
 *   out_dtype FP8L_BF16 / FP8L_F16: y[m,n] = v[m,n] rounded to nearest
 *   out_dtype FP8L_E4M3:            y[m,n] = E4M3(v[m,n] / out_scale[0])
 *
 * a: [M, K] E4M3 codes; w: [N, K] E4M3 codes; y: [M, N] of out_dtype.
 * a_scale: 1 float (M floats with FP8L_A_PER_TOKEN: finer-than-per-tensor
 * scales, which "RFC: FP8 Quantization Schema in vLLM", Scope, leaves for
 * later; read here as one scale per token); w_scale: 1 or N floats;
 * out_scale: 1 float, required
 * when out_dtype is FP8L_E4M3 and ignored otherwise.
 * M >= 0 (M == 0 launches nothing); N and K are positive multiples of 16
 * (the FP8 GEMM shape rule), N, K <= 2^20, M <= 2^31 - 1.
 * Kernels (fp8_scaled_mm_kernel names the one a call runs): up to 16 tokens
 * with small weights, weight streaming on the CUDA cores; up to 128 tokens,
 * a tcgen05 product with the operands swapped (128 weight rows by the
 * tokens per tile, clusters of CTAs splitting K when the weight blocks are
 * few); otherwise tcgen05 token x channel tiles: a persistent kernel whose
 * 256 x 256 tiles each span a pair of SMs (tcgen05.mma.cta_group::2), or
 * 128 x 256 tiles on one SM each with FP8L_SINGLE_SM_TILES, or clusters
 * splitting K when the tiles are few.  workspace: fp8l_workspace_bytes()
 * bytes (status word).  flags: any of FP8L_WEIGHTS_STABLE,
 * FP8L_A_PER_TOKEN, FP8L_SINGLE_SM_TILES and one FP8L_KERNEL_* choice
 * (other bits are FP8L_EINVAL; FP8L_KERNEL_SWAPPED with M > 128 is
 * FP8L_ESHAPE). */
FP8L_API int fp8_scaled_mm(const uint8_t *a, const uint8_t *w, int64_t M, int64_t N,
                  int64_t K, const float *a_scale, const float *w_scale,
                  int w_per_channel, const float *out_scale, void *y,
                  int out_dtype, void *workspace, unsigned flags, void *stream);

/* Largest x (bytes) of a dynamic-scale fp8_quant_scaled_mm: every CTA of the
 * product reads all of it to take its maximum. */
#define FP8L_FUSED_DYNAMIC_MAX_BYTES 65536

/* W8A8 product of few tokens with the activation quantization fused into it
 * ("Condition to achieve linear speedup?": quantization fused into another
 * kernel instead of its own launch; "RFC: FP8 Quantization Schema in
 * vLLM": static input scales):
 *
 *   dynamic:  a_scale[0] = amax(|x|) / 448 (1 if that is 0), written
 *   static:   a_scale[0] read
 *   a = E4M3(x / a_scale[0])  (the codes of fp8_quant_per_tensor, bit for bit)
 *   y = fp8_scaled_mm(a, w, a_scale, w_scale, ...)
 *
 * in one kernel and without writing the codes: the kernel fp8_scaled_mm
 * runs for the shape (fp8_scaled_mm_kernel; its token x channel tiles
 * excepted, which become the swapped-operand product) with the codes made
 * from x inside it, so up to 64 tokens the result is bit-for-bit that of
 * fp8_quant_per_tensor followed by fp8_scaled_mm with the same kernel
 * choice (above, the 16-bit token stages of the swapped-operand product
 * leave room for one CTA per SM, K may be split over fewer CTAs and the
 * fp32 sums round differently, within the layer's tolerance).  x: [M, K] of
 * x_dtype
 * (FP8L_F16 or FP8L_BF16), 0 <= M <= 128 (FP8L_ESHAPE above); a dynamic
 * scale also needs 2 M K <= FP8L_FUSED_DYNAMIC_MAX_BYTES (every CTA reads
 * all of x; FP8L_ESHAPE otherwise).  w, w_scale, w_per_channel, out_scale,
 * y, out_dtype and workspace as for fp8_scaled_mm; per-tensor a_scale only.
 * flags: FP8L_WEIGHTS_STABLE and one of FP8L_KERNEL_STREAM (the CUDA-core
 * weight stream, up to 16 tokens: FP8L_ESHAPE above) or
 * FP8L_KERNEL_SWAPPED (other bits, FP8L_KERNEL_TILED among them, are
 * FP8L_EINVAL). */
FP8L_API int fp8_quant_scaled_mm(const void *x, int x_dtype, const uint8_t *w, int64_t M,
                                 int64_t N, int64_t K, float *a_scale, int dynamic,
                                 const float *w_scale, int w_per_channel,
                                 const float *out_scale, void *y, int out_dtype,
                                 void *workspace, unsigned flags, void *stream);

/* 1 when fp8_quant_scaled_mm accepts this shape (dynamic: the scale is
 * taken in the call) and was measured faster on a GB300 than
 * fp8_quant_per_tensor followed by fp8_scaled_mm, else 0.  On the
 * swapped-operand product: up to 8 tokens with at most 304 blocks of 128
 * weight rows, 9 to 16 tokens with at most 152 (beyond, every CTA converts
 * all the tokens of its K range itself, and with fewer weight stages in
 * flight than the plain product a CTA streams its weights more slowly).  On
 * the CUDA-core weight stream (small weights): up to 8 tokens, or
 * M * K <= 16384.  A pure function of its arguments; needs no GPU. */
FP8L_API int fp8_quant_scaled_mm_preferred(int64_t M, int64_t N, int64_t K, int dynamic);

/* The kernel fp8_scaled_mm runs for this shape and these flags:
 * FP8L_KERNEL_STREAM, FP8L_KERNEL_SWAPPED or FP8L_KERNEL_TILED (the flags'
 * own choice when they make one).  A pure function of its arguments; needs
 * no GPU. */
FP8L_API unsigned fp8_scaled_mm_kernel(int64_t M, int64_t N, int64_t K, unsigned flags);

/* W8A16 weight-only product ("Marlin fp8"): 16-bit activations times E4M3
 * weights with one scale per output channel.
 *
 *   y[m,n] = w_scale[n] * sum_k x[m,k] * dec(w[n,k])  (fp32 accumulation,
 *            rounded to nearest in x_dtype)
 *
 * x: [M, K] of x_dtype (FP8L_F16 or FP8L_BF16); w: [N, K] E4M3 codes, or
 * with FP8L_WEIGHTS_PACKED the packed layout of them
 * (fp8_pack_w8a16_weights; the result is bit-for-bit the same);
 * w_scale: [N] floats; y: [M, N] of x_dtype.  M >= 0; N and K positive
 * multiples of 16, at most 2^20.  Built for decode batches.  Kernels
 * (fp8_w8a16_mm_kernel names the one a call runs): up to 16 tokens, and
 * above 64, a weight-streaming kernel on the CUDA cores (a larger M is
 * computed correctly in groups of 16 rows, each group re-reading W); from
 * 17 to 64 tokens a tcgen05 product that widens the weights to x_dtype
 * (exactly) into tensor memory, 128 weight rows by the tokens per tile.  The
 * tcgen05 kernel's device-side waits are bounded; a time-out is recorded in
 * a status word held by the library (this call takes no workspace) and
 * reported by the next fp8l_read_status.  flags: any of
 * FP8L_WEIGHTS_STABLE and FP8L_WEIGHTS_PACKED, and FP8L_KERNEL_STREAM or
 * FP8L_KERNEL_SWAPPED (the tcgen05 kernel; FP8L_ESHAPE above 64 tokens);
 * other bits, and FP8L_KERNEL_TILED, are FP8L_EINVAL. */
FP8L_API int fp8_w8a16_mm(const void *x, int x_dtype, const uint8_t *w,
                 const float *w_scale, int64_t M, int64_t N, int64_t K,
                 void *y, unsigned flags, void *stream);

/* The kernel fp8_w8a16_mm runs for this shape and these flags:
 * FP8L_KERNEL_STREAM or FP8L_KERNEL_SWAPPED (the flags' own choice when
 * they make one).  A pure function of its arguments; needs no GPU. */
FP8L_API unsigned fp8_w8a16_mm_kernel(int64_t M, int64_t N, int64_t K, unsigned flags);

/* Grouped W8A8 product for mixture-of-experts layers ("RFC: FP8
 * Quantization Schema in vLLM", the gate_proj question: FP8 products need
 * shapes divisible by 16; the experts' products are FP8, and a gate whose
 * expert count is not a multiple of 16 is run through fp8_scaled_mm with
 * its weights padded by zero rows to the next multiple of 16, the extra
 * output columns then being exactly 0).  The tokens routed to expert e are
 * the rows group_offsets[e] .. group_offsets[e+1]-1 of `a`:
 *
 *   y[m,n] = E(acc_e[m,n] * as(m) * ws_e(n))   for those rows, with
 *   acc_e[m,n] = sum_k dec(a[m,k]) * dec(w[e][n,k])   (fp32 accumulation)
 *   ws_e(n) = w_scale[e*N + n] when w_per_channel, else w_scale[e];
 *   as(m) and the output cast E() as in fp8_scaled_mm.
 *
 * a: [M, K] E4M3 codes (rows sorted by expert); w: [num_groups, N, K] E4M3
 * codes; group_offsets: num_groups + 1 int32 in DEVICE memory (written by
 * the routing step, read by the kernel, so no host round trip), with
 * 0 <= offsets[0] <= offsets[1] <= ... <= offsets[num_groups] <= M; rows
 * outside [offsets[0], offsets[num_groups]) are not written (values are
 * clamped to [0, M] and made non-decreasing).  a_scale: 1 float, or M with
 * FP8L_A_PER_TOKEN; w_scale: num_groups floats, or num_groups * N with
 * w_per_channel; out_scale and out_dtype as in fp8_scaled_mm.
 * 1 <= num_groups <= 256; N, K positive multiples of 16 at most 2^20;
 * num_groups * N < 2^31; 0 <= M <= 2^31 - 1.  Runs the tcgen05 kernel with
 * one persistent CTA per SM whatever the group sizes.  workspace: status
 * word.  flags: any of FP8L_WEIGHTS_STABLE and FP8L_A_PER_TOKEN. */
FP8L_API int fp8_grouped_mm(const uint8_t *a, const uint8_t *w, const int32_t *group_offsets,
                            int64_t num_groups, int64_t M, int64_t N, int64_t K,
                            const float *a_scale, const float *w_scale, int w_per_channel,
                            const float *out_scale, void *y, int out_dtype, void *workspace,
                            unsigned flags, void *stream);

/* Size in bytes of the packed layout of an [N, K] E4M3 weight tensor:
 * N * ceil(K / 64) * 64.  Returns 0 when N or K is not a positive multiple
 * of 16 at most 2^20. */
FP8L_API size_t fp8_packed_weight_bytes(int64_t N, int64_t K);

/* Repacks [N, K] E4M3 weight codes, once after they are loaded, into the
 * order in which the W8A16 kernel reads them (Marlin-format weights are
 * permuted at packing time to match the tensor-core mma fragments:
 * "Condition to achieve linear speedup?").  fp8_w8a16_mm with
 * FP8L_WEIGHTS_PACKED then reads each 16-channel group's weights as one
 * contiguous block, 512 contiguous bytes per warp load.
 *
 * Layout, with C = ceil(K / 64): output channel n = 16G + 8h + g (g < 8,
 * h < 2) and k = 64c + 16t + j (t < 4, j < 16) go to byte
 *     (G * C + c) * 1024 + h * 512 + (4g + t) * 16 + j;
 * bytes with k >= K are zero.
 *
 * w: [N, K] codes (16-byte aligned); w_packed: fp8_packed_weight_bytes(N, K)
 * bytes (16-byte aligned, not overlapping w), written in full.  N and K are
 * positive multiples of 16, at most 2^20.  Asynchronous on `stream`; the
 * codes are only moved, never changed. */
FP8L_API int fp8_pack_w8a16_weights(const uint8_t *w, int64_t N, int64_t K,
                                    uint8_t *w_packed, void *stream);

/* Modes of fp8_rmsnorm_quant. */
#define FP8L_NQ_DYNAMIC 0   /* per-tensor scale amax|h| / 448, written to *scale    */
#define FP8L_NQ_STATIC 1    /* per-tensor scale read from *scale (input_scale)     */
#define FP8L_NQ_PER_TOKEN 2 /* scale[m] = amax_k |h[m,k]| / 448, M scales written   */
#define FP8L_NQ_NORM_ONLY 3 /* h only, no codes: the unfused layer's norm step     */

/* RMS normalization with the activation quantization fused into it
 * ("Condition to achieve linear speedup?": the quantization of the
 * activations is fused into the element-wise kernel before the product,
 * such as RMSNorm, instead of a separate pass; the pages do not define
 * RMSNorm, so this is the plain Llama definition).  Per row m:
 *
 *   r[m]   = 1 / sqrt( (1/K) sum_k x[m,k]^2 + eps )   (float32, IEEE ops)
 *   h[m,k] = RN16( (x[m,k] * r[m]) * gamma[k] )      (x's 16-bit format)
 *   codes  = the E4M3 quantization of h, exactly as fp8_quant_per_tensor
 *            (FP8L_NQ_DYNAMIC / FP8L_NQ_STATIC) or fp8_quant_per_row
 *            (FP8L_NQ_PER_TOKEN) quantize the 16-bit tensor h.
 *
 * x: [M, K] of x_dtype (FP8L_F16 or FP8L_BF16); gamma: [K] of x_dtype;
 * eps >= 0 and finite.  q: [M, K] uint8 codes (unused in FP8L_NQ_NORM_ONLY).
 * scale: 1 float (written in FP8L_NQ_DYNAMIC, read in FP8L_NQ_STATIC) or M
 * floats (FP8L_NQ_PER_TOKEN); unused in FP8L_NQ_NORM_ONLY.  h: NULL, or
 * [M, K] of x_dtype receiving the normalized activations (required in
 * FP8L_NQ_NORM_ONLY); the codes are the same whether or not h is written.
 * workspace: fp8l_workspace_bytes() bytes, required in FP8L_NQ_DYNAMIC
 * (grid barrier words and status word), optional otherwise (status word).
 * K is a positive multiple of 16 and at most 32768; 0 <= M <= 2^31 - 1
 * (M == 0 writes only the dynamic scale, 1.0f).  Deterministic. */
FP8L_API int fp8_rmsnorm_quant(const void *x, int x_dtype, const void *gamma, float eps,
                               int64_t M, int64_t K, uint8_t *q, float *scale, int mode,
                               void *h, void *workspace, void *stream);

/* Dynamic per-tensor quantization that allocates nothing and takes no
 * workspace.  The pages have no counterpart to this entry point.
 *
 * It is for callers that cannot allocate device memory themselves: for
 * example a plug-in running inside a framework that owns every device
 * allocation through its own pool, or a serving loop whose memory footprint
 * is fixed at start-up and that has no workspace to pass down.  It computes
 * exactly what fp8_quant_per_tensor computes with dynamic != 0 (same codes,
 * same scale, bit for bit), with the same arguments minus `dynamic` and
 * `workspace`.
 *
 * Scratch: the per-block partial maxima and a ticket counter live in an
 * array of 2048 + 64 floats (8448 bytes) inside the library image, which
 * every GPU that loads the library holds until the process exits.  A call
 * never needs more than those 2048 partial entries, so every size
 * fp8_quant_per_tensor accepts is accepted here; rows*cols above 2^40 is
 * rejected with FP8L_ESHAPE.  Every call on a device shares that one array:
 * calls whose kernels may overlap on the GPU (different streams without
 * ordering between them) race on it and must not be issued.  Only the
 * ticket counter must start at zero: it is zero when the library loads and
 * every completed call leaves it at zero; each call writes the partial
 * entries it reads.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it together with
 * the id of the CUDA context it was taken in; a call made while another
 * context is current on that device (a context created after
 * cudaDeviceReset, or the caller's own) looks it up again for that context.
 * Make the first call in each context before any stream capture begins.
 * The entry point calls no cudaMalloc, cudaFree or other allocating
 * routine. */
FP8L_API int fp8_quant_per_tensor_noalloc(const void *x, int x_dtype, int64_t rows,
                                          int64_t cols, uint8_t *q, float *scale,
                                          void *stream);

/* Waits for `stream`, then reads and clears the workspace's status word and
 * the library's own status word on the current device (where
 * fp8_w8a16_mm, which takes no workspace, records its time-outs; looked up
 * per CUDA context like the no-alloc quantizer's scratch, so make a first
 * call before any stream capture).  Returns FP8L_OK, FP8L_ETIMEOUT if a
 * device-side wait of an earlier call gave up (that call's outputs are then
 * undefined; the workspace's barrier words are zeroed as well, so the next
 * call starts clean), or FP8L_ECUDA. */
FP8L_API int fp8l_read_status(void *workspace, void *stream);

/* Testing hook for the bounded device-side waits (this library's failure
 * detection; the pages have no counterpart).  Every device-side wait of the
 * tcgen05 product and of the dynamic quantizer gives up after a limit,
 * records FP8L_ETIMEOUT in the workspace status word, lets the block's
 * copies in flight land, frees what the block holds and returns, so the
 * CUDA context stays usable.  This call lets a test drive that path without
 * faulting or hanging a GPU.  For every later launch, on every device:
 *   wait_cycles > 0    limit, in SM clock cycles, of the main waits (the
 *                      product's stage and accumulator waits, the
 *                      quantizer's stage waits and grid barrier); 0 restores
 *                      the default of 2^32 cycles (about 2 s).  Waits that
 *                      drain copies in flight before a block exits always
 *                      keep the default.
 *   FP8L_STALL_MMA     the product's MMA role first waits on a barrier that
 *                      nothing completes;
 *   FP8L_STALL_GRID    the dynamic quantizer's grid barrier waits for one
 *                      block more than the grid has.
 * A stalled call's outputs are undefined; fp8l_read_status reports
 * FP8L_ETIMEOUT and resets the workspace.  The setting is process-wide and
 * meant for tests only.  Returns FP8L_EINVAL for a negative limit or an
 * unknown bit. */
#define FP8L_STALL_MMA 1u
#define FP8L_STALL_GRID 2u
FP8L_API int fp8l_debug_waits(long long wait_cycles, unsigned stall_mask);

/* Static, human-readable name of a status code. */
FP8L_API const char *fp8l_strerror(int status);

/* FP8L_ABI_VERSION of the built library. */
FP8L_API int fp8l_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8LINEAR_H */

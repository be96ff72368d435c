// Weight-streaming products for small token counts (up to 16 tokens per CTA):
//   * W8A16 ("Marlin fp8"): fp16/bf16 activations x E4M3 weights with one
//     scale per output channel;
//   * W8A8 small-M branch of the scaled product ("[Kernel][FP8] Initial
//     support ...", the M = 1..16 rows of the microbenchmark list, where the
//     product is bound by reading the weights).
//
// Design (HBM-bound: the weights are read once, every other operand is small)
//   * One CTA owns 16 output channels (rows of W) and one group of up to 16
//     tokens; its 16 warps split K in 64-element chunks (chunk c goes to warp
//     c mod 16), then add their partial tiles in shared memory.  A warp
//     loads two chunks before computing (four for one token tile on packed
//     weights: a K = 4096 slab in a single round trip), and two CTAs fit on
//     an SM.
//   * Lane (g, t) = (lane / 4, lane % 4) reads 16 contiguous weight bytes
//     of channel rows g and g + 8 per chunk with one streaming 16-byte load
//     each (a warp load covers 8 rows x 64 contiguous bytes).  The K order
//     inside a chunk is permuted identically for weights and activations, so
//     every lane's 16 bytes feed its own tensor-core fragment slots and no
//     shuffle is needed; a sum over k does not depend on the order of k.
//   * Tensor cores (mma.sync): weights are the 16-row A operand, tokens the
//     8-column B operand (two B tiles for 9..16 tokens), fp32 accumulation.
//     W8A16 decodes E4M3 to f16 with the hardware conversion (exact), taking
//     both byte pairs of a 32-bit word as 16-bit register halves; for bf16
//     activations the f16 values are widened to bf16 (exact).  W8A8 uses the
//     E4M3 x E4M3 tensor-core form directly (m16n8k32).
//   * Packed weights (FP8L_WEIGHTS_PACKED): the [N, K] codes are permuted
//     once at load time into the order the loads above consume them (the
//     Marlin practice of packing weights to match the tensor-core fragments,
//     "Condition to achieve linear speedup?").  Each CTA's 16 x K slab is
//     then one contiguous block, and each warp load reads 512 contiguous
//     bytes instead of 64 bytes from each of 8 rows.
//   * With FP8L_WEIGHTS_STABLE the kernel is launched as a programmatic
//     dependent of the preceding kernel on the stream: its first weight loads
//     are issued before it waits for that kernel (griddepcontrol.wait), so
//     consecutive products overlap at their boundaries.  Activations, scales
//     and outputs are only touched after the wait.
//   * Epilogue: per-channel (or per-tensor) scale, activation scale, then an
//     f16/bf16 round-to-nearest store or an E4M3 re-quantization through
//     output_scale, one output element per thread with coalesced stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "skinny_device.cuh"

namespace fp8l {
namespace {

enum XKind { kXF16 = 0, kXBF16 = 1, kXE4M3 = 2 };

struct SkinnyArgs {
    const uint8_t *w;  // [N, K] E4M3
    const void *x;     // [M, K] f16 / bf16 / E4M3
    int M, N, K;
    const float *a_scale;    // E4M3 activations only: [1], or [M] per token
    int a_per_token;
    const float *w_scale;    // [1] or [N]
    int w_per_channel;
    const float *out_scale;  // E4M3 output only
    void *y;                 // [M, N]
    int out_dtype;
};

// both byte pairs of a 32-bit word as f16x2: bytes (0,1) -> lo, (2,3) -> hi
__device__ __forceinline__ void dec_f16x2_halves(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
    float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t *>(&b);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Bytes of one token's activations per 64-element chunk: 128 (16-bit) or 64.
template <int XK> struct XBytes { static constexpr int kPerLane = (XK == kXE4M3) ? 16 : 32; };

// Packed layout: 16-channel group G, 64-element chunk c (C = ceil(K / 64)
// chunks per row) form the 1024-byte block at (G * C + c) * 1024; in it, the
// 16 bytes of lane L = 4g + t for row 16G + g sit at 16L and those for row
// 16G + g + 8 at 512 + 16L, covering k = 64c + 16t .. 64c + 16t + 15.  Bytes
// with k >= K are zero.
constexpr int kPackBlock = 1024;

template <int XK, int NT, int WARPS, int UNROLL, bool PACKED>
__global__ void __launch_bounds__(WARPS * 32, 2)
skinny_kernel(const SkinnyArgs args) {
    constexpr int kXWords = XBytes<XK>::kPerLane / 4;  // 32-bit words per lane per token
    __shared__ float red[WARPS][NT][4][32];

    // the next kernel on the stream may be scheduled once every CTA of this
    // one has started; it waits for our results itself
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 2;
    const int t4 = lane & 3;
    const int n0 = blockIdx.x * 16;
    const int m0 = blockIdx.y * 16;
    const int K = args.K;
    const int M = args.M;
    const int nchunks = (K + 63) >> 6;

    // chunk c of rows g and g + 8: packed, the two halves of the 1024-byte
    // block at w_g + c * 1024; row-major, w_g + 64c and w_g8 + 64c
    const uint8_t *w_g =
        PACKED ? args.w + static_cast<size_t>(blockIdx.x) * nchunks * kPackBlock + 16 * lane
               : args.w + static_cast<size_t>(n0 + g) * K + 16 * t4;
    const uint8_t *w_g8 = w_g + static_cast<size_t>(8) * K;  // row-major only
    const char *xbase = static_cast<const char *>(args.x);
    constexpr int kXElt = (XK == kXE4M3) ? 1 : 2;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[nt][r] = 0.0f;

    for (int c0 = warp; c0 < nchunks; c0 += WARPS * UNROLL) {
        uint4 wa[UNROLL], wb[UNROLL];
        uint32_t xw[UNROLL][NT][kXWords];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int c = c0 + u * WARPS;
            const int kk = c * 64 + 16 * t4;  // first k of this lane's 16
            const bool kin = (c < nchunks) && (kk < K);
            if constexpr (PACKED) {
                const uint8_t *wp = w_g + static_cast<size_t>(c) * kPackBlock;
                wa[u] = kin ? ld_stream16(wp) : make_uint4(0, 0, 0, 0);
                wb[u] = kin ? ld_stream16(wp + kPackBlock / 2) : make_uint4(0, 0, 0, 0);
            } else {
                wa[u] = kin ? ld_stream16(w_g + static_cast<size_t>(c) * 64)
                            : make_uint4(0, 0, 0, 0);
                wb[u] = kin ? ld_stream16(w_g8 + static_cast<size_t>(c) * 64)
                            : make_uint4(0, 0, 0, 0);
            }
            // everything but the weights may come from the preceding kernel:
            // wait for it once, after the first weight loads are in flight
            // (a no-op unless launched as a programmatic dependent)
            if (u == 0 && c0 == warp) pdl_wait();
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int m = m0 + g + 8 * nt;
                const bool in = kin && (m < M);
                const uint4 *xp = reinterpret_cast<const uint4 *>(
                    xbase + (static_cast<size_t>(m) * K + kk) * kXElt);
#pragma unroll
                for (int v = 0; v < kXWords / 4; ++v) {
                    uint4 t = in ? ld_act16(xp + v) : make_uint4(0, 0, 0, 0);
                    xw[u][nt][4 * v + 0] = t.x;
                    xw[u][nt][4 * v + 1] = t.y;
                    xw[u][nt][4 * v + 2] = t.z;
                    xw[u][nt][4 * v + 3] = t.w;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint32_t ra[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};  // row g
            const uint32_t rb[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};  // row g + 8
            if constexpr (XK == kXE4M3) {
                // two k32 steps; step j uses bytes 8j..8j+7 of the lane's 16
#pragma unroll
                for (int j = 0; j < 2; ++j) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_e4m3(acc[nt], ra[2 * j], rb[2 * j], ra[2 * j + 1], rb[2 * j + 1],
                                 xw[u][nt][2 * j], xw[u][nt][2 * j + 1]);
                }
            } else {
                // four k16 steps; step j uses bytes 4j..4j+3 of the lane's 16:
                // (4j, 4j+1) fill the low-k slots, (4j+2, 4j+3) the high-k slots
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t a0, a1, a2, a3;
                    dec_f16x2_halves(ra[j], a0, a2);
                    dec_f16x2_halves(rb[j], a1, a3);
                    if constexpr (XK == kXBF16) {
                        a0 = f16x2_to_bf16x2(a0);
                        a1 = f16x2_to_bf16x2(a1);
                        a2 = f16x2_to_bf16x2(a2);
                        a3 = f16x2_to_bf16x2(a3);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if constexpr (XK == kXF16)
                            mma_f16(acc[nt], a0, a1, a2, a3, xw[u][nt][2 * j], xw[u][nt][2 * j + 1]);
                        else
                            mma_bf16(acc[nt], a0, a1, a2, a3, xw[u][nt][2 * j], xw[u][nt][2 * j + 1]);
                    }
                }
            }
        }
    }

    pdl_wait();  // before any store (covers warps that had no chunk)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) red[warp][nt][r][lane] = acc[nt][r];
    __syncthreads();

    // one (token, channel) output per thread: channel fastest for coalescing
    for (int o = threadIdx.x; o < 16 * 8 * NT; o += WARPS * 32) {
        const int ch = o & 15;
        const int tk = o >> 4;  // token within the group, 0 .. 8*NT-1
        const int m = m0 + tk;
        if (m >= M) continue;
        const int nt = tk >> 3;
        const int col = tk & 7;
        const int lane_src = ((ch & 7) << 2) | (col >> 1);
        const int r = ((ch >> 3) << 1) | (col & 1);
        float sum = 0.0f;
#pragma unroll
        for (int wi = 0; wi < WARPS; ++wi) sum += red[wi][nt][r][lane_src];
        const int n = n0 + ch;
        float sc = args.w_per_channel ? __ldg(args.w_scale + n) : __ldg(args.w_scale);
        if constexpr (XK == kXE4M3) sc *= ld_act_f32(args.a_scale + (args.a_per_token ? m : 0));
        const float v = sum * sc;
        const size_t yi = static_cast<size_t>(m) * args.N + n;
        if (args.out_dtype == FP8L_F16) {
            static_cast<__half *>(args.y)[yi] = __float2half_rn(v);
        } else if (args.out_dtype == FP8L_BF16) {
            static_cast<__nv_bfloat16 *>(args.y)[yi] = __float2bfloat16_rn(v);
        } else {
            const float t = __fdiv_rn(v, ld_act_f32(args.out_scale));
            static_cast<uint8_t *>(args.y)[yi] = static_cast<uint8_t>(
                __nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3));
        }
    }
}

constexpr int kWarps = 16;
// chunks a warp loads before it computes: 2, and 4 for one token tile on
// packed weights (a K = 4096 slab in a single round trip; 64 registers
// still hold it, the two-tile form would spill).  Measured on the decode
// step: 4634 GB/s with 2, 4449 with 3, 4802 with 4.
constexpr int kUnroll = 2;
constexpr int kUnrollPacked1 = 4;

template <int XK, int NT, bool PACKED>
int launch_nt(const SkinnyArgs &a, bool stable_weights, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.N / 16), static_cast<unsigned>((a.M + 15) / 16), 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = stable_weights ? 1 : 0;
    constexpr int unroll = (NT == 1 && (PACKED || XK == kXE4M3)) ? kUnrollPacked1 : kUnroll;
    if (cudaLaunchKernelEx(&cfg, skinny_kernel<XK, NT, kWarps, unroll, PACKED>, a) != cudaSuccess)
        return FP8L_ECUDA;
    return launch_status();
}

template <int XK, bool PACKED = false>
int launch(const SkinnyArgs &a, bool stable_weights, cudaStream_t stream) {
    if (a.M == 0) return FP8L_OK;
    const int tokens_in_group = a.M < 16 ? a.M : 16;
    if (tokens_in_group <= 8) return launch_nt<XK, 1, PACKED>(a, stable_weights, stream);
    return launch_nt<XK, 2, PACKED>(a, stable_weights, stream);
}

// One thread per 16 packed bytes: block (G, c), half h, lane L (see the
// packed layout above).
__global__ void pack_weights_kernel(const uint8_t *__restrict__ w, int N, int K, int nchunks,
                                    uint8_t *__restrict__ wp) {
    const size_t words = static_cast<size_t>(N / 16) * nchunks * (kPackBlock / 16);
    for (size_t o = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; o < words;
         o += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int L = static_cast<int>(o & 31);
        const int h = static_cast<int>((o >> 5) & 1);
        const size_t blk = o >> 6;
        const int c = static_cast<int>(blk % nchunks);
        const size_t G = blk / nchunks;
        const size_t row = G * 16 + 8 * h + (L >> 2);
        const int k0 = 64 * c + 16 * (L & 3);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (k0 < K) v = __ldg(reinterpret_cast<const uint4 *>(w + row * K + k0));
        reinterpret_cast<uint4 *>(wp)[o] = v;
    }
}

}  // namespace

int launch_skinny_e4m3(const uint8_t *a, const uint8_t *w, int M, int N, int K,
                       const float *a_scale, int a_per_token, const float *w_scale,
                       int w_per_channel, const float *out_scale, void *y, int out_dtype,
                       bool stable_weights, cudaStream_t stream) {
    SkinnyArgs args{w,       a,           M,         N, K, a_scale, a_per_token,
                    w_scale, w_per_channel, out_scale, y, out_dtype};
    return launch<kXE4M3>(args, stable_weights, stream);
}

}  // namespace fp8l

extern "C" size_t fp8_packed_weight_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || N > (1 << 20) || K > (1 << 20) || N % 16 != 0 || K % 16 != 0)
        return 0;
    return static_cast<size_t>(N) * static_cast<size_t>((K + 63) / 64) * 64;
}

extern "C" int fp8_pack_w8a16_weights(const uint8_t *w, int64_t N, int64_t K, uint8_t *w_packed,
                                      void *stream) {
    using namespace fp8l;
    if (fp8_packed_weight_bytes(N, K) == 0) return FP8L_ESHAPE;
    if (w == nullptr || w_packed == nullptr) return FP8L_EINVAL;
    if (!aligned16(w) || !aligned16(w_packed)) return FP8L_EALIGN;
    int sms = 0;
    int st = check_device(&sms);
    if (st != FP8L_OK) return st;
    const int nchunks = static_cast<int>((K + 63) / 64);
    const size_t words = static_cast<size_t>(N / 16) * nchunks * (kPackBlock / 16);
    const size_t want = (words + 255) / 256;
    const unsigned blocks = static_cast<unsigned>(want < static_cast<size_t>(sms) * 8
                                                      ? want
                                                      : static_cast<size_t>(sms) * 8);
    pack_weights_kernel<<<blocks, 256, 0, as_stream(stream)>>>(w, static_cast<int>(N),
                                                               static_cast<int>(K), nchunks,
                                                               w_packed);
    return launch_status();
}

// The kernel fp8_w8a16_mm runs for FP8L_KERNEL_AUTO: the CUDA-core kernel up
// to 16 tokens (0.45-0.82 of HBM on the decode shapes, against 0.26-0.50
// for the tensor-core product); from 17 to 64 tokens the tensor-core
// product (weights widened in TMEM, tokens as the MMA's N side), which
// streams the weights once whatever the token count (0.24-0.48 of HBM at
// 32-64 tokens against 0.15-0.33 for the CUDA-core kernel, whose token
// groups of 16 each re-read W).
extern "C" unsigned fp8_w8a16_mm_kernel(int64_t M, int64_t N, int64_t K, unsigned flags) {
    (void)N;
    (void)K;
    const unsigned k = flags & FP8L_KERNEL_MASK;
    if (k != FP8L_KERNEL_AUTO) return k;
    return (M >= 17 && M <= 64) ? FP8L_KERNEL_SWAPPED : FP8L_KERNEL_STREAM;
}

extern "C" int fp8_w8a16_mm(const void *x, int x_dtype, const uint8_t *w, const float *w_scale,
                            int64_t M, int64_t N, int64_t K, void *y, unsigned flags,
                            void *stream) {
    using namespace fp8l;
    if (x_dtype != FP8L_F16 && x_dtype != FP8L_BF16) return FP8L_EINVAL;
    if ((flags & ~(FP8L_WEIGHTS_STABLE | FP8L_WEIGHTS_PACKED | FP8L_KERNEL_MASK)) != 0u)
        return FP8L_EINVAL;
    const unsigned kernel = fp8_w8a16_mm_kernel(M, N, K, flags);
    if (kernel == FP8L_KERNEL_TILED) return FP8L_EINVAL;
    if (kernel == FP8L_KERNEL_SWAPPED && M > 64) return FP8L_ESHAPE;
    if (M < 0 || M > 0x7FFFFFFF || N <= 0 || K <= 0 || N > (1 << 20) || K > (1 << 20) ||
        N % 16 != 0 || K % 16 != 0)
        return FP8L_ESHAPE;
    if (w == nullptr || w_scale == nullptr || (M > 0 && (x == nullptr || y == nullptr)))
        return FP8L_EINVAL;
    if (!aligned16(w) || (M > 0 && (!aligned16(x) || !aligned16(y))) ||
        (reinterpret_cast<uintptr_t>(w_scale) & 3u) != 0)
        return FP8L_EALIGN;
    int sms = 0;
    int st = check_device(&sms);
    if (st != FP8L_OK) return st;
    if (M == 0) return FP8L_OK;
    if (kernel == FP8L_KERNEL_SWAPPED) {
        unsigned *status = nullptr;
        if (library_status_word(&status) != FP8L_OK) return FP8L_ECUDA;
        return launch_w8a16_tc(x, x_dtype, w, (flags & FP8L_WEIGHTS_PACKED) != 0u, w_scale,
                               static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), y, status,
                               sms, (flags & FP8L_WEIGHTS_STABLE) != 0u, as_stream(stream));
    }
    SkinnyArgs args{w, x, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                    nullptr, 0, w_scale, 1, nullptr, y, x_dtype};
    const bool stable = (flags & FP8L_WEIGHTS_STABLE) != 0u;
    const cudaStream_t s = as_stream(stream);
    if ((flags & FP8L_WEIGHTS_PACKED) != 0u)
        return x_dtype == FP8L_F16 ? launch<kXF16, true>(args, stable, s)
                                   : launch<kXBF16, true>(args, stable, s);
    return x_dtype == FP8L_F16 ? launch<kXF16>(args, stable, s) : launch<kXBF16>(args, stable, s);
}

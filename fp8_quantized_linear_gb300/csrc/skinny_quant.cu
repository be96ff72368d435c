// W8A8 product of up to 16 tokens of 16-bit activations with their
// per-tensor E4M3 quantization inside the weight-streaming kernel
// ("Condition to achieve linear speedup?": activation quantization fused
// into another kernel rather than its own launch; "RFC: FP8 Quantization
// Schema in vLLM": static input scales; "[Kernel][FP8] Initial support with
// dynamic per-tensor scaling": the dynamic scale amax / 448).  The small-
// weight branch of fp8_quant_scaled_mm: the layout and MMAs of the CUDA-core
// W8A8 kernel in skinny.cu (16 output channels per CTA, 16 warps splitting
// K in 64-element chunks, E4M3 x E4M3 m16n8k32 on the tensor cores, the
// same partial-tile sum and epilogue), with the activations' codes made
// here from x with the quantizer's arithmetic, so the result is that of
// fp8_quant_per_tensor followed by that kernel, bit for bit.
//   * Scale: static, read; dynamic, every CTA takes amax(|x|) over all of x
//     (at most FP8L_FUSED_DYNAMIC_MAX_BYTES) and derives the same scale, the
//     CTA at x = 0 storing it.
//   * Codes: for one or two tokens every CTA writes the codes of all of x
//     into shared memory before its main loop, which then reads codes as the
//     plain kernel reads them from HBM (four chunks in flight); for more
//     tokens each warp makes the codes of its own chunks in the main loop,
//     under its weight loads (staging all of x per CTA cost more there).
//   * With FP8L_WEIGHTS_STABLE a programmatic dependent: the first chunks'
//     weight lines are asked of L2 before the kernel waits for the preceding
//     one; x, the scales and y are touched only after the wait.
// A separate kernel from skinny.cu's so that the W8A16 and plain W8A8
// instances there compile as they did: adding these paths to that template
// changed the compiler's register allocation of the W8A16 instances and
// slowed the decode layer by 7-11 %.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"
#include "quant_device.cuh"
#include "skinny_device.cuh"

namespace fp8l {
namespace {

struct QuantSkinnyArgs {
    const uint8_t *w;  // [N, K] E4M3, row-major
    const void *x;     // [M, K] f16 / bf16, M <= 16
    int M, N, K;
    float *a_scale;    // [1]: read (static) or written (dynamic)
    int dynamic;
    const float *w_scale;  // [1] or [N]
    int w_per_channel;
    const float *out_scale;  // E4M3 output only
    void *y;                 // [M, N]
    int out_dtype;
};

constexpr int kQWarps = 16;
// staged codes: row m of x at m * (K + kStagePad) (16 bytes of padding: the
// 8 rows a warp reads at one k fall in different banks)
constexpr int kStagePad = 16;
constexpr int kStageMaxBytes = 96 * 1024;

// amax(|x|) / 448 over all of x (eight 16-byte loads in flight per thread),
// or the given scale; every thread of the block calls it
template <int DT>
__device__ float act_scale(const QuantSkinnyArgs &a, uint32_t *red) {
    if (!a.dynamic) return ld_act_f32(a.a_scale);
    const uint4 *xv = static_cast<const uint4 *>(a.x);
    const int words = a.M * a.K / 8;  // 8 16-bit values per word
    uint32_t m = 0;
    for (int w0 = threadIdx.x; w0 < words; w0 += 8 * kQWarps * 32) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int w = w0 + u * kQWarps * 32;
            v[u] = w < words ? ld_act16(xv + w) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) m = word_mag_max<DT>(v[u], m);
    }
    m = block_max_u32(fold_mag<DT>(m), red);
    const float sa = scale_from_amax(mag_bits_to_float<DT>(m));
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.a_scale = sa;
    return sa;
}

template <int DT, int NT, int UNROLL, bool STAGED>
__global__ void __launch_bounds__(kQWarps * 32, 2) skinny_quant_kernel(const QuantSkinnyArgs a) {
    // 16-bit words (8 per lane per token and chunk), or staged codes (4)
    constexpr int kXWords = STAGED ? 4 : 8;
    __shared__ float red[kQWarps][NT][4][32];
    __shared__ uint32_t mred[33];
    __shared__ float sa_sh;
    extern __shared__ uint4 xcodes[];  // staged codes (dynamic shared memory)

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 2;
    const int t4 = lane & 3;
    const int n0 = blockIdx.x * 16;
    const int K = a.K;
    const int M = a.M;
    const int nchunks = (K + 63) >> 6;
    const uint8_t *w_g = a.w + static_cast<size_t>(n0 + g) * K + 16 * t4;
    const uint8_t *w_g8 = w_g + static_cast<size_t>(8) * K;

    // the first chunks' weight lines on their way while the kernel waits
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int c = warp + u * kQWarps;
        if (c < nchunks && c * 64 + 16 * t4 < K) {
            asm volatile("prefetch.global.L2 [%0];" ::"l"(w_g + static_cast<size_t>(c) * 64));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(w_g8 + static_cast<size_t>(c) * 64));
        }
    }
    pdl_wait();
    const float sa = act_scale<DT>(a, mred);
    if (threadIdx.x == 0) sa_sh = sa;  // read after the barrier before the epilogue
    const Quot d = Quot::make<DT>(sa);
    const uint32_t xs = static_cast<uint32_t>(__cvta_generic_to_shared(xcodes));
    if constexpr (STAGED) {
        // word w (8 values) of row m to m * (K + kStagePad) + 8 (w mod K/8)
        const uint4 *xv = static_cast<const uint4 *>(a.x);
        const int row_words = K / 8, words = M * row_words;
        for (int w = threadIdx.x; w < words; w += kQWarps * 32) {
            const uint4 v = ld_act16(xv + w);
            const uint2 cq = a.dynamic ? codes_of_word<DT, false>(v, d) : codes_of_word<DT, true>(v, d);
            const int m = w / row_words;
            const uint32_t off = static_cast<uint32_t>(m * (K + kStagePad) + 8 * (w - m * row_words));
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(xs + off), "r"(cq.x), "r"(cq.y)
                         : "memory");
        }
        __syncthreads();
    }

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[nt][r] = 0.0f;

    for (int c0 = warp; c0 < nchunks; c0 += kQWarps * UNROLL) {
        uint4 wa[UNROLL], wb[UNROLL];
        uint32_t xw[UNROLL][NT][kXWords];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int c = c0 + u * kQWarps;
            const int kk = c * 64 + 16 * t4;  // first k of this lane's 16
            const bool kin = (c < nchunks) && (kk < K);
            wa[u] = kin ? ld_stream16(w_g + static_cast<size_t>(c) * 64) : make_uint4(0, 0, 0, 0);
            wb[u] = kin ? ld_stream16(w_g8 + static_cast<size_t>(c) * 64) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int m = g + 8 * nt;
                const bool in = kin && (m < M);
                uint4 t[kXWords / 4];
#pragma unroll
                for (int v = 0; v < kXWords / 4; ++v) t[v] = make_uint4(0, 0, 0, 0);
                if (in) {
                    if constexpr (STAGED) {
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(t[0].x), "=r"(t[0].y), "=r"(t[0].z), "=r"(t[0].w)
                                     : "r"(xs + static_cast<uint32_t>(m * (K + kStagePad) + kk)));
                    } else {
                        const uint4 *xp = static_cast<const uint4 *>(a.x) +
                                          (static_cast<size_t>(m) * K + kk) / 8;
                        t[0] = ld_act16(xp);
                        t[1] = ld_act16(xp + 1);
                    }
                }
#pragma unroll
                for (int v = 0; v < kXWords / 4; ++v) {
                    xw[u][nt][4 * v + 0] = t[v].x;
                    xw[u][nt][4 * v + 1] = t[v].y;
                    xw[u][nt][4 * v + 2] = t[v].z;
                    xw[u][nt][4 * v + 3] = t[v].w;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint32_t ra[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};  // row g
            const uint32_t rb[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};  // row g + 8
            // two k32 steps; step j takes the codes of values 8j..8j+7 of
            // the lane's 16 (the k order inside a chunk is the same permuted
            // order on both operands, as in the plain kernel)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    uint32_t b0, b1;
                    if constexpr (STAGED) {
                        b0 = xw[u][nt][2 * j];
                        b1 = xw[u][nt][2 * j + 1];
                    } else {
                        const uint4 xv = make_uint4(xw[u][nt][4 * j], xw[u][nt][4 * j + 1],
                                                    xw[u][nt][4 * j + 2], xw[u][nt][4 * j + 3]);
                        const uint2 cq = a.dynamic ? codes_of_word<DT, false>(xv, d)
                                                   : codes_of_word<DT, true>(xv, d);
                        b0 = cq.x;
                        b1 = cq.y;
                    }
                    mma_e4m3(acc[nt], ra[2 * j], rb[2 * j], ra[2 * j + 1], rb[2 * j + 1], b0, b1);
                }
            }
        }
    }

#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) red[warp][nt][r][lane] = acc[nt][r];
    __syncthreads();

    // one (token, channel) output per thread, channel fastest; the warps'
    // partial tiles added in warp order, as in the plain kernel
    const float sa_e = sa_sh;
    for (int o = threadIdx.x; o < 16 * 8 * NT; o += kQWarps * 32) {
        const int ch = o & 15;
        const int tk = o >> 4;
        if (tk >= M) continue;
        const int nt = tk >> 3;
        const int col = tk & 7;
        const int lane_src = ((ch & 7) << 2) | (col >> 1);
        const int r = ((ch >> 3) << 1) | (col & 1);
        float sum = 0.0f;
#pragma unroll
        for (int wi = 0; wi < kQWarps; ++wi) sum += red[wi][nt][r][lane_src];
        const int n = n0 + ch;
        float sc = a.w_per_channel ? __ldg(a.w_scale + n) : __ldg(a.w_scale);
        sc *= sa_e;
        const float v = sum * sc;
        const size_t yi = static_cast<size_t>(tk) * a.N + n;
        if (a.out_dtype == FP8L_F16) {
            static_cast<__half *>(a.y)[yi] = __float2half_rn(v);
        } else if (a.out_dtype == FP8L_BF16) {
            static_cast<__nv_bfloat16 *>(a.y)[yi] = __float2bfloat16_rn(v);
        } else {
            const float t = __fdiv_rn(v, ld_act_f32(a.out_scale));
            static_cast<uint8_t *>(a.y)[yi] =
                static_cast<uint8_t>(__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3));
        }
    }
}

template <int DT, int NT, int UNROLL, bool STAGED>
int launch_q(const QuantSkinnyArgs &a, bool stable_weights, cudaStream_t stream) {
    auto kernel = skinny_quant_kernel<DT, NT, UNROLL, STAGED>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.N / 16), 1, 1);
    cfg.blockDim = dim3(kQWarps * 32, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = stable_weights ? 1 : 0;
    if constexpr (STAGED) {
        // at most kStageMaxBytes (two CTAs per SM still fit); the opt-in size
        // set once per device
        static std::atomic<int> attr_set[64];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8L_ECUDA;
        if (!attr_set[dev].load(std::memory_order_acquire)) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kStageMaxBytes) != cudaSuccess)
                return FP8L_ECUDA;
            attr_set[dev].store(1, std::memory_order_release);
        }
        cfg.dynamicSmemBytes = static_cast<size_t>(a.M) * (a.K + kStagePad);
    }
    if (cudaLaunchKernelEx(&cfg, kernel, a) != cudaSuccess) return FP8L_ECUDA;
    return launch_status();
}

template <int DT>
int launch_dt(const QuantSkinnyArgs &a, bool stable_weights, cudaStream_t stream) {
    // staged codes for one or two tokens (M = 1, 4096 x 4096, static scale:
    // 6.2 us against 7.0 making them in the main loop; M = 8: 10.6 against
    // 7.3, every CTA staging all of x before its main loop); chunks in
    // flight per warp: four reading codes, two making them for one token
    // tile, one for two (two spilled 160 bytes of the 64 registers)
    if (a.M <= 2 && int64_t(a.M) * (a.K + kStagePad) <= kStageMaxBytes)
        return launch_q<DT, 1, 4, true>(a, stable_weights, stream);
    if (a.M <= 8) return launch_q<DT, 1, 2, false>(a, stable_weights, stream);
    return launch_q<DT, 2, 1, false>(a, stable_weights, stream);
}

}  // namespace

int launch_skinny_quant(const void *x, int x_dtype, const uint8_t *w, int M, int N, int K,
                        float *a_scale, int dynamic, const float *w_scale, int w_per_channel,
                        const float *out_scale, void *y, int out_dtype, bool stable_weights,
                        cudaStream_t stream) {
    if (M < 1 || M > 16) return FP8L_ESHAPE;  // one token group
    const QuantSkinnyArgs a{w,       x,         M,         N, K, a_scale, dynamic,
                            w_scale, w_per_channel, out_scale, y, out_dtype};
    return x_dtype == FP8L_F16 ? launch_dt<FP8L_F16>(a, stable_weights, stream)
                               : launch_dt<FP8L_BF16>(a, stable_weights, stream);
}

}  // namespace fp8l

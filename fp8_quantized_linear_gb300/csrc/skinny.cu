// Weight-streaming products for small token counts (up to 16 tokens per CTA):
//   * W8A16 ("Marlin fp8"): fp16/bf16 activations x E4M3 weights with one
//     scale per output channel;
//   * W8A8 small-M branch of the scaled product ("[Kernel][FP8] Initial
//     support ...", the M = 1..16 rows of the microbenchmark list, where the
//     product is bound by reading the weights).
//
// Design (HBM-bound: the weights are read once, the activations are small)
//   * A CTA owns 64 output channels (rows of W) and up to 16 tokens.  It walks
//     its K range in stages of 512 elements; a stage holds the 64 x 512 weight
//     bytes and the 16 x 512 activations, copied with 16-byte cp.async into a
//     4-deep shared-memory ring, so about 150-200 KB of loads are in flight
//     per SM at all times.  A warp of the copy reads one full 512-byte row
//     segment (coalesced).
//   * Warp w computes the 64 x 16 tile over k = [64w, 64w + 64) of every
//     stage on the tensor cores (mma.sync; weights are the 16-row A operand,
//     tokens the 8-column B operand, fp32 accumulation).  Lane (g, t) reads
//     16 contiguous weight bytes of rows g and g+8 of each 16-row tile; the k
//     order inside those 64 elements is permuted identically for weights and
//     activations, so no shuffle is needed (a sum over k does not depend on
//     the order of k).  Rows are padded in shared memory so that every
//     fragment read and every copy is free of bank conflicts.
//   * W8A16 decodes E4M3 to f16 with the hardware conversion (exact); for
//     bf16 activations the f16 values are widened to bf16 (exact).  W8A8 uses
//     the E4M3 x E4M3 tensor-core form (m16n8k32) with no decode.
//   * The 8 warps' partial tiles are added in shared memory.  When the grid
//     would have too few CTAs to keep HBM busy, CL CTAs of a thread-block
//     cluster split K and add their tiles through distributed shared memory.
//   * Epilogue: per-channel (or per-tensor) weight scale times the activation
//     scale, then an f16/bf16 round-to-nearest store or an E4M3
//     re-quantization through output_scale; consecutive threads store
//     consecutive channels.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"

namespace fp8l {
namespace {

enum XKind { kXF16 = 0, kXBF16 = 1, kXE4M3 = 2 };

struct SkinnyArgs {
    const uint8_t *w;  // [N, K] E4M3
    const void *x;     // [M, K] f16 / bf16 / E4M3
    int M, N, K;
    const float *a_scale;    // E4M3 activations only
    const float *w_scale;    // [1] or [N]
    int w_per_channel;
    const float *out_scale;  // E4M3 output only
    void *y;                 // [M, N]
    int out_dtype;
    int k_per_cta;           // K range of one CTA of a cluster (multiple of 16)
};

constexpr int kRows = 64;      // channels per CTA
constexpr int kBK = 512;       // k elements per stage
constexpr int kStages = 4;
constexpr int kWarps = 8;      // one 64-element k slice of a stage each
constexpr int kThreads = kWarps * 32;
constexpr int kWPitch = kBK + 64;  // bytes per weight row in shared memory

template <int XK> struct XLayout {
    static constexpr int kElt = (XK == kXE4M3) ? 1 : 2;
    static constexpr int kPitch = (XK == kXE4M3) ? kBK + 64 : 2 * kBK + 16;  // bytes per token
};

template <int XK, int NT> struct Smem {
    static constexpr int kWBytes = kRows * kWPitch;
    static constexpr int kXBytes = 8 * NT * XLayout<XK>::kPitch;
    static constexpr int kStageBytes = kWBytes + kXBytes;
    static constexpr int kPartOffset = kStages * kStageBytes;
    static constexpr int kPartBytes = kRows * 8 * NT * 4;  // CTA partial tile, floats
    static constexpr int kTotal = kPartOffset + kPartBytes;
    static_assert(kWarps * 4 * NT * 4 * 32 * 4 <= kStages * kStageBytes, "reduction fits");
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t dec_f16x2(uint32_t pair) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair & 0xFFFFu),
                                               __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

__device__ __forceinline__ uint32_t dec_bf16x2(uint32_t pair) {
    uint32_t h = dec_f16x2(pair);
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

__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

template <int XK, int NT>
__global__ void __launch_bounds__(kThreads, 1)
skinny_kernel(const SkinnyArgs args) {
    using S = Smem<XK, NT>;
    using XL = XLayout<XK>;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int g = lane >> 2;
    const int t4 = lane & 3;
    const int K = args.K;
    const int N = args.N;

    const uint32_t crank = cluster_rank();
    const uint32_t csize = cluster_size();
    const int n0 = static_cast<int>(blockIdx.x / csize) * kRows;
    const int m0 = blockIdx.y * 16;
    const int m_here = min(args.M - m0, 8 * NT);       // tokens of this CTA
    const int tiles = min(4, (N - n0) >> 4);           // valid 16-row tiles
    const int kb = static_cast<int>(crank) * args.k_per_cta;
    const int ke = min(K, kb + args.k_per_cta);
    const int nst = ke > kb ? (ke - kb + kBK - 1) / kBK : 0;

    const uint8_t *wg = args.w + static_cast<size_t>(n0) * K;
    const char *xg = static_cast<const char *>(args.x) + static_cast<size_t>(m0) * K * XL::kElt;

    // copy one stage: weights 64 x 512 B (32 pieces of 16 B per row) and
    // activations (8*NT tokens x 512 elements); pieces beyond K are zero-filled
    auto load_stage = [&](int slot, int k0) {
        const uint32_t sw = sbase + slot * S::kStageBytes;
        const uint32_t sx = sw + S::kWBytes;
#pragma unroll
        for (int j = 0; j < kRows * 32 / kThreads; ++j) {
            const int p = tid + j * kThreads;
            const int r = p >> 5;
            const int kk = k0 + ((p & 31) << 4);
            if (r < tiles * 16) {
                const bool in = kk < ke;
                cp_async16(sw + r * kWPitch + ((p & 31) << 4),
                           in ? static_cast<const void *>(wg + static_cast<size_t>(r) * K + kk) : args.w,
                           in ? 16u : 0u);
            }
        }
        constexpr int kPiecesPerToken = kBK * XL::kElt / 16;
        constexpr int kXPieces = 8 * NT * kPiecesPerToken;
#pragma unroll
        for (int j = 0; j < (kXPieces + kThreads - 1) / kThreads; ++j) {
            const int p = tid + j * kThreads;
            if (p < kXPieces) {
                const int t = p / kPiecesPerToken;
                const int q = p % kPiecesPerToken;
                const int kk = k0 + q * (16 / XL::kElt);
                if (t < m_here) {
                    const bool in = kk < ke;
                    cp_async16(sx + t * XL::kPitch + q * 16,
                               in ? static_cast<const void *>(xg + (static_cast<size_t>(t) * K + kk) * XL::kElt)
                                  : args.x,
                               in ? 16u : 0u);
                }
            }
        }
    };

    float acc[4][NT][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[i][nt][r] = 0.0f;

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nst) load_stage(s, kb + s * kBK);
        cp_async_commit();
    }

    for (int it = 0; it < nst; ++it) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        const int slot = it % kStages;
        const uint32_t sw = sbase + slot * S::kStageBytes;
        const uint32_t sx = sw + S::kWBytes;
        // activation fragments of this warp's 64 k, for every token tile
        constexpr int kXW = (XK == kXE4M3) ? 4 : 8;
        uint32_t xw[NT][kXW];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int t = 8 * nt + g;
            if (t < m_here) {
                if constexpr (XK == kXE4M3) {
                    const uint4 v = lds128(sx + t * XL::kPitch + 64 * warp + 16 * t4);
                    xw[nt][0] = v.x; xw[nt][1] = v.y; xw[nt][2] = v.z; xw[nt][3] = v.w;
                } else {
                    const uint32_t a = sx + t * XL::kPitch + 128 * warp + 32 * t4;
                    const uint4 v0 = lds128(a);
                    const uint4 v1 = lds128(a + 16);
                    xw[nt][0] = v0.x; xw[nt][1] = v0.y; xw[nt][2] = v0.z; xw[nt][3] = v0.w;
                    xw[nt][4] = v1.x; xw[nt][5] = v1.y; xw[nt][6] = v1.z; xw[nt][7] = v1.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < kXW; ++q) xw[nt][q] = 0u;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i < tiles) {
                const uint32_t wa = sw + (16 * i + g) * kWPitch + 64 * warp + 16 * t4;
                const uint4 va = lds128(wa);                 // row g of tile i
                const uint4 vb = lds128(wa + 8 * kWPitch);   // row g + 8
                const uint32_t ra[4] = {va.x, va.y, va.z, va.w};
                const uint32_t rb[4] = {vb.x, vb.y, vb.z, vb.w};
                if constexpr (XK == kXE4M3) {
                    // two k32 steps; step j uses bytes 8j..8j+7 of the lane's 16
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_e4m3(acc[i][nt], ra[2 * j], rb[2 * j], ra[2 * j + 1], rb[2 * j + 1],
                                     xw[nt][2 * j], xw[nt][2 * j + 1]);
                } else {
                    // four k16 steps; step j uses bytes 4j..4j+3: (4j, 4j+1) fill the
                    // low-k fragment slots, (4j+2, 4j+3) the high-k slots
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t a0, a1, a2, a3;
                        if constexpr (XK == kXF16) {
                            a0 = dec_f16x2(ra[j]);
                            a1 = dec_f16x2(rb[j]);
                            a2 = dec_f16x2(ra[j] >> 16);
                            a3 = dec_f16x2(rb[j] >> 16);
                        } else {
                            a0 = dec_bf16x2(ra[j]);
                            a1 = dec_bf16x2(rb[j]);
                            a2 = dec_bf16x2(ra[j] >> 16);
                            a3 = dec_bf16x2(rb[j] >> 16);
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            if constexpr (XK == kXF16)
                                mma_f16(acc[i][nt], a0, a1, a2, a3, xw[nt][2 * j], xw[nt][2 * j + 1]);
                            else
                                mma_bf16(acc[i][nt], a0, a1, a2, a3, xw[nt][2 * j], xw[nt][2 * j + 1]);
                        }
                    }
                }
            }
        }
        // the slot read in the previous iteration is free: every warp passed
        // the barrier above after finishing it
        const int nxt = it + kStages - 1;
        if (nxt < nst) load_stage(nxt % kStages, kb + nxt * kBK);
        cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();

    // add the 8 warps' tiles: red[warp][i][nt][r][lane] reuses the ring
    float *red = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r)
                red[(((warp * 4 + i) * NT + nt) * 4 + r) * 32 + lane] = acc[i][nt][r];
    __syncthreads();
    // CTA partial tile, token-major: part[t * 64 + row]
    float *part = reinterpret_cast<float *>(smem + S::kPartOffset);
    constexpr int kOut = kRows * 8 * NT;
    for (int o = tid; o < kOut; o += kThreads) {
        const int t = o >> 6;
        const int row = o & 63;
        const int i = row >> 4;
        const int rr = (((row >> 3) & 1) << 1) | (t & 1);
        const int src = ((row & 7) << 2) | ((t & 7) >> 1);
        const int nt = t >> 3;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[(((w * 4 + i) * NT + nt) * 4 + rr) * 32 + src];
        part[o] = s;
    }
    if (csize > 1) cluster_sync();
    else __syncthreads();

    // CTA `crank` of the cluster finishes outputs [crank*kOut/csize, ...)
    const int per = kOut / static_cast<int>(csize);
    const uint32_t part_addr = sbase + S::kPartOffset;
    for (int o = static_cast<int>(crank) * per + tid; o < static_cast<int>(crank + 1) * per;
         o += kThreads) {
        const int t = o >> 6;
        const int row = o & 63;
        const int m = m0 + t;
        const int n = n0 + row;
        float s;
        if (csize > 1) {
            s = 0.0f;
            for (uint32_t q = 0; q < csize; ++q) s += ld_cluster_f32(part_addr + 4u * o, q);
        } else {
            s = part[o];
        }
        if (t >= m_here || row >= tiles * 16) continue;
        float sc = args.w_per_channel ? __ldg(args.w_scale + n) : __ldg(args.w_scale);
        if constexpr (XK == kXE4M3) sc *= __ldg(args.a_scale);
        const float v = s * sc;
        const size_t yi = static_cast<size_t>(m) * N + n;
        if (args.out_dtype == FP8L_F16) {
            static_cast<__half *>(args.y)[yi] = __float2half_rn(v);
        } else if (args.out_dtype == FP8L_BF16) {
            static_cast<__nv_bfloat16 *>(args.y)[yi] = __float2bfloat16_rn(v);
        } else {
            const float q = __fdiv_rn(v, __ldg(args.out_scale));
            static_cast<uint8_t *>(args.y)[yi] =
                static_cast<uint8_t>(__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3));
        }
    }
    // peers may still be reading this CTA's partial tile
    if (csize > 1) cluster_sync();
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_attr_done[kMaxDevices][3][2];

template <int XK, int NT>
int prepare_attr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8L_ECUDA;
    std::atomic<int> &flag = g_attr_done[dev][XK][NT - 1];
    if (flag.load(std::memory_order_acquire)) return FP8L_OK;
    if (cudaFuncSetAttribute(skinny_kernel<XK, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<XK, NT>::kTotal) != cudaSuccess)
        return FP8L_ECUDA;
    flag.store(1, std::memory_order_release);
    return FP8L_OK;
}

// K split over a cluster so that the grid has enough CTAs to keep HBM busy:
// the smallest power of two (at most 8) giving >= 120 CTAs per token group,
// keeping at least one 512-element stage per CTA.
int choose_cluster(int N, int K) {
    const int groups = (N + kRows - 1) / kRows;
    int cl = 1;
    while (cl < 8 && groups * cl < 120 && K / (2 * cl) >= kBK) cl *= 2;
    return cl;
}

template <int XK, int NT>
int launch_t(SkinnyArgs a, cudaStream_t stream) {
    if (prepare_attr<XK, NT>() != FP8L_OK) return FP8L_ECUDA;
    const int cl = choose_cluster(a.N, a.K);
    const int per = (a.K + cl - 1) / cl;
    a.k_per_cta = (per + 15) / 16 * 16;
    const int groups = (a.N + kRows - 1) / kRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(groups * cl), static_cast<unsigned>((a.M + 15) / 16), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Smem<XK, NT>::kTotal;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, skinny_kernel<XK, NT>, a) != cudaSuccess) return FP8L_ECUDA;
    return launch_status();
}

template <int XK>
int launch(const SkinnyArgs &a, cudaStream_t stream) {
    if (a.M == 0) return FP8L_OK;
    const int tokens_in_group = a.M < 16 ? a.M : 16;
    if (tokens_in_group <= 8) return launch_t<XK, 1>(a, stream);
    return launch_t<XK, 2>(a, stream);
}

}  // namespace

int launch_skinny_e4m3(const uint8_t *a, const uint8_t *w, int M, int N, int K,
                       const float *a_scale, const float *w_scale, int w_per_channel,
                       const float *out_scale, void *y, int out_dtype, cudaStream_t stream) {
    SkinnyArgs args{w, a, M, N, K, a_scale, w_scale, w_per_channel, out_scale, y, out_dtype, 0};
    return launch<kXE4M3>(args, stream);
}

}  // namespace fp8l

extern "C" int fp8_w8a16_mm(const void *x, int x_dtype, const uint8_t *w, const float *w_scale,
                            int64_t M, int64_t N, int64_t K, void *y, void *stream) {
    using namespace fp8l;
    if (x_dtype != FP8L_F16 && x_dtype != FP8L_BF16) return FP8L_EINVAL;
    if (M < 0 || M > 0x7FFFFFFF || N <= 0 || K <= 0 || N > (1 << 20) || K > (1 << 20) ||
        N % 16 != 0 || K % 16 != 0)
        return FP8L_ESHAPE;
    if (w == nullptr || w_scale == nullptr || (M > 0 && (x == nullptr || y == nullptr)))
        return FP8L_EINVAL;
    if (!aligned16(w) || (M > 0 && (!aligned16(x) || !aligned16(y))) ||
        (reinterpret_cast<uintptr_t>(w_scale) & 3u) != 0)
        return FP8L_EALIGN;
    int st = check_device(nullptr);
    if (st != FP8L_OK) return st;
    SkinnyArgs args{w, x, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                    nullptr, w_scale, 1, nullptr, y, x_dtype, 0};
    if (x_dtype == FP8L_F16) return launch<kXF16>(args, as_stream(stream));
    return launch<kXBF16>(args, as_stream(stream));
}

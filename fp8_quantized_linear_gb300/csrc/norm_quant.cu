// RMS normalization with the activation quantization fused into it.
//
// "Condition to achieve linear speedup?" (the QQQ issue): the activation
// quantization of a W8A8 layer is fused into the element-wise kernel before
// it, such as RMSNorm, instead of running as a separate pass.  The layer
// computes, per row m of X [M, K] (the plain Llama RMSNorm; the pages do not
// define it):
//   r[m]    = 1 / sqrt( (1/K) sum_k x[m,k]^2 + eps )
//   h[m,k]  = RN16( (x[m,k] * r[m]) * gamma[k] )   (x's 16-bit format)
// and then quantizes h exactly as fp8_quant_per_tensor / fp8_quant_per_row
// quantize a 16-bit tensor ("[Kernel][FP8] Initial support with dynamic
// per-tensor scaling", Algorithm): dynamic per-tensor (s = amax|h| / 448,
// a grid-wide maximum), static per-tensor (s given), or per token
// (s[m] = amax_k |h[m,k]| / 448).  h itself is written only when asked for;
// the norm-only mode writes h and no codes (the unfused layer's first step).
//
// Design: one CTA of 512 threads per SM, persistent over rows b, b + G, ...
// Rows stream into a ring of shared-memory stages by bulk copies (TMA) with
// one mbarrier per stage, so many rows per SM are in flight.  A thread owns
// the same 16-byte words of every row (word w = t + 512 j), so its gamma
// words stay in registers for the whole kernel.  Per row: the thread's x
// words move to registers, a block sum of squares gives r (IEEE division and
// square root), h is formed in registers, and the codes are the quantizer's
// (correctly rounded quotient, saturating E4M3 conversion).  Per-token and
// static modes read X once.  Dynamic per-tensor mode needs amax|h| over the
// whole tensor first: pass 1 forms h for the maximum, the blocks meet at a
// grid barrier (cooperative launch, the workspace's barrier words), and
// pass 2 recomputes h (the same operations in the same order, so the same
// values) from the rows still in shared memory, then from the others,
// re-read.
#include <atomic>

#include "quant_device.cuh"

namespace fp8l {
namespace {

// 256 threads per block for K <= 8192 (up to four blocks per SM, so one
// block's per-row barriers overlap the others' work), 512 above; a thread
// holds at most 8 words (64 elements) of a row
constexpr int kNormMaxK = 32768;
constexpr int kNormSmemBudget = 200 * 1024;      // bytes of row stages per SM
constexpr int kNormMaxStages = 32;

enum NqMode { kNqDynamic = 0, kNqStatic = 1, kNqPerToken = 2, kNqNormOnly = 3 };

template <int DT>
__device__ __forceinline__ float2 to_float2(uint32_t w) {
    if constexpr (DT == FP8L_BF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    } else {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    }
}

template <int DT>
__device__ __forceinline__ uint32_t to_16x2(float a, float b) {
    if constexpr (DT == FP8L_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

template <int DT>
__device__ __forceinline__ uint64_t to_pair(uint32_t w) {
    const float2 f = to_float2<DT>(w);
    return f2_pack(__float_as_uint(f.x), __float_as_uint(f.y));
}

// h word (8 elements) of x word xv and gamma word gv: RN16((x * r) * gamma),
// two products on float pairs
template <int DT>
__device__ __forceinline__ uint4 norm_word(const uint4 &xv, const uint4 &gv, uint64_t r2) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t hw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint64_t h = f2_mul(f2_mul(to_pair<DT>(xw[i]), r2), to_pair<DT>(gw[i]));
        hw[i] = to_16x2<DT>(__uint_as_float(static_cast<uint32_t>(h)),
                            __uint_as_float(static_cast<uint32_t>(h >> 32)));
    }
    return make_uint4(hw[0], hw[1], hw[2], hw[3]);
}

// squares of the 8 elements of a word added to a pair of partial sums (x^2 is
// exact in float32 for 16-bit x)
template <int DT>
__device__ __forceinline__ uint64_t word_sumsq(const uint4 &xv, uint64_t acc) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint64_t f = to_pair<DT>(xw[i]);
        acc = f2_fma(f, f, acc);
    }
    return acc;
}

// Sum over the block with one barrier: warp sums go to buffer `flip` of red,
// then every thread adds the 16 warp sums in the same order.  Alternating
// the buffer between calls keeps a call's writes clear of the previous
// call's reads (every thread has passed this call's barrier by then).
template <int THREADS>
__device__ __forceinline__ float block_sum(float v, float (*red)[THREADS / 32], int &flip) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[flip][warp] = v;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int i = 0; i < THREADS / 32; ++i) t += red[flip][i];
    flip ^= 1;
    return t;
}

// the same for a maximum of magnitude bits
template <int THREADS>
__device__ __forceinline__ uint32_t block_max(uint32_t v, uint32_t (*red)[THREADS / 32], int &flip) {
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[flip][warp] = v;
    __syncthreads();
    uint32_t t = 0;
#pragma unroll
    for (int i = 0; i < THREADS / 32; ++i) t = max(t, red[flip][i]);
    flip ^= 1;
    return t;
}

struct NormArgs {
    const void *x;
    const void *gamma;
    float eps;
    int M, K;
    uint8_t *q;
    float *scale;  // [1] (tensor modes) or [M] (per token)
    void *h;       // optional
    int mode;
    unsigned *epoch, *arrive, *amax, *status;  // dynamic mode: workspace words
    int stages;
    long long wait_cycles;
    unsigned stall;
};

template <int DT, int THREADS, int NW>
__global__ void __launch_bounds__(THREADS) rmsnorm_quant_kernel(const NormArgs a) {
    constexpr int kNThreads = THREADS;
    extern __shared__ __align__(128) uint4 rows_smem[];
    __shared__ __align__(8) uint64_t full[kNormMaxStages];
    __shared__ float fred[2][THREADS / 32];
    __shared__ uint32_t ured[2][THREADS / 32];
    __shared__ uint32_t bred[33];
    __shared__ int abort_sh;
    __shared__ unsigned epoch_sh;

    // a product launched as a programmatic dependent may be scheduled now;
    // it waits for this grid's writes itself
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int G = static_cast<int>(gridDim.x);
    const int b = static_cast<int>(blockIdx.x);
    const int words = a.K / 8;  // 16-byte words per row
    const uint32_t row_bytes = static_cast<uint32_t>(a.K) * 2u;
    const int S = a.stages;
    const int n = a.M > b ? (a.M - b + G - 1) / G : 0;  // rows of this block
    const bool dyn = a.mode == kNqDynamic;
    const uint32_t smem0 = smem_u32(rows_smem);

    // gamma words of this thread, for every row
    uint4 gw[NW];
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        const int w = tid + j * kNThreads;
        gw[j] = w < words ? __ldg(static_cast<const uint4 *>(a.gamma) + w) : make_uint4(0, 0, 0, 0);
    }

    if (tid == 0) {
        for (int i = 0; i < S; ++i) q_mbar_init(smem_u32(&full[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_sh = 0;
        if (dyn) {
            const unsigned e = *reinterpret_cast<volatile unsigned *>(a.epoch);
            epoch_sh = e;
            if (b == 0) {
                a.arrive[(e & 1u) ^ 1u] = 0u;
                a.amax[(e & 1u) ^ 1u] = 0u;
            }
        }
    }
    __syncthreads();

    // position i of a pass is row b + G * rowidx(i); it lives in stage
    // stage_of(i); after position i is consumed, position i + S is loaded
    // into the same stage.
    const int n_res = n < S ? n : S;  // rows still in shared memory after pass 1
    const int first_res = n - n_res;
    uint32_t pending = 0, par = 0;  // thread 0: copies not yet waited for; phase parities
    auto issue = [&](int row_idx, int s, bool keep) {
        const char *src = static_cast<const char *>(a.x) +
                          static_cast<size_t>(b + static_cast<size_t>(G) * row_idx) * row_bytes;
        bulk_load(smem0 + static_cast<uint32_t>(s) * row_bytes, src, row_bytes, smem_u32(&full[s]),
                  keep ? l2_evict_last() : l2_evict_first());
        pending |= 1u << s;
    };
    // every thread waits (bounded) for stage s itself; a time-out is noted in
    // abort_sh and acted on after the next block barrier, which keeps the
    // barriers uniform
    auto wait_stage = [&](int s) {
        if (!q_mbar_wait(smem_u32(&full[s]), (par >> s) & 1u, a.wait_cycles))
            abort_sh = 1;
        else if (tid == 0)
            pending &= ~(1u << s);
        par ^= 1u << s;
    };
    // the row's x words into registers and r = 1 / sqrt(ss / K + eps); after
    // the block sum every thread has read the stage, so thread 0 may refill
    // it
    int fflip = 0, uflip = 0;
    uint4 xv[NW];
    auto load_row = [&](int s) {
        const uint4 *src = rows_smem + static_cast<size_t>(s) * words;
        uint64_t acc = 0;
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const int w = tid + j * kNThreads;
            xv[j] = w < words ? src[w] : make_uint4(0, 0, 0, 0);
            acc = word_sumsq<DT>(xv[j], acc);
        }
        const float part = __fadd_rn(__uint_as_float(static_cast<uint32_t>(acc)),
                                     __uint_as_float(static_cast<uint32_t>(acc >> 32)));
        const float ss = block_sum<THREADS>(part, fred, fflip);
        const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(a.K)), a.eps)));
        return f2_pack(__float_as_uint(r), __float_as_uint(r));
    };
    auto store_row = [&](int row, const uint4 (&hv)[NW], const Quot *d, bool clamp) {
        const size_t base = static_cast<size_t>(row) * words;
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const int w = tid + j * kNThreads;
            if (w >= words) continue;
            if (a.h != nullptr) static_cast<uint4 *>(a.h)[base + w] = hv[j];
            if (d != nullptr) {
                const uint2 c = clamp ? codes_of_word<DT, true>(hv[j], *d) : codes_of_word<DT, false>(hv[j], *d);
                reinterpret_cast<uint2 *>(a.q)[base + w] = c;
            }
        }
    };

    if (tid == 0)
        for (int i = 0; i < n && i < S; ++i) issue(i, i, dyn && i < first_res);

    float s_static = 0.0f;
    if (a.mode == kNqStatic) s_static = *a.scale;
    uint32_t m_all = 0;  // dynamic: running magnitude maximum of h
    // ---- pass 1 (the only pass except in dynamic mode)
    for (int i = 0; i < n; ++i) {
        const int s = i % S;
        wait_stage(s);
        const uint64_t r2 = load_row(s);
        if (abort_sh) goto teardown;
        if (tid == 0 && i + S < n) issue(i + S, s, dyn && i + S < first_res);
        const int row = b + G * i;
        uint4 hv[NW];
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            hv[j] = norm_word<DT>(xv[j], gw[j], r2);
            m = word_mag_max<DT>(hv[j], m);  // zero words beyond the row add nothing
        }
        if (dyn) {
            m_all = max(m_all, fold_mag<DT>(m));  // m holds two 16-bit maxima
            if (i >= first_res) {
                // a row that stays on chip keeps h in place of x (each thread
                // rewrites only its own words): pass 2 only casts it
                uint4 *dst = rows_smem + static_cast<size_t>(s) * words;
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    const int w = tid + j * kNThreads;
                    if (w < words) dst[w] = hv[j];
                }
            }
        } else if (a.mode == kNqPerToken) {
            const uint32_t rm = block_max<THREADS>(fold_mag<DT>(m), ured, uflip);
            const float sc = scale_from_amax(mag_bits_to_float<DT>(rm));
            if (tid == 0) a.scale[row] = sc;
            const Quot d = Quot::make<DT>(sc);
            store_row(row, hv, &d, false);
        } else if (a.mode == kNqStatic) {
            const Quot d = Quot::make<DT>(s_static);
            store_row(row, hv, &d, true);
        } else {
            store_row(row, hv, nullptr, false);
        }
    }
    if (!dyn) return;
    {
        // ---- grid maximum, then pass 2: resident rows first (h already in
        // shared memory), then the others, re-read and normalized again
        const uint32_t bm = block_max_u32(fold_mag<DT>(m_all), bred);
        const unsigned pair = epoch_sh & 1u;
        // a single block has the maximum already and skips the barrier words
        const bool barrier = G > 1 || (a.stall & kStallGrid) != 0u;
        const unsigned expect = gridDim.x + ((a.stall & kStallGrid) ? 1u : 0u);
        uint32_t mm = bm;
        if (barrier && !grid_max(a.arrive + pair, a.amax + pair, bm, a.status, &mm, expect, a.wait_cycles))
            return;  // every copy of pass 1 was waited for
        const float sc = scale_from_amax(mag_bits_to_float<DT>(mm));
        if (b == 0 && tid == 0) {
            *a.scale = sc;
            if (barrier) *a.epoch = epoch_sh + 1u;
        }
        const Quot d = Quot::make<DT>(sc);
        for (int j = 0; j < n; ++j) {
            const int s = (first_res + j) % S;
            uint4 hv[NW];
            int idx;
            if (j < n_res) {
                idx = first_res + j;
                const uint4 *src = rows_smem + static_cast<size_t>(s) * words;
#pragma unroll
                for (int jj = 0; jj < NW; ++jj) {
                    const int w = tid + jj * kNThreads;
                    hv[jj] = w < words ? src[w] : make_uint4(0, 0, 0, 0);
                }
                if (j + S < n) {
                    __syncthreads();  // every thread has read the stage
                    if (tid == 0) issue(j + S - n_res, s, false);
                }
            } else {
                idx = j - n_res;
                wait_stage(s);
                const uint64_t r2 = load_row(s);
                if (abort_sh) goto teardown;
                if (tid == 0 && j + S < n) issue(j + S - n_res, s, false);
#pragma unroll
                for (int jj = 0; jj < NW; ++jj) hv[jj] = norm_word<DT>(xv[jj], gw[jj], r2);
            }
            store_row(b + G * idx, hv, &d, false);
        }
        return;
    }
teardown:
    // a wait gave up: record it, let this block's copies in flight land
    // before its shared memory is released (again bounded)
    if (tid == 0) {
        flag_timeout(a.status);
        for (int i = 0; i < S; ++i)
            if (pending & (1u << i)) q_mbar_wait(smem_u32(&full[i]), (par >> i) & 1u, kDefaultWaitCycles);
    }
}

__global__ void set_one_kernel(float *scale) { *scale = 1.0f; }

constexpr int kMaxDevicesN = 64;
constexpr int kNormVariants = 8;  // (dtype, threads, words per thread) instances
std::atomic<int> g_norm_ready[kMaxDevicesN][2][kNormVariants];

template <int DT, int THREADS, int NW>
bool norm_prepare(int variant) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesN) return false;
    auto &ready = g_norm_ready[dev][DT == FP8L_BF16 ? 1 : 0][variant];
    if (ready.load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(rmsnorm_quant_kernel<DT, THREADS, NW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kNormSmemBudget) != cudaSuccess)
        return false;
    ready.store(1, std::memory_order_release);
    return true;
}

// Blocks per SM and stages: up to 4 blocks of 256 threads (2 of 512) share
// the SM's row stages; the grid is every block that fits at once (all
// co-resident, as the dynamic mode's grid barrier needs), at most one per
// row.
template <int DT, int THREADS, int NW>
int launch_norm(NormArgs a, int sms, int variant, cudaStream_t stream) {
    if (!norm_prepare<DT, THREADS, NW>(variant)) return FP8L_ECUDA;
    const int row_bytes = a.K * 2;
    const int want = THREADS == 256 ? 4 : 2;
    int stages = (kNormSmemBudget / want) / row_bytes;
    if (stages < 1) stages = 1;
    if (stages > kNormMaxStages) stages = kNormMaxStages;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rmsnorm_quant_kernel<DT, THREADS, NW>,
                                                      THREADS, static_cast<size_t>(stages) * row_bytes) !=
            cudaSuccess ||
        per_sm < 1)
        return FP8L_ECUDA;
    const int64_t slots = int64_t(per_sm) * sms;
    const int grid = static_cast<int>(a.M < slots ? a.M : slots);
    const int rows_per = (a.M + grid - 1) / grid;
    if (stages > rows_per) stages = rows_per;
    a.stages = stages;
    const WaitConfig wc = wait_config();
    a.wait_cycles = wc.cycles;
    a.stall = wc.stall;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(stages) * row_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.mode == kNqDynamic ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, rmsnorm_quant_kernel<DT, THREADS, NW>, a) != cudaSuccess)
        return FP8L_ECUDA;
    return launch_status();
}

template <int DT>
int dispatch_nw(const NormArgs &a, int sms, cudaStream_t stream) {
    const int words = a.K / 8;
    if (words <= 256) return launch_norm<DT, 256, 1>(a, sms, 0, stream);
    if (words <= 512) return launch_norm<DT, 256, 2>(a, sms, 1, stream);
    if (words <= 1024) return launch_norm<DT, 256, 4>(a, sms, 2, stream);
    if (words <= 2048) return launch_norm<DT, 512, 4>(a, sms, 3, stream);
    return launch_norm<DT, 512, 8>(a, sms, 4, stream);
}

}  // namespace
}  // namespace fp8l

extern "C" int fp8_rmsnorm_quant(const void *x, int x_dtype, const void *gamma, float eps,
                                 int64_t M, int64_t K, uint8_t *q, float *scale, int mode,
                                 void *h, void *workspace, void *stream) {
    using namespace fp8l;
    if (x_dtype != FP8L_F16 && x_dtype != FP8L_BF16) return FP8L_EINVAL;
    if (mode < kNqDynamic || mode > kNqNormOnly) return FP8L_EINVAL;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return FP8L_EINVAL;  // also rejects NaN
    if (M < 0 || M > 0x7FFFFFFF || K <= 0 || K % 16 != 0 || K > kNormMaxK) return FP8L_ESHAPE;
    if (gamma == nullptr) return FP8L_EINVAL;
    if (mode == kNqNormOnly) {
        if (M > 0 && (x == nullptr || h == nullptr)) return FP8L_EINVAL;
    } else {
        if (scale == nullptr) return FP8L_EINVAL;
        if (M > 0 && (x == nullptr || q == nullptr)) return FP8L_EINVAL;
    }
    if (mode == kNqDynamic && workspace == nullptr) return FP8L_EINVAL;
    if (!aligned16(gamma) || (M > 0 && (!aligned16(x) || (q != nullptr && !aligned16(q)) ||
                                        (h != nullptr && !aligned16(h)))) ||
        (workspace != nullptr && !aligned16(workspace)) ||
        (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
        return FP8L_EALIGN;
    int sms = 0;
    int st = check_device(&sms);
    if (st != FP8L_OK) return st;
    cudaStream_t s = as_stream(stream);
    if (M == 0) {
        if (mode != kNqDynamic) return FP8L_OK;
        set_one_kernel<<<1, 1, 0, s>>>(scale);  // an empty tensor's dynamic scale
        return launch_status();
    }
    NormArgs a{};
    a.x = x;
    a.gamma = gamma;
    a.eps = eps;
    a.M = static_cast<int>(M);
    a.K = static_cast<int>(K);
    a.q = q;
    a.scale = scale;
    a.h = h;
    a.mode = mode;
    if (mode == kNqDynamic) {
        a.epoch = epoch_word(workspace);
        a.arrive = arrive_words(workspace);
        a.amax = amax_words(workspace);
    }
    a.status = workspace != nullptr ? status_word(workspace) : nullptr;
    return x_dtype == FP8L_BF16 ? dispatch_nw<FP8L_BF16>(a, sms, s) : dispatch_nw<FP8L_F16>(a, sms, s);
}

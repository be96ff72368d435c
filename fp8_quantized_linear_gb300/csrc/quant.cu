// Per-tensor and per-row quantization to OCP E4M3.
//
// Per-tensor, dynamic ("[Kernel][FP8] Initial support with dynamic per-tensor
// scaling", Algorithm): two bandwidth-bound launches.
//   1. absmax_kernel: every thread streams 16-element chunks with 16-byte
//      loads and keeps the running maximum of the magnitude BITS (sign bit
//      cleared; for finite IEEE values a larger magnitude has larger unsigned
//      bits, so the maximum is exact and needs no float compare).  Warp
//      reduction with redux.sync, block reduction in shared memory, one
//      partial per block.  The last block to finish (a ticket counter; no
//      block waits for another) reduces the partials, forms s = amax / 448
//      (one IEEE division; 1 when zero), writes s and resets the counter.
//   2. cast_kernel: q = E4M3_satRNE(fp32(x / s)) with the hardware saturating
//      round-to-nearest-even conversion.  The quotient is taken as
//      x * RN(1/s), which lies within 2 ulps of RN(x / s); where that product
//      is within 3 ulps of an E4M3 rounding midpoint (every normal-range
//      midpoint has the low 20 fp32 mantissa bits equal to 0x80000) or below
//      2^-6 (the E4M3 subnormal range), the IEEE division is taken instead.
//      Elsewhere both values round to the same code, so the codes equal
//      those of the division everywhere.
//   The cast re-reads X, which up to ~100 MB is still in the 126 MB L2.
// Static mode ("RFC: FP8 Quantization Schema in vLLM", input scales) runs
// only the cast kernel with s read from device memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"

namespace fp8l {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 16;  // elements per chunk (one 16-byte store of codes)

// uint4 words per chunk = bytes per element (16 elements)
template <int DT> struct Elt;
template <> struct Elt<FP8L_F16> { static constexpr int kBytes = 2; };
template <> struct Elt<FP8L_BF16> { static constexpr int kBytes = 2; };
template <> struct Elt<FP8L_F32> { static constexpr int kBytes = 4; };

template <int DT>
__device__ __forceinline__ void load_chunk(const uint4 *__restrict__ base, int64_t c,
                                           uint4 (&v)[Elt<DT>::kBytes]) {
#pragma unroll
    for (int i = 0; i < Elt<DT>::kBytes; ++i) v[i] = __ldg(base + c * Elt<DT>::kBytes + i);
}

// running max of magnitude bits; for 16-bit types two magnitudes per word
template <int DT>
__device__ __forceinline__ uint32_t chunk_mag_max(const uint4 (&v)[Elt<DT>::kBytes], uint32_t m) {
#pragma unroll
    for (int i = 0; i < Elt<DT>::kBytes; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (DT == FP8L_F32)
                m = max(m, w[j] & 0x7FFFFFFFu);
            else
                m = __vmaxu2(m, w[j] & 0x7FFF7FFFu);
        }
    }
    return m;
}

// fold packed 16-bit maxima into one magnitude bit pattern
template <int DT>
__device__ __forceinline__ uint32_t fold_mag(uint32_t m) {
    if constexpr (DT == FP8L_F32) return m;
    return max(m & 0xFFFFu, m >> 16);
}

template <int DT>
__device__ __forceinline__ float mag_bits_to_float(uint32_t m) {
    if constexpr (DT == FP8L_F32) return __uint_as_float(m);
    if constexpr (DT == FP8L_BF16) return __uint_as_float(m << 16);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(m)));
}

template <int DT>
__device__ __forceinline__ uint32_t scalar_mag_bits(const void *x, int64_t i) {
    if constexpr (DT == FP8L_F32)
        return __float_as_uint(static_cast<const float *>(x)[i]) & 0x7FFFFFFFu;
    return static_cast<uint32_t>(static_cast<const unsigned short *>(x)[i]) & 0x7FFFu;
}

template <int DT>
__device__ __forceinline__ float scalar_value(const void *x, int64_t i) {
    if constexpr (DT == FP8L_F32) return static_cast<const float *>(x)[i];
    if constexpr (DT == FP8L_BF16)
        return __uint_as_float(static_cast<uint32_t>(static_cast<const unsigned short *>(x)[i]) << 16);
    return __half2float(static_cast<const __half *>(x)[i]);
}

// the 16 values of a chunk as floats (exact widening)
template <int DT>
__device__ __forceinline__ void chunk_values(const uint4 (&v)[Elt<DT>::kBytes], float (&f)[kChunk]) {
#pragma unroll
    for (int i = 0; i < Elt<DT>::kBytes; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (DT == FP8L_F32) {
                f[i * 4 + j] = __uint_as_float(w[j]);
            } else if constexpr (DT == FP8L_BF16) {
                f[i * 8 + 2 * j] = __uint_as_float(w[j] << 16);
                f[i * 8 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            } else {
                __half2 h = *reinterpret_cast<const __half2 *>(&w[j]);
                float2 p = __half22float2(h);
                f[i * 8 + 2 * j] = p.x;
                f[i * 8 + 2 * j + 1] = p.y;
            }
        }
    }
}

// saturating round-to-nearest-even E4M3 codes of (a, b); a in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint8_t e4m3(float a) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3));
}

// A float whose saturating RNE E4M3 code is the code of RN(x / s), given
// r = RN(1 / s); `fast` is false when r is not a normal float.
__device__ __forceinline__ float quotient(float x, float s, float r, bool fast) {
    const float q = x * r;
    const uint32_t b = __float_as_uint(q) & 0x7FFFFFFFu;
    const bool tiny = (b - 1u) < 0x3C7FFFFFu;               // 0 < |q| < 2^-6
    const bool near_mid = ((b & 0xFFFFFu) - 0x7FFFDu) < 7u;  // within 3 ulps of ...8p
    if (!fast || tiny || near_mid) return __fdiv_rn(x, s);
    return q;
}

struct Divisor {
    float s, r;
    bool fast;
    __device__ __forceinline__ explicit Divisor(float scale) : s(scale) {
        r = __frcp_rn(scale);
        fast = r >= 1.17549435e-38f && r <= 3.40282347e+38f;
    }
    __device__ __forceinline__ float operator()(float x) const { return quotient(x, s, r, fast); }
};

__device__ __forceinline__ uint4 quant_chunk(const float (&f)[kChunk], const Divisor &d) {
    uint32_t p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = e4m3x2(d(f[2 * i]), d(f[2 * i + 1]));
    return make_uint4(p[0] | (p[1] << 16), p[2] | (p[3] << 16), p[4] | (p[5] << 16),
                      p[6] | (p[7] << 16));
}

// maximum over the block; every thread gets the result
__device__ __forceinline__ uint32_t block_max_u32(uint32_t m, uint32_t *red) {
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
        uint32_t v = lane < (blockDim.x >> 5) ? red[lane] : 0u;
        v = __reduce_max_sync(0xFFFFFFFFu, v);
        if (lane == 0) red[32] = v;
    }
    __syncthreads();
    return red[32];
}

__device__ __forceinline__ float scale_from_amax(float amax) {
    float s = __fdiv_rn(amax, kE4M3Max);
    return s == 0.0f ? 1.0f : s;
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
absmax_kernel(const void *__restrict__ x, int64_t numel, float *__restrict__ part,
              unsigned *__restrict__ ticket, float *__restrict__ scale) {
    __shared__ uint32_t red[33];
    __shared__ bool last;
    const uint4 *xv = static_cast<const uint4 *>(x);
    const int64_t n_chunks = numel / kChunk;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t c = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    uint32_t m = 0;
    for (; c + stride < n_chunks; c += 2 * stride) {
        uint4 v0[Elt<DT>::kBytes], v1[Elt<DT>::kBytes];
        load_chunk<DT>(xv, c, v0);
        load_chunk<DT>(xv, c + stride, v1);
        m = chunk_mag_max<DT>(v0, m);
        m = chunk_mag_max<DT>(v1, m);
    }
    if (c < n_chunks) {
        uint4 v0[Elt<DT>::kBytes];
        load_chunk<DT>(xv, c, v0);
        m = chunk_mag_max<DT>(v0, m);
    }
    m = fold_mag<DT>(m);
    const int64_t tail = numel - n_chunks * kChunk;
    if (blockIdx.x == 0 && threadIdx.x < tail)
        m = max(m, scalar_mag_bits<DT>(x, n_chunks * kChunk + threadIdx.x));
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) {
        part[blockIdx.x] = mag_bits_to_float<DT>(m);
        __threadfence();  // the partial is visible before the ticket is taken
        last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    // last block: every other block's partial is visible (their fences
    // precede their tickets); read them past L1
    __threadfence();
    uint32_t mm = 0;  // partials are non-negative floats: compare their bits
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += kThreads)
        mm = max(mm, __float_as_uint(__ldcg(part + i)));
    mm = block_max_u32(mm, red);
    if (threadIdx.x == 0) {
        *scale = scale_from_amax(__uint_as_float(mm));
        *ticket = 0u;  // ready for the next call
    }
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
cast_kernel(const void *__restrict__ x, int64_t numel, uint8_t *__restrict__ q,
            const float *__restrict__ scale) {
    const Divisor d(*scale);
    const uint4 *xv = static_cast<const uint4 *>(x);
    uint4 *qv = reinterpret_cast<uint4 *>(q);
    const int64_t n_chunks = numel / kChunk;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t c = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (; c + stride < n_chunks; c += 2 * stride) {
        uint4 v0[Elt<DT>::kBytes], v1[Elt<DT>::kBytes];
        float f[kChunk];
        load_chunk<DT>(xv, c, v0);
        load_chunk<DT>(xv, c + stride, v1);
        chunk_values<DT>(v0, f);
        qv[c] = quant_chunk(f, d);
        chunk_values<DT>(v1, f);
        qv[c + stride] = quant_chunk(f, d);
    }
    if (c < n_chunks) {
        uint4 v[Elt<DT>::kBytes];
        float f[kChunk];
        load_chunk<DT>(xv, c, v);
        chunk_values<DT>(v, f);
        qv[c] = quant_chunk(f, d);
    }
    const int64_t tail = numel - n_chunks * kChunk;
    if (blockIdx.x == 0 && threadIdx.x < tail) {
        const int64_t i = n_chunks * kChunk + threadIdx.x;
        q[i] = e4m3(d(scalar_value<DT>(x, i)));
    }
}

// one block per row; cols is a multiple of 16
template <int DT>
__global__ void __launch_bounds__(kThreads)
row_quant_kernel(const void *__restrict__ x, int64_t cols, uint8_t *__restrict__ q,
                 float *__restrict__ row_scale) {
    __shared__ uint32_t red[33];
    const int64_t r = blockIdx.x;
    const int64_t n_chunks = cols / kChunk;
    const uint4 *xv = reinterpret_cast<const uint4 *>(
        static_cast<const char *>(x) + r * cols * Elt<DT>::kBytes);
    uint4 *qv = reinterpret_cast<uint4 *>(q + r * cols);
    uint32_t m = 0;
    for (int64_t c = threadIdx.x; c < n_chunks; c += kThreads) {
        uint4 v[Elt<DT>::kBytes];
        load_chunk<DT>(xv, c, v);
        m = chunk_mag_max<DT>(v, m);
    }
    m = block_max_u32(fold_mag<DT>(m), red);
    const float s = scale_from_amax(mag_bits_to_float<DT>(m));
    if (threadIdx.x == 0) row_scale[r] = s;
    const Divisor d(s);
    for (int64_t c = threadIdx.x; c < n_chunks; c += kThreads) {
        uint4 v[Elt<DT>::kBytes];
        float f[kChunk];
        load_chunk<DT>(xv, c, v);
        chunk_values<DT>(v, f);
        qv[c] = quant_chunk(f, d);
    }
}

constexpr int64_t kMaxNumel = int64_t(1) << 40;

// absmax blocks: about two 16-element chunks per thread, at most 8 per SM
// and at most `max_part` (the room for partial maxima)
int absmax_blocks(int64_t numel, int sms, int max_part) {
    const int64_t n_chunks = numel / kChunk;
    int64_t blocks = (n_chunks + 2 * kThreads - 1) / (2 * kThreads);
    if (blocks < 1) blocks = 1;
    if (blocks > int64_t(sms) * 8) blocks = int64_t(sms) * 8;
    if (blocks > max_part) blocks = max_part;
    return static_cast<int>(blocks);
}

int cast_blocks(int64_t numel, int sms) {
    const int64_t need = (numel / kChunk + 2 * kThreads - 1) / (2 * kThreads);
    const int64_t cap = int64_t(sms) * 8;
    return static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
}

// dynamic: absmax (+ scale) then cast; static: cast with the given scale.
// `part` holds max_part floats; `ticket` is zero between calls.
template <int DT>
int run_quant(const void *x, int64_t numel, uint8_t *q, float *scale, bool dynamic, float *part,
              unsigned *ticket, int max_part, cudaStream_t stream, int sms) {
    if (dynamic) {
        absmax_kernel<DT><<<absmax_blocks(numel, sms, max_part), kThreads, 0, stream>>>(
            x, numel, part, ticket, scale);
        if (launch_status() != FP8L_OK) return FP8L_ECUDA;
    }
    if (numel == 0) return FP8L_OK;
    cast_kernel<DT><<<cast_blocks(numel, sms), kThreads, 0, stream>>>(x, numel, q, scale);
    return launch_status();
}

// ---------------------------------------------------------------------------
// Single-pass dynamic quantization: one cooperative launch whose blocks are
// all resident.  Each block owns a contiguous run of chunks; it loads them
// (keeping them in shared memory when they fit), writes its partial maximum,
// meets the other blocks at a grid barrier, reduces all partials to the same
// scale, and casts its chunks from shared memory (or from a second read of X
// when they did not fit).

constexpr long long kBarrierCycles = 4LL << 30;  // ~2 s: a healthy barrier takes microseconds
constexpr int kCacheBytes = 100 * 1024;          // per block; two blocks per SM

// Grid barrier for a co-resident grid.  Thread 0 of every block arrives on
// `count`; the last arrival resets it and advances `gen`; the others wait,
// bounded, for `gen` to move.  Returns false after a time-out, which is
// recorded in `status`.
__device__ bool grid_barrier(unsigned *count, unsigned *gen, unsigned *status) {
    __shared__ int ok_sh;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        volatile unsigned *vgen = gen;
        const unsigned g0 = *vgen;
        __threadfence();
        if (atomicAdd(count, 1u) == gridDim.x - 1) {
            *count = 0u;
            __threadfence();
            atomicAdd(gen, 1u);
        } else {
            const long long t0 = clock64();
            while (*vgen == g0) {
                if (clock64() - t0 > kBarrierCycles) {
                    atomicOr(status, kStatusTimeout);
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
        ok_sh = ok;
    }
    __syncthreads();
    return ok_sh != 0;
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
quant_fused_kernel(const void *__restrict__ x, int64_t numel, uint8_t *__restrict__ q,
                   float *__restrict__ scale, float *__restrict__ part, unsigned *count,
                   unsigned *gen, unsigned *status, int64_t per, int64_t cache_chunks) {
    extern __shared__ __align__(16) uint4 cache[];
    __shared__ uint32_t red[33];
    constexpr int V = Elt<DT>::kBytes;  // uint4 words per chunk
    const uint4 *xv = static_cast<const uint4 *>(x);
    uint4 *qv = reinterpret_cast<uint4 *>(q);
    const int64_t n_chunks = numel / kChunk;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t c1 = c0 + per < n_chunks ? c0 + per : n_chunks;
    const bool cached = c1 - c0 <= cache_chunks;

    // up to four chunks per thread requested at once (one round trip)
    uint32_t m = 0;
    int64_t c;
    for (int64_t base = c0 + threadIdx.x; base < c1; base += 4 * kThreads) {
        uint4 v[4][V];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (base + u * kThreads < c1) load_chunk<DT>(xv, base + u * kThreads, v[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t cu = base + u * kThreads;
            if (cu < c1) {
                m = chunk_mag_max<DT>(v[u], m);
                if (cached)
#pragma unroll
                    for (int i = 0; i < V; ++i) cache[(cu - c0) * V + i] = v[u][i];
            }
        }
    }
    m = fold_mag<DT>(m);
    const int64_t tail = numel - n_chunks * kChunk;
    if (blockIdx.x == 0 && threadIdx.x < tail)
        m = max(m, scalar_mag_bits<DT>(x, n_chunks * kChunk + threadIdx.x));
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) part[blockIdx.x] = mag_bits_to_float<DT>(m);

    if (!grid_barrier(count, gen, status)) return;

    uint32_t mm = 0;  // partials are non-negative floats: compare their bits
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += kThreads)
        mm = max(mm, __float_as_uint(__ldcg(part + i)));
    mm = block_max_u32(mm, red);
    const float s = scale_from_amax(__uint_as_float(mm));
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale = s;
    const Divisor d(s);
    for (c = c0 + threadIdx.x; c < c1; c += kThreads) {
        uint4 v[V];
        if (cached) {
#pragma unroll
            for (int i = 0; i < V; ++i) v[i] = cache[(c - c0) * V + i];
        } else {
            load_chunk<DT>(xv, c, v);
        }
        float f[kChunk];
        chunk_values<DT>(v, f);
        qv[c] = quant_chunk(f, d);
    }
    if (blockIdx.x == 0 && threadIdx.x < tail) {
        const int64_t i = n_chunks * kChunk + threadIdx.x;
        q[i] = e4m3(d(scalar_value<DT>(x, i)));
    }
}

constexpr int kMaxDevicesQ = 64;
std::atomic<int> g_fused_blocks[kMaxDevicesQ][4];  // co-resident blocks per SM, uncached

template <int DT>
int fused_blocks_per_sm_uncached() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesQ) return 0;
    int nb = g_fused_blocks[dev][DT].load(std::memory_order_acquire);
    if (nb == 0) {
        if (cudaFuncSetAttribute(quant_fused_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kCacheBytes) != cudaSuccess)
            return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, quant_fused_kernel<DT>, kThreads, 0) !=
                cudaSuccess ||
            nb < 1)
            return 0;
        g_fused_blocks[dev][DT].store(nb, std::memory_order_release);
    }
    return nb;
}

template <int DT>
int run_fused(const void *x, int64_t numel, uint8_t *q, float *scale, void *workspace,
              cudaStream_t stream, int sms) {
    const int nb = fused_blocks_per_sm_uncached<DT>();
    if (nb == 0) return FP8L_ECUDA;
    const int64_t n_chunks = numel / kChunk;
    constexpr int64_t kChunkBytes = int64_t(kChunk) * Elt<DT>::kBytes;
    // cached: two blocks per SM hold their whole run in shared memory
    int64_t grid = int64_t(sms) * 2;
    int64_t per = (n_chunks + grid - 1) / grid;
    int64_t smem = per * kChunkBytes;
    if (smem > kCacheBytes) {
        // too large to keep on chip: as many resident blocks as fit, X read twice
        grid = int64_t(sms) * nb;
        if (grid > kMaxPartials) grid = kMaxPartials;
        per = (n_chunks + grid - 1) / grid;
        smem = 0;
    }
    // no more blocks than chunks need (at least one block)
    const int64_t need = (n_chunks + kThreads - 1) / kThreads;
    if (grid > need) {
        grid = need < 1 ? 1 : need;
        per = (n_chunks + grid - 1) / grid;
        if (smem) smem = per * kChunkBytes;
    }
    const int64_t cache_chunks = smem / kChunkBytes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, quant_fused_kernel<DT>, x, numel, q, scale, partials(workspace),
                           ticket_word(workspace), gen_word(workspace),
                           status_word(workspace), per, cache_chunks) != cudaSuccess)
        return FP8L_ECUDA;
    return launch_status();
}

template <int DT>
int run_per_tensor(const void *x, int64_t numel, uint8_t *q, float *scale, bool dynamic,
                   void *workspace, cudaStream_t stream, int sms) {
    if (dynamic && numel > 0) return run_fused<DT>(x, numel, q, scale, workspace, stream, sms);
    float *part = dynamic ? partials(workspace) : nullptr;
    unsigned *tk = dynamic ? ticket_word(workspace) : nullptr;
    return run_quant<DT>(x, numel, q, scale, dynamic, part, tk, kMaxPartials, stream, sms);
}

template <int DT>
int run_per_row(const void *x, int64_t rows, int64_t cols, uint8_t *q, float *row_scale,
                cudaStream_t stream) {
    if (rows == 0) return FP8L_OK;
    // an empty row (cols == 0) gets amax 0, hence scale 1
    row_quant_kernel<DT><<<static_cast<unsigned>(rows), kThreads, 0, stream>>>(x, cols, q, row_scale);
    return launch_status();
}

bool valid_in_dtype(int dt) { return dt == FP8L_F16 || dt == FP8L_BF16 || dt == FP8L_F32; }

}  // namespace
}  // namespace fp8l

extern "C" int fp8_quant_per_tensor(const void *x, int x_dtype, int64_t rows, int64_t cols,
                                    uint8_t *q, float *scale, int dynamic, void *workspace,
                                    void *stream) {
    using namespace fp8l;
    if (!valid_in_dtype(x_dtype) || scale == nullptr) return FP8L_EINVAL;
    if (rows < 0 || cols < 0) return FP8L_ESHAPE;
    if (cols != 0 && rows > kMaxNumel / cols) return FP8L_ESHAPE;
    const int64_t numel = rows * cols;
    if (numel > 0 && (x == nullptr || q == nullptr)) return FP8L_EINVAL;
    if (dynamic && workspace == nullptr) return FP8L_EINVAL;
    if ((numel > 0 && (!aligned16(x) || !aligned16(q))) || !aligned16(workspace))
        return FP8L_EALIGN;
    if ((reinterpret_cast<uintptr_t>(scale) & 3u) != 0) return FP8L_EALIGN;
    int sms = 0;
    int st = check_device(&sms);
    if (st != FP8L_OK) return st;
    cudaStream_t s = as_stream(stream);
    switch (x_dtype) {
        case FP8L_F16: return run_per_tensor<FP8L_F16>(x, numel, q, scale, dynamic != 0, workspace, s, sms);
        case FP8L_BF16: return run_per_tensor<FP8L_BF16>(x, numel, q, scale, dynamic != 0, workspace, s, sms);
        default: return run_per_tensor<FP8L_F32>(x, numel, q, scale, dynamic != 0, workspace, s, sms);
    }
}

extern "C" int fp8_quant_per_row(const void *x, int x_dtype, int64_t rows, int64_t cols,
                                 uint8_t *q, float *row_scale, void *stream) {
    using namespace fp8l;
    if (!valid_in_dtype(x_dtype)) return FP8L_EINVAL;
    if (rows < 0 || cols < 0 || rows > 0x7FFFFFFF || cols > (int64_t(1) << 20) || cols % 16 != 0)
        return FP8L_ESHAPE;
    if (rows > 0 && (x == nullptr || q == nullptr || row_scale == nullptr)) return FP8L_EINVAL;
    if (rows > 0 && (!aligned16(x) || !aligned16(q) ||
                     (reinterpret_cast<uintptr_t>(row_scale) & 3u) != 0))
        return FP8L_EALIGN;
    int st = check_device(nullptr);
    if (st != FP8L_OK) return st;
    cudaStream_t s = as_stream(stream);
    switch (x_dtype) {
        case FP8L_F16: return run_per_row<FP8L_F16>(x, rows, cols, q, row_scale, s);
        case FP8L_BF16: return run_per_row<FP8L_BF16>(x, rows, cols, q, row_scale, s);
        default: return run_per_row<FP8L_F32>(x, rows, cols, q, row_scale, s);
    }
}

// ---------------------------------------------------------------------------
// Dynamic per-tensor quantization without a caller-provided workspace.
//
// Some callers cannot allocate device memory: a plug-in that runs inside a
// host framework which owns every device allocation through its own pool and
// forbids direct cudaMalloc, or a serving loop that fixed its memory
// footprint at start-up and has no way to hand a workspace down to this
// call.  For them, the per-block partial maxima live in the array below,
// which is part of the library image: every GPU that loads the library holds
// it (8 KiB) until the process exits.
#include <atomic>

namespace fp8l {
namespace {

// 2048 partial maxima, then one ticket word that is zero between calls (zero
// at load, and every call leaves it at zero)
constexpr int kNoallocMaxPartials = 2048;
static __device__ __align__(256) float g_noalloc_partials[kNoallocMaxPartials + 64];

constexpr int kNoallocMaxDevices = 64;
std::atomic<float *> g_noalloc_ptr[kNoallocMaxDevices];

// Device address of g_noalloc_partials on the current device.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
int noalloc_scratch(float **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8L_ECUDA;
    if (dev < 0 || dev >= kNoallocMaxDevices) return FP8L_EUNSUPPORTED;
    float *p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_partials) != cudaSuccess || addr == nullptr)
            return FP8L_ECUDA;
        p = static_cast<float *>(addr);
        g_noalloc_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return FP8L_OK;
}

template <int DT>
int run_noalloc(const void *x, int64_t numel, uint8_t *q, float *scale, float *part,
                cudaStream_t stream, int sms) {
    // each block writes its own partial and the last block reads exactly the
    // partials this call wrote; only the ticket word must start at zero
    unsigned *tk = reinterpret_cast<unsigned *>(part + kNoallocMaxPartials);
    return run_quant<DT>(x, numel, q, scale, true, part, tk, kNoallocMaxPartials, stream, sms);
}

}  // namespace
}  // namespace fp8l

extern "C" int fp8_quant_per_tensor_noalloc(const void *x, int x_dtype, int64_t rows,
                                            int64_t cols, uint8_t *q, float *scale,
                                            void *stream) {
    using namespace fp8l;
    if (!valid_in_dtype(x_dtype) || scale == nullptr) return FP8L_EINVAL;
    if (rows < 0 || cols < 0) return FP8L_ESHAPE;
    if (cols != 0 && rows > kMaxNumel / cols) return FP8L_ESHAPE;
    const int64_t numel = rows * cols;
    if (numel > 0 && (x == nullptr || q == nullptr)) return FP8L_EINVAL;
    if (numel > 0 && (!aligned16(x) || !aligned16(q))) return FP8L_EALIGN;
    if ((reinterpret_cast<uintptr_t>(scale) & 3u) != 0) return FP8L_EALIGN;
    int sms = 0;
    int st = check_device(&sms);
    if (st != FP8L_OK) return st;
    float *part = nullptr;
    st = noalloc_scratch(&part);
    if (st != FP8L_OK) return st;
    cudaStream_t s = as_stream(stream);
    switch (x_dtype) {
        case FP8L_F16: return run_noalloc<FP8L_F16>(x, numel, q, scale, part, s, sms);
        case FP8L_BF16: return run_noalloc<FP8L_BF16>(x, numel, q, scale, part, s, sms);
        default: return run_noalloc<FP8L_F32>(x, numel, q, scale, part, s, sms);
    }
}

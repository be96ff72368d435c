// Per-tensor and per-row quantization to OCP E4M3.
//
// Per-tensor ("[Kernel][FP8] Initial support with dynamic per-tensor scaling",
// Algorithm; static input scales: "RFC: FP8 Quantization Schema in vLLM"):
// one launch, quant_tma_kernel, one block per SM.  X is cut into pieces that
// the blocks stream through shared memory with bulk copies (TMA).  Dynamic
// mode reads X once for the maximum magnitude (exact: the maximum of the
// magnitude bit patterns), meets at a grid barrier to form s = amax / 448
// (one IEEE division; 1 when zero), and casts the pieces still on chip, then
// the rest; static mode reads s from device memory and casts in one pass.
// Every code is E4M3_satRNE(RN(x / s)): the hardware saturating
// round-to-nearest-even conversion of the correctly rounded fp32 quotient,
// which is formed with fused multiply-adds (see Quot).
//
// The two-launch variant (absmax_kernel, then cast_kernel: no block waits for
// another) serves the entry point without a workspace and the empty tensor.
// Per-row quantization (the per-output-channel weight scale) is one block per
// row.
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

// saturating round-to-nearest-even E4M3 codes of (a, b); a in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint8_t e4m3(float a) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3));
}

// ---------------------------------------------------------------------------
// E4M3 codes of x / s, equal to the codes of the IEEE quotient RN(x / s).
//
// The quotient is formed without a division.  With y = RN(1/s):
//   q0 = RN(x * y)
//   q1 = RN(q0 + r0 * y),  r0 = RN(x - s * q0)
//   q2 = RN(q1 + r1 * y),  r1 = RN(x - s * q1)
// (each residual and each correction is one fused multiply-add).  q1 is a
// faithful rounding of x / s, and from a faithful quotient and the correctly
// rounded reciprocal one more correction gives the correctly rounded
// quotient (Markstein's theorem: P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop.
// 34(1), 1990), as long as the residual x - s*q does not underflow and no
// intermediate overflows.  For 16-bit inputs q1 is already RN(x / s): all
// these quantities scale exactly with powers of two, so the claim reduces to
// every pair (significand of x, significand of s), 2^30 pairs for bfloat16
// and 2^33 for fp16, and an exhaustive check over all of them finds q1 equal
// to the IEEE quotient in every case.  fp32 inputs take both corrections.  That holds here when 2^-92 <= s <= 2^100 (then
// every x that can reach a nonzero code has |x| >= 2^-103, where the residual
// is exact) and |x / s| stays finite: a static scale with 16-bit brain-float
// or fp32 input clamps |x| below 1024 * s first, which leaves every code
// unchanged (beyond 464 * s all codes saturate to 448).  Outside that range of
// s every element takes the IEEE division.  The arithmetic runs on pairs with
// the packed f32x2 instructions.  The sign of each code is taken from its
// input, which keeps -0 (and anything that rounds to zero) signed.
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f2_pack(uint32_t lo_bits, uint32_t hi_bits) {
    return (static_cast<uint64_t>(hi_bits) << 32) | lo_bits;
}

// codes of the four floats of two pairs, packed in order (first float in the
// low byte)
__device__ __forceinline__ uint32_t f2_codes4(uint64_t q01, uint64_t q23) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(__uint_as_float(static_cast<uint32_t>(q01))), "f"(__uint_as_float(static_cast<uint32_t>(q01 >> 32))),
          "f"(__uint_as_float(static_cast<uint32_t>(q23))), "f"(__uint_as_float(static_cast<uint32_t>(q23 >> 32))));
    return r;
}

struct Quot {
    float s;
    uint64_t y2, ns2;  // {RN(1/s), RN(1/s)}, {-s, -s}
    uint32_t clamp;    // clamp of |x| (16-bit pairs for 16-bit types), static mode
    bool fast;

    template <int DT>
    __device__ __forceinline__ static Quot make(float scale) {
        Quot d;
        d.s = scale;
        d.fast = scale >= 0x1p-92f && scale <= 0x1p100f;
        const float y = __frcp_rn(scale);
        d.y2 = f2_pack(__float_as_uint(y), __float_as_uint(y));
        d.ns2 = f2_pack(__float_as_uint(-scale), __float_as_uint(-scale));
        const uint32_t c = __float_as_uint(1024.0f * scale);  // finite and normal when fast
        d.clamp = DT == FP8L_F32 ? c : ((c >> 16) | (c & 0xFFFF0000u));
        return d;
    }

    // RN(x / s) for a pair; CORRECTIONS = 2 in general, 1 for 16-bit inputs
    template <int CORRECTIONS>
    __device__ __forceinline__ uint64_t pair(uint64_t x) const {
        uint64_t q = f2_mul(x, y2);
#pragma unroll
        for (int i = 0; i < CORRECTIONS; ++i) {
            const uint64_t r = f2_fma(ns2, q, x);
            q = f2_fma(r, y2, q);
        }
        return q;
    }
};

// widen the 16-bit pair in w (element 0 in the low half) to a float pair
template <int DT>
__device__ __forceinline__ uint64_t widen16(uint32_t w) {
    if constexpr (DT == FP8L_BF16) {
        return f2_pack(w << 16, w & 0xFFFF0000u);
    } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
        return f2_pack(__float_as_uint(f.x), __float_as_uint(f.y));
    }
}

// E4M3 codes of one 16-byte word of X: 8 codes for 16-bit types (uint2), 4
// for fp32 (in .x).  CLAMP: static scale (see above).
template <int DT, bool CLAMP>
__device__ __forceinline__ uint2 codes_of_word(const uint4 &v, const Quot &d) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (DT == FP8L_F32) {
        uint32_t c;
        if (d.fast) {
            uint32_t m[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) m[j] = CLAMP ? min(w[j] & 0x7FFFFFFFu, d.clamp) : w[j];
            c = f2_codes4(d.pair<2>(f2_pack(m[0], m[1])), d.pair<2>(f2_pack(m[2], m[3])));
        } else {
            c = __byte_perm(e4m3x2(__fdiv_rn(__uint_as_float(w[0]), d.s), __fdiv_rn(__uint_as_float(w[1]), d.s)),
                            e4m3x2(__fdiv_rn(__uint_as_float(w[2]), d.s), __fdiv_rn(__uint_as_float(w[3]), d.s)),
                            0x5410);
        }
        const uint32_t signs = __byte_perm(__byte_perm(w[0], w[1], 0x0073), __byte_perm(w[2], w[3], 0x0073), 0x5410);
        return make_uint2((c & 0x7F7F7F7Fu) | (signs & 0x80808080u), 0u);
    } else {
        uint32_t lo, hi;
        if (d.fast) {
            uint64_t q[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t m = (CLAMP && DT == FP8L_BF16) ? __vminu2(w[j] & 0x7FFF7FFFu, d.clamp) : w[j];
                q[j] = d.pair<1>(widen16<DT>(m));
            }
            lo = f2_codes4(q[0], q[1]);
            hi = f2_codes4(q[2], q[3]);
        } else {
            uint32_t c[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint64_t x = widen16<DT>(w[j]);
                c[j] = e4m3x2(__fdiv_rn(__uint_as_float(static_cast<uint32_t>(x)), d.s),
                              __fdiv_rn(__uint_as_float(static_cast<uint32_t>(x >> 32)), d.s));
            }
            lo = __byte_perm(c[0], c[1], 0x5410);
            hi = __byte_perm(c[2], c[3], 0x5410);
        }
        return make_uint2((lo & 0x7F7F7F7Fu) | (__byte_perm(w[0], w[1], 0x7531) & 0x80808080u),
                          (hi & 0x7F7F7F7Fu) | (__byte_perm(w[2], w[3], 0x7531) & 0x80808080u));
    }
}

// codes of one 16-element chunk (Elt<DT>::kBytes words) as one 16-byte store
template <int DT, bool CLAMP>
__device__ __forceinline__ uint4 quant_chunk(const uint4 (&v)[Elt<DT>::kBytes], const Quot &d) {
    if constexpr (DT == FP8L_F32) {
        return make_uint4(codes_of_word<DT, CLAMP>(v[0], d).x, codes_of_word<DT, CLAMP>(v[1], d).x,
                          codes_of_word<DT, CLAMP>(v[2], d).x, codes_of_word<DT, CLAMP>(v[3], d).x);
    } else {
        const uint2 a = codes_of_word<DT, CLAMP>(v[0], d), b = codes_of_word<DT, CLAMP>(v[1], d);
        return make_uint4(a.x, a.y, b.x, b.y);
    }
}

// code of one element (ragged tails): the IEEE division itself
__device__ __forceinline__ uint8_t code_of(float x, float s) { return e4m3(__fdiv_rn(x, s)); }

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
    const float sc = *scale;
    const Quot d = Quot::make<DT>(sc);
    const uint4 *xv = static_cast<const uint4 *>(x);
    uint4 *qv = reinterpret_cast<uint4 *>(q);
    const int64_t n_chunks = numel / kChunk;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t c = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (; c + stride < n_chunks; c += 2 * stride) {
        uint4 v0[Elt<DT>::kBytes], v1[Elt<DT>::kBytes];
        load_chunk<DT>(xv, c, v0);
        load_chunk<DT>(xv, c + stride, v1);
        qv[c] = quant_chunk<DT, true>(v0, d);
        qv[c + stride] = quant_chunk<DT, true>(v1, d);
    }
    if (c < n_chunks) {
        uint4 v[Elt<DT>::kBytes];
        load_chunk<DT>(xv, c, v);
        qv[c] = quant_chunk<DT, true>(v, d);
    }
    const int64_t tail = numel - n_chunks * kChunk;
    if (blockIdx.x == 0 && threadIdx.x < tail) {
        const int64_t i = n_chunks * kChunk + threadIdx.x;
        q[i] = code_of(scalar_value<DT>(x, i), sc);
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
    const Quot d = Quot::make<DT>(s);
    for (int64_t c = threadIdx.x; c < n_chunks; c += kThreads) {
        uint4 v[Elt<DT>::kBytes];
        load_chunk<DT>(xv, c, v);
        qv[c] = quant_chunk<DT, true>(v, d);
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
// Single-read dynamic quantization staged by the bulk-copy (TMA) engine.
//
// One block per SM, all blocks co-resident (cooperative launch).  X is cut
// into pieces of whole 16-byte words dealt round-robin to the blocks; each
// block streams its pieces through a ring of shared-memory stages with
// cp.async.bulk, each stage completed by an mbarrier transaction count, so up
// to kStages * kPieceBytes bytes per SM are in flight with no registers held
// for them.
//   pass 1: the magnitude maximum of every piece as it lands; the last
//           `stages` pieces stay in shared memory.
//   barrier: the block maximums meet in one workspace word (atomicMax) at a
//           grid barrier; every block derives the same scale from it (block 0
//           stores it).
//   pass 2: the resident pieces are cast first; the pieces that did not stay
//           resident are streamed again, most recently read first (the ones
//           most likely still in L2).
// When the whole tensor fits in the stages (up to ~29 MB of X on 152 SMs) X is
// read from HBM exactly once.  Static mode skips pass 1 and the barrier and
// streams every piece once.

constexpr int kTThreads = 512;
constexpr int kPieceBytes = 32 * 1024;
constexpr int kPieceWords = kPieceBytes / 16;
constexpr int kStages = 6;
// Pass 1 reads each block's pieces from the highest address down and keeps the
// last ones read (the lowest) on chip; pass 2 then casts those and re-reads
// the rest in ascending order, most recently read (likeliest in L2) first.
constexpr bool kPass1Descending = true;
constexpr bool kRecentFirst = true;
constexpr int kMinPieceWords = 512;              // 8 KB: fewer, fuller blocks for small tensors
constexpr long long kWaitCycles = 4LL << 30;     // ~2 s: a healthy wait takes microseconds

__device__ __forceinline__ void q_mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool q_mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// bounded wait for the phase of parity `parity`; false after ~2 s
__device__ __forceinline__ bool q_mbar_wait(uint32_t bar, uint32_t parity) {
    if (q_mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!q_mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// one bulk copy of `bytes` (a multiple of 16) from global to shared memory,
// completing on mbarrier `bar`
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// L2 eviction priorities for the bulk copies
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// record a given-up wait (static mode may run without a workspace)
__device__ __forceinline__ void flag_timeout(unsigned *status) {
    if (status != nullptr) atomicOr(status, kStatusTimeout);
}

// Grid-wide maximum and barrier for a co-resident grid.  Thread 0 of every
// block folds its block maximum into `amax` (atomicMax on the magnitude bits)
// and then arrives on `arrive` with a release add; every block waits, bounded,
// until all gridDim.x arrivals are visible (acquire), which orders every
// block's maximum before its read of `amax`.  The chain is one atomic, one
// fenced add and the polling; nothing is reset here (the caller's pair of
// words alternates between calls).  Returns false after a time-out, which is
// recorded in `status`; *out receives the grid maximum.
__device__ bool grid_max(unsigned *arrive, unsigned *amax, uint32_t m, unsigned *status, uint32_t *out) {
    __shared__ int ok_sh;
    __shared__ uint32_t max_sh;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        atomicMax(amax, m);
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(arrive) : "memory");
        const long long t0 = clock64();
        for (;;) {
            unsigned c;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(arrive) : "memory");
            if (c >= gridDim.x) break;
            if (clock64() - t0 > kWaitCycles) {
                flag_timeout(status);
                ok = 0;
                break;
            }
        }
        uint32_t v;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(amax) : "memory");
        max_sh = v;
        ok_sh = ok;
    }
    __syncthreads();
    *out = max_sh;
    return ok_sh != 0;
}

// magnitude maximum of one 16-byte word (packed for 16-bit types)
template <int DT>
__device__ __forceinline__ uint32_t word_mag_max(const uint4 &v, uint32_t m) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (DT == FP8L_F32)
            m = max(m, w[j] & 0x7FFFFFFFu);
        else
            m = __vmaxu2(m, w[j] & 0x7FFF7FFFu);
    }
    return m;
}

// codes of one 16-byte word of X stored at q + word * (16 / element bytes)
template <int DT, bool CLAMP>
__device__ __forceinline__ void cast_word(const uint4 &v, const Quot &d, uint8_t *q, int word) {
    const uint2 c = codes_of_word<DT, CLAMP>(v, d);
    if constexpr (DT == FP8L_F32)
        reinterpret_cast<uint32_t *>(q)[word] = c.x;
    else
        reinterpret_cast<uint2 *>(q)[word] = c;
}

template <int DT, bool DYN>
__global__ void __launch_bounds__(kTThreads, 1)
quant_tma_kernel(const void *__restrict__ x, int64_t numel, uint8_t *__restrict__ q,
                 float *__restrict__ scale, unsigned *epoch, unsigned *arrive, unsigned *amax,
                 unsigned *status, int piece_words, int total_pieces, int stages, int keep_pieces) {
    extern __shared__ __align__(128) uint4 stage_mem[];
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ uint32_t red[33];
    __shared__ int abort_sh;
    __shared__ unsigned epoch_sh;
    constexpr int EB = Elt<DT>::kBytes;
    constexpr int EPW = 16 / EB;  // elements per 16-byte word
    const int tid = threadIdx.x;
    const int G = static_cast<int>(gridDim.x);
    const int b = static_cast<int>(blockIdx.x);
    const int64_t n_words = numel / EPW;
    // piece k of this block is piece b + k * G of X: the blocks sweep X
    // together, so the pages in use at any time stay few.  Only the last
    // piece of X can be short.
    const int npieces = total_pieces > b ? (total_pieces - b + G - 1) / G : 0;
    const int last_words = static_cast<int>(n_words - static_cast<int64_t>(total_pieces - 1) * piece_words);
    auto words_of = [&](int k) { return b + k * G == total_pieces - 1 ? last_words : piece_words; };
    auto first_word = [&](int k) { return static_cast<int64_t>(b + k * G) * piece_words; };
    const uint32_t smem0 = smem_u32(stage_mem);
    const uint32_t stage_bytes = static_cast<uint32_t>(piece_words) * 16u;

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) q_mbar_init(smem_u32(&full[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_sh = 0;
        if constexpr (DYN) {
            // this call's pair of barrier words is zero; clear the other pair
            // for the next call (the previous call has finished with it)
            const unsigned e = *reinterpret_cast<volatile unsigned *>(epoch);
            epoch_sh = e;
            if (blockIdx.x == 0) {
                arrive[(e & 1u) ^ 1u] = 0u;
                amax[(e & 1u) ^ 1u] = 0u;
            }
        }
    }
    __syncthreads();

    uint32_t pending = 0;  // thread 0: stages with a copy not yet waited for
    // keep: the piece is read again soon (pass 2 of a tensor too large for the
    // stages) and should stay in L2; every other read of X is its last
    auto issue = [&](int k, int s, bool keep) {
        bulk_load(smem0 + s * stage_bytes, static_cast<const char *>(x) + first_word(k) * 16,
                  static_cast<uint32_t>(words_of(k)) * 16u, smem_u32(&full[s]),
                  keep ? l2_evict_last() : l2_evict_first());
        pending |= 1u << s;
    };
    uint32_t par = 0;  // bit s: parity of the next phase of stage s
    // One step of a pass.  Thread 0 waits (bounded) for stage s to land when
    // `need`; the block barrier then releases the other threads (they wait
    // in the barrier instead of polling), orders the landed copy before their
    // reads, and certifies that every thread is done with the previous
    // step's stage, which thread 0 may then refill.  False for every thread
    // after a time-out.
    auto step = [&](int s, bool need) {
        if (tid == 0 && need) {
            if (q_mbar_wait(smem_u32(&full[s]), (par >> s) & 1u))
                pending &= ~(1u << s);
            else
                abort_sh = 1;
        }
        __syncthreads();
        if (abort_sh) return false;
        if (need) par ^= 1u << s;
        return true;
    };

    // step i of pass 1 reads piece seq(i) into stage i % stages; the
    // keep_pieces steps before the resident ones are the first that pass 2
    // reads again
    auto seq = [&](int i) { return kPass1Descending ? npieces - 1 - i : i; };
    auto kept = [&](int i) { return i < npieces - stages && i >= npieces - stages - keep_pieces; };
    float sc;
    int n_res = 0, first_res = 0;
    if constexpr (DYN) {
        // pass 1: the maximum magnitude of the block's pieces
        if (tid == 0)
            for (int i = 0; i < npieces && i < stages; ++i) issue(seq(i), i, kept(i));
        uint32_t m = 0;
        bool aborted = false;
        for (int i = 0, s = 0, sp = 0; i < npieces; ++i) {
            if (!step(s, true)) {
                aborted = true;
                break;
            }
            if (tid == 0 && i >= 1 && i - 1 + stages < npieces) issue(seq(i - 1 + stages), sp, kept(i - 1 + stages));
            const uint4 *src = stage_mem + s * piece_words;
            const int words = words_of(seq(i));
            for (int w = tid; w < words; w += 2 * kTThreads) {
                m = word_mag_max<DT>(src[w], m);
                if (w + kTThreads < words) m = word_mag_max<DT>(src[w + kTThreads], m);
            }
            sp = s;
            s = s + 1 == stages ? 0 : s + 1;
        }
        m = fold_mag<DT>(m);
        const int64_t tail = numel - n_words * EPW;
        if (blockIdx.x == 0 && tid < tail) m = max(m, scalar_mag_bits<DT>(x, n_words * EPW + tid));
        m = block_max_u32(m, red);
        if (aborted) {
            if (tid == 0) flag_timeout(status);
            goto teardown;
        }
        const unsigned pair = epoch_sh & 1u;
        uint32_t mm;
        if (!grid_max(arrive + pair, amax + pair, m, status, &mm)) return;  // no copy in flight here
        sc = scale_from_amax(mag_bits_to_float<DT>(mm));
        if (blockIdx.x == 0 && tid == 0) {
            *scale = sc;
            *epoch = epoch_sh + 1u;  // every block read the counter before arriving
        }
        first_res = npieces > stages ? npieces - stages : 0;
        n_res = npieces - first_res;
    } else {
        sc = *scale;
        if (tid == 0)
            for (int k = 0; k < npieces && k < stages; ++k) issue(k, k, false);
    }
    {
        // pass 2: cast.  Dynamic: the pieces still on chip first, then the
        // others, most recently read first; static: piece j.
        const Quot d = Quot::make<DT>(sc);
        auto piece_of = [&](int j) {
            if (!DYN) return j;
            if (j < n_res) return seq(first_res + j);
            return seq(kRecentFirst ? first_res - 1 - (j - n_res) : j - n_res);
        };
        int s = DYN ? first_res % stages : 0, sp = 0;
        for (int j = 0; j < npieces; ++j) {
            if (!step(s, j >= n_res)) {
                if (tid == 0) flag_timeout(status);
                goto teardown;
            }
            if (tid == 0 && j >= 1 && j - 1 + stages < npieces) issue(piece_of(j - 1 + stages), sp, false);
            const int k = piece_of(j);
            const uint4 *src = stage_mem + s * piece_words;
            const int words = words_of(k);
            uint8_t *qk = q + first_word(k) * EPW;
            for (int w = tid; w < words; w += 2 * kTThreads) {
                const uint4 a = src[w];
                if (w + kTThreads < words) {
                    const uint4 c = src[w + kTThreads];
                    cast_word<DT, !DYN>(a, d, qk, w);
                    cast_word<DT, !DYN>(c, d, qk, w + kTThreads);
                } else {
                    cast_word<DT, !DYN>(a, d, qk, w);
                }
            }
            sp = s;
            s = s + 1 == stages ? 0 : s + 1;
        }
        const int64_t tail = numel - n_words * EPW;
        if (blockIdx.x == 0 && tid < tail) {
            const int64_t i = n_words * EPW + tid;
            q[i] = code_of(scalar_value<DT>(x, i), sc);
        }
        return;
    }
teardown:
    // a wait gave up: let this block's copies in flight land before the
    // block's shared memory is released (again bounded)
    if (tid == 0)
        for (int i = 0; i < stages; ++i)
            if (pending & (1u << i)) q_mbar_wait(smem_u32(&full[i]), (par >> i) & 1u);
}

constexpr int kMaxDevicesQ = 64;
std::atomic<int> g_tma_ready[kMaxDevicesQ][4][2];  // dynamic shared memory raised, per device

std::atomic<int64_t> g_l2_bytes[kMaxDevicesQ];

// L2 size of the current device (0 if unknown: then nothing is kept in L2)
int64_t l2_bytes() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesQ) return 0;
    int64_t v = g_l2_bytes[dev].load(std::memory_order_acquire);
    if (v == 0) {
        int l2 = 0;
        if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0) return 0;
        v = l2;
        g_l2_bytes[dev].store(v, std::memory_order_release);
    }
    return v;
}

template <int DT, bool DYN>
bool tma_prepare() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesQ) return false;
    if (g_tma_ready[dev][DT][DYN].load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(quant_tma_kernel<DT, DYN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kStages * kPieceBytes) != cudaSuccess)
        return false;
    g_tma_ready[dev][DT][DYN].store(1, std::memory_order_release);
    return true;
}

// Pieces of X (whole 16-byte words, at most kPieceWords) dealt round-robin to
// at most one block per SM; every block gets the same number of pieces, give
// or take one, and small tensors use fewer blocks of at least kMinPieceWords.
struct TmaPlan {
    int grid, piece_words, stages, keep_pieces;
    int64_t total_pieces;
};

TmaPlan plan_tma(int64_t n_words, int sms, int64_t l2_bytes) {
    TmaPlan p;
    const int64_t per_block = (n_words + int64_t(sms) * kPieceWords - 1) / (int64_t(sms) * kPieceWords);
    int64_t pw = per_block > 0 ? (n_words + int64_t(sms) * per_block - 1) / (int64_t(sms) * per_block) : 1;
    pw = (pw + 63) / 64 * 64;  // whole kilobytes
    if (pw < kMinPieceWords) pw = kMinPieceWords;
    if (pw > kPieceWords) pw = kPieceWords;
    p.piece_words = static_cast<int>(pw);
    p.total_pieces = (n_words + pw - 1) / pw;
    p.grid = static_cast<int>(p.total_pieces < sms ? (p.total_pieces < 1 ? 1 : p.total_pieces) : sms);
    const int64_t max_pieces = (p.total_pieces + p.grid - 1) / p.grid;
    p.stages = static_cast<int>(max_pieces < kStages ? (max_pieces < 1 ? 1 : max_pieces) : kStages);
    // pieces per block held in L2 between the passes: half of L2 over the grid
    const int64_t keep = (l2_bytes / 2) / (int64_t(p.grid) * pw * 16);
    p.keep_pieces = static_cast<int>(keep < (int64_t(1) << 20) ? keep : (int64_t(1) << 20));
    return p;
}

template <int DT>
int run_tma(const void *x, int64_t numel, uint8_t *q, float *scale, bool dynamic, void *workspace,
            cudaStream_t stream, int sms) {
    const bool ready = dynamic ? tma_prepare<DT, true>() : tma_prepare<DT, false>();
    if (!ready) return FP8L_ECUDA;
    const TmaPlan p = plan_tma(numel / (16 / Elt<DT>::kBytes), sms, l2_bytes());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid), 1, 1);
    cfg.blockDim = dim3(kTThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.stages) * p.piece_words * 16;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dynamic ? 1 : 0;
    cudaError_t e;
    if (dynamic)
        e = cudaLaunchKernelEx(&cfg, quant_tma_kernel<DT, true>, x, numel, q, scale, epoch_word(workspace),
                               arrive_words(workspace), amax_words(workspace), status_word(workspace),
                               p.piece_words, static_cast<int>(p.total_pieces), p.stages, p.keep_pieces);
    else
        e = cudaLaunchKernelEx(&cfg, quant_tma_kernel<DT, false>, x, numel, q, scale,
                               static_cast<unsigned *>(nullptr), static_cast<unsigned *>(nullptr),
                               static_cast<unsigned *>(nullptr),
                               workspace ? status_word(workspace) : static_cast<unsigned *>(nullptr),
                               p.piece_words, static_cast<int>(p.total_pieces), p.stages, 0);
    if (e != cudaSuccess) return FP8L_ECUDA;
    return launch_status();
}

template <int DT>
int run_per_tensor(const void *x, int64_t numel, uint8_t *q, float *scale, bool dynamic,
                   void *workspace, cudaStream_t stream, int sms) {
    if (numel > 0) return run_tma<DT>(x, numel, q, scale, dynamic, workspace, stream, sms);
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

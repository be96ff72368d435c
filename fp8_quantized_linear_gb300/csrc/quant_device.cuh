// Device-side pieces shared by the quantizers (per-tensor, per-row, and the
// RMS normalization that feeds them): E4M3 conversion, the division-free
// correctly rounded quotient, magnitude maxima, block and grid maxima, and
// the bulk-copy (TMA) staging helpers.  Each translation unit that includes
// this header gets its own copies (anonymous namespace).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace fp8l {
namespace {

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

// bounded wait for the phase of parity `parity`; false after `limit` cycles
__device__ __forceinline__ bool q_mbar_wait(uint32_t bar, uint32_t parity, long long limit) {
    if (q_mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!q_mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return false;
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
__device__ bool grid_max(unsigned *arrive, unsigned *amax, uint32_t m, unsigned *status, uint32_t *out,
                         unsigned expect, long long limit) {
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
            if (c >= expect) break;
            if (clock64() - t0 > limit) {
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

}  // namespace
}  // namespace fp8l

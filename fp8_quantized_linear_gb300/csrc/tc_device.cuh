// Device-side pieces shared by the tcgen05 products: mbarrier waits with a
// cycle limit, TMA tile loads, tcgen05 fences, shared-memory operand
// descriptors, commits, TMEM loads, distributed shared memory access, and the
// output conversions (16-bit rounding, the division-free E4M3 quotient).
// Each translation unit that includes this header gets its own copies
// (anonymous namespace).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace fp8l {
namespace {

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Bounded wait for the phase of parity `parity`.  Gives up when another
// role raised the abort flag, or after `limit` cycles (then raises it and
// records the time-out).
// In a CTA pair (peer_abort != 0, the peer's flag as a shared::cluster
// address) a time-out raises the peer's flag too, and the wait acquires at
// cluster scope (the barrier may be completed by the peer CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                       unsigned *status, long long limit, uint32_t peer_abort = 0) {
    auto ready = [&]() { return peer_abort ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (ready()) return true;
    const long long t0 = clock64();
    for (uint32_t i = 1;; ++i) {
        if (ready()) return true;
        if ((i & 63u) == 0u) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
                *abort_flag = 1;
                if (peer_abort)
                    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
}

// The common case first: one test of the phase inline, the bounded loop only
// when it is not complete yet (keeps the MMA issue loop short).
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                               unsigned *status, long long limit,
                                               uint32_t peer_abort = 0) {
    if (peer_abort ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    return mbar_wait(bar, parity, abort_flag, status, limit, peer_abort);
}

// Bounded wait used while tearing down: ignores the abort flag.
__device__ __noinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, unsigned *status) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kDefaultWaitCycles) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format) of a K-major operand tile
// laid out by TMA with the 128-byte swizzle: 128-byte rows, 8-row groups
// 1024 bytes apart (stride byte offset), version field 1, swizzle mode 2.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) |
           (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// shared::cluster address of `local` (a shared::cta address) in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- output conversions

__device__ __forceinline__ uint32_t pack_out16(float a, float b, int out_dtype) {
    if (out_dtype == FP8L_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t out_e4m3x2(float a, float b) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// E4M3 output codes of v / output_scale.  The quotient is the correctly
// rounded RN(v / os) without a division: with y = RN(1/os), q0 = RN(v y) and
// two corrections q <- RN(q + RN(v - os q) y) (fused multiply-adds), the
// second of which is correctly rounded by Markstein's theorem (P. Markstein,
// IBM J. Res. Develop. 34(1), 1990) when the residual does not underflow and
// nothing overflows.  That holds for 2^-92 <= os <= 2^100 once |v| is
// clamped to 1024 os (every code from 464 os up saturates to 448 anyway);
// other output scales take the IEEE division.
struct OutDiv {
    float os, y, cap;
    bool fast;
    __device__ __forceinline__ static OutDiv make(float os) {
        OutDiv d;
        d.os = os;
        d.y = __frcp_rn(os);
        d.cap = 1024.0f * os;
        d.fast = os >= 0x1p-92f && os <= 0x1p100f;
        return d;
    }
    __device__ __forceinline__ float quot(float v) const {
        if (!fast) return __fdiv_rn(v, os);
        const float vc = copysignf(fminf(fabsf(v), cap), v);
        float q = __fmul_rn(vc, y);
        q = __fmaf_rn(__fmaf_rn(-os, q, vc), y, q);
        return __fmaf_rn(__fmaf_rn(-os, q, vc), y, q);
    }
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// v4 load from CTA `rank`'s shared memory at this CTA's offset `local_addr`
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t local_addr, uint32_t rank) {
    const uint32_t remote = map_to_rank(local_addr, rank);
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}

}  // namespace
}  // namespace fp8l

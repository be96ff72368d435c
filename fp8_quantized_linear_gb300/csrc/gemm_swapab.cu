// W8A8 scaled product for few tokens (M <= 128) on the tcgen05 tensor cores,
// operands swapped (sm_103a).
//
// ("[Kernel][FP8] Initial support with dynamic per-tensor scaling": the
// W8A8 product and its microbenchmark, where FP8 pays off only once the
// weights are not the whole cost; "Marlin fp8": decode batches are bound by
// reading the weights.)
//
//   y[m, n] = cast( sum_k dec(a[m,k]) dec(w[n,k]) * a_scale(m) * w_scale(n) )
//
// With a few tokens the product is a weight stream: every weight byte is
// read once and used M times.  The MMA computes the transposed tile
// D^T = W A^T: its M side (128 rows) is a block of weight rows and its N side
// the T token rows (T = M rounded up to 16, at most 128), so no MMA slot is
// spent on padding rows and the accumulator is only T TMEM columns.  Weight
// tiles come straight from HBM by TMA into shared memory and are read there
// by the tensor core; nothing decodes E4M3 on the CUDA cores.
//
// Structure (128 threads, one tile of 128 weight rows per CTA, several CTAs
// per SM so that one CTA's epilogue overlaps the others' streams):
//   warp 0 lane 0  TMA producer: the 16 KB weight block and the T x 128
//                  token block of each k-block into a ring of stages
//                  (full/empty mbarriers).  With stable weights the kernel
//                  is a programmatic dependent of the preceding kernel and
//                  issues the weight blocks of its first stages before it
//                  waits for that kernel.
//   warp 1         TMEM allocation; lane 0 issues
//                  tcgen05.mma.cta_group::1.kind::f8f6f4 (M=128, N=T, K=32),
//                  four per k-block, and commits each stage back to the
//                  producer and the finished accumulator to the epilogue.
//   all warps      epilogue: tcgen05.ld of the 128 x T accumulator into a
//                  [T][128] fp32 tile in the (idle) stage ring, then scale,
//                  cast and store four consecutive channels per thread, so a
//                  warp writes 128 consecutive outputs of one token.
// When there are fewer weight blocks than CTA slots, a cluster of `split`
// CTAs shares a tile and splits its k-blocks; each owner adds the cluster's
// fp32 partial tiles through distributed shared memory (fixed order).
// Every mbarrier wait is bounded as in the other tcgen05 products.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "quant_device.cuh"
#include "tc_device.cuh"

namespace fp8l {
namespace {

constexpr int SW_BM = 128;                 // weight rows per tile = MMA M
constexpr int SW_BK = 128;                 // k-block, bytes = swizzle span
constexpr int SW_UMMA_K = 32;
constexpr int kSwThreads = 128;
constexpr int kSwWBytes = SW_BM * SW_BK;   // 16 KB of weights per stage
constexpr int kSwMaxT = 128;               // tokens per tile at most
constexpr int kSwMaxStages = 16;
constexpr int kSwMaxSplit = 8;             // portable cluster size
constexpr int kSwPitch = SW_BM + 4;        // floats per token row of the fp32 tile
// shared memory per CTA aimed at: two CTAs per SM
constexpr int kSwSmemTarget = 112 * 1024;

struct SwapParams {
    int M, N, K;
    int T;            // MMA N: M rounded up to 16
    int stages;       // ring depth
    int stage_bytes;  // kSwWBytes + T * SW_BK
    int num_k_blocks;
    int split;        // CTAs of a cluster sharing a tile (1: no cluster)
    int prefetch;     // stable weights: weight blocks issued before griddepcontrol.wait
    int x_stages;     // fused quantization: stages of the 16-bit token ring
    const float *a_scale;
    const float *w_scale;
    int w_per_channel;
    int a_per_token;
    const float *out_scale;
    void *y;
    int out_dtype;
    unsigned *status;
    long long wait_cycles;
    unsigned stall;
};

__device__ __forceinline__ void mma_f8_n(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_shared_v4u(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Coherent scalar load that stays after griddepcontrol.wait (the scales may
// be written by the preceding kernel on the stream).
__device__ __forceinline__ float ld_f32(const float *p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kSwThreads, 1)
gemm_f8_swapab(const __grid_constant__ CUtensorMap tmap_w,
               const __grid_constant__ CUtensorMap tmap_a, const SwapParams p) {
    // all CTAs have started: the next kernel on the stream may be scheduled
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
    uint8_t *gbase = smem_raw + (sbase - raw);
    const int S = p.stages;
    const uint32_t ring_bytes = static_cast<uint32_t>(S * p.stage_bytes);
    const uint32_t bar0 = sbase + ring_bytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * S);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + ring_bytes + (2 * S + 1) * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t tmem_cols = p.T <= 32 ? 32u : (p.T <= 64 ? 64u : 128u);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = p.split;
    const int rank = split > 1 ? static_cast<int>(blockIdx.x) % split : 0;
    const int tile = static_cast<int>(blockIdx.x) / split;
    const int base = p.num_k_blocks / split, rem = p.num_k_blocks % split;
    const int kb_begin = rank * base + (rank < rem ? rank : rem);
    const int nkb = base + (rank < rem ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
            const int w_row = tile * SW_BM;
            const uint32_t sb = static_cast<uint32_t>(p.stage_bytes);
            // stable weights: the first stages' weight blocks before the wait
            const int pre = p.prefetch ? (nkb < S ? nkb : S) : 0;
            for (int i = 0; i < pre; ++i) {
                const uint32_t st = sbase + i * sb;
                mbar_expect_tx(full_bar(i), sb);
                tma_load_2d(st, &tmap_w, (kb_begin + i) * SW_BK, w_row, full_bar(i));
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int i = 0; i < pre; ++i)
                tma_load_2d(sbase + i * sb + kSwWBytes, &tmap_a, (kb_begin + i) * SW_BK, 0, full_bar(i));
            uint32_t issued = (1u << pre) - 1u;  // stages with a load in flight (parity 0 so far)
            uint32_t issued_parity = 0;
            int stage = pre == S ? 0 : pre;
            uint32_t phase = pre == S ? 1u : 0u;
            for (int i = pre; i < nkb; ++i) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_cycles)) break;
                const uint32_t st = sbase + stage * sb;
                const int kx = (kb_begin + i) * SW_BK;
                mbar_expect_tx(full_bar(stage), sb);
                tma_load_2d(st, &tmap_w, kx, w_row, full_bar(stage));
                tma_load_2d(st + kSwWBytes, &tmap_a, kx, 0, full_bar(stage));
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // every load this thread issued lands before the CTA exits
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s)) mbar_wait_drain(full_bar(s), (issued_parity >> s) & 1u, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // kind::f8f6f4, D f32, A and B E4M3 K-major, N = T, M = 128
            const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(p.T >> 3) << 17) |
                                   (static_cast<uint32_t>(SW_BM >> 4) << 24);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            if (p.stall & kStallMma) ok = mbar_wait(done_bar, 0, abort_flag, p.status, p.wait_cycles);
            for (int i = 0; ok && i < nkb; ++i) {
                if (!mbar_wait_fast(full_bar(stage), phase, abort_flag, p.status, p.wait_cycles)) break;
                tc_fence_after();
                const uint32_t st = sbase + stage * static_cast<uint32_t>(p.stage_bytes);
                const uint64_t dw = sw128_desc(st), da = sw128_desc(st + kSwWBytes);
#pragma unroll
                for (int k = 0; k < SW_BK / SW_UMMA_K; ++k)
                    mma_f8_n(tmem_base, dw + 2 * k, da + 2 * k, idesc, (i | k) != 0 ? 1u : 0u);
                mma_commit(empty_bar(stage));
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // the accumulator is complete (or abandoned) once these retire
            mma_commit(done_bar);
        }
        __syncwarp();
    }

    // ---- epilogue: every thread
    asm volatile("griddepcontrol.wait;" ::: "memory");
    bool ok = mbar_wait(done_bar, 0, abort_flag, p.status, p.wait_cycles);
    tc_fence_after();
    // accumulator row (weight row) 32*warp + lane, token columns 0..T-1,
    // into part[t][row] at the start of the ring
    const int row = warp * 32 + lane;
    if (ok && !*abort_flag) {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
        for (int c = 0; c < p.T; c += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + static_cast<uint32_t>(c), r);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                st_shared_f32(sbase + static_cast<uint32_t>(((c + j) * kSwPitch + row) * 4), r[j]);
        }
    }
    tc_fence_before();
    if (split > 1)
        cluster_sync_all();
    else
        __syncthreads();

    // owner work: items (token t, channel group of 4) of this tile, split
    // evenly over the cluster's CTAs; consecutive threads on consecutive
    // channel groups
    ok = !*abort_flag;
    const int items = p.M * (SW_BM / 4);
    const int i0 = static_cast<int>((static_cast<long long>(items) * rank) / split);
    const int i1 = static_cast<int>((static_cast<long long>(items) * (rank + 1)) / split);
    const float sa0 = ld_f32(p.a_scale);
    const float sw0 = ld_f32(p.w_scale);
    const OutDiv od = OutDiv::make(p.out_dtype == FP8L_E4M3 ? ld_f32(p.out_scale) : 1.0f);
    for (int i = i0 + static_cast<int>(threadIdx.x); ok && i < i1; i += kSwThreads) {
        const int t = i >> 5;
        const int c4 = (i & 31) * 4;
        const int n = tile * SW_BM + c4;
        if (n >= p.N) continue;  // N % 16 == 0: a group is all in or all out
        const uint32_t off = sbase + static_cast<uint32_t>((t * kSwPitch + c4) * 4);
        float4 acc;
        if (split == 1) {
            acc = ld_shared_v4(off);
        } else {
            float4 part[kSwMaxSplit];
#pragma unroll
            for (int q = 0; q < kSwMaxSplit; ++q)
                if (q < split) part[q] = ld_cluster_v4(off, static_cast<uint32_t>(q));
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < kSwMaxSplit; ++q) {  // the same order in every run
                if (q < split) {
                    acc.x += part[q].x;
                    acc.y += part[q].y;
                    acc.z += part[q].z;
                    acc.w += part[q].w;
                }
            }
        }
        const float sa = p.a_per_token ? ld_f32(p.a_scale + t) : sa0;
        float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] *= sa * (p.w_per_channel ? ld_f32(p.w_scale + n + j) : sw0);
        const size_t o = static_cast<size_t>(t) * p.N + n;
        if (p.out_dtype == FP8L_E4M3) {
            const uint32_t lo = out_e4m3x2(od.quot(v[0]), od.quot(v[1]));
            const uint32_t hi = out_e4m3x2(od.quot(v[2]), od.quot(v[3]));
            *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(p.y) + o) = lo | (hi << 16);
        } else {
            *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.y) + o) =
                make_uint2(pack_out16(v[0], v[1], p.out_dtype), pack_out16(v[2], v[3], p.out_dtype));
        }
    }
    if (split > 1) cluster_sync_all();  // peers may still be reading this CTA's partials

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(tmem_cols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- with the quantization fused
//
// The same product with the activations' E4M3 codes made inside the kernel
// from 16-bit x ("Condition to achieve linear speedup?": activation
// quantization fused into another kernel; "RFC: FP8 Quantization Schema in
// vLLM": static input scales), so no quantizer launch precedes it:
//   static scale    a_scale given; each CTA quantizes only the token
//                   columns of its own k-blocks;
//   dynamic scale   every CTA first takes the magnitude maximum of the whole
//                   x (a few to a few tens of KB for a few tokens; read from
//                   L2) and derives the same scale = amax / 448; CTA 0 stores
//                   it in a_scale.
// The codes are those of the quantizer bit for bit (the same division-free
// quotient and E4M3 conversion), so the result equals quantizer + product.
//   warp 0      lane 0: weight stages (as above).
//   warp 1      TMEM; lane 0 issues the MMAs once a stage's weights have
//               landed and its token codes are written.
//   warps 2-3   converters: the codes of the M token rows of each k-block,
//               16 per thread and step, into the stage's swizzled B tile
//               (rows M .. T-1 stay zero), then a proxy fence.
//   warp 4      lane 0: the tokens' 16-bit k-blocks (two M x 64 boxes:
//               only the real token rows) into a ring of up to 16 stages
//               (24 KB).
// Every weight stage and token stage has one consumer in k-block order (no
// barrier can be waited on two phases ahead).
// Token ring: kSqXRingBytes, 2 to kSqMaxXStages stages (with two stages a
// CTA streaming 32 k-blocks waited on its token loads: 34 us against 25 us
// for quantizer + product at M = 1, N = 28672; at 16 tokens 4 weight and 6
// token stages beat 5 and 5).  Weight ring: the rest of kSqSmemTarget, two
// CTAs per SM (233472 bytes of shared memory per SM, 1024 reserved per CTA,
// 512 left for the kernel's static shared variables: a CTA 20 bytes over
// the limit ran one per SM and took 1.7x as long).  Above 64 tokens the
// rings take the shared memory past two CTAs per SM: one CTA per SM then,
// up to kSqSmemMax.
constexpr int kSqMaxXStages = 16;
constexpr int kSqMinXStagesTrade = 8;
constexpr size_t kSqXRingBytes = 24 * 1024;
constexpr size_t kSqSmemTarget = 233472 / 2 - 1024 - 512;
constexpr size_t kSqSmemMax = 220 * 1024;
constexpr int kSqConvThreads = 64;
// warp 4 loads the tokens: in lane 1 of the weight producer's warp its
// spin-waits and the weight producer's took turns (N = 28672 at M = 1:
// 32 us against 25 us for quantizer + product)
constexpr int kSqThreads = 160;

template <int XDT>
__global__ void __launch_bounds__(kSqThreads, 1)
gemm_f8_swapab_q(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                 const SwapParams p, float *a_scale_out, int dynamic, const void *x_raw) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw);
    const int S = p.stages, SX = p.x_stages;
    const uint32_t sb = static_cast<uint32_t>(p.stage_bytes);   // 16 KB of weights + T x 128 codes
    const uint32_t xsb = static_cast<uint32_t>(p.M) * 256u;      // M rows x 128 16-bit values
    const uint32_t xbase = sbase + static_cast<uint32_t>(S) * sb;
    const uint32_t ring_bytes = static_cast<uint32_t>(S) * sb + static_cast<uint32_t>(SX) * xsb;
    const uint32_t bar0 = (sbase + ring_bytes + 7u) & ~7u;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto bready_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    auto xfull_bar = [&](int s) { return bar0 + 8u * (3 * S + s); };
    auto xempty_bar = [&](int s) { return bar0 + 8u * (3 * S + SX + s); };
    const uint32_t done_bar = bar0 + 8u * (3 * S + 2 * SX);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + (bar0 - sbase) + (3 * S + 2 * SX + 1) * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ uint32_t red[33];
    const uint32_t tmem_cols = p.T <= 32 ? 32u : (p.T <= 64 ? 64u : 128u);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = p.split;
    const int rank = split > 1 ? static_cast<int>(blockIdx.x) % split : 0;
    const int tile = static_cast<int>(blockIdx.x) / split;
    const int base = p.num_k_blocks / split, rem = p.num_k_blocks % split;
    const int kb_begin = rank * base + (rank < rem ? rank : rem);
    const int nkb = base + (rank < rem ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(bready_bar(s), kSqConvThreads);
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(xfull_bar(s), 1);
            mbar_init(xempty_bar(s), kSqConvThreads);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // stable weights: the first stages' weight blocks before the wait
    const int pre = p.prefetch ? (nkb < S ? nkb : S) : 0;
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
        for (int i = 0; i < pre; ++i) {
            mbar_expect_tx(full_bar(i), kSwWBytes);
            tma_load_2d(sbase + i * sb, &tmap_w, (kb_begin + i) * SW_BK, tile * SW_BM, full_bar(i));
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // the activation scale: given, or the dynamic one from the whole of x
    float sa;
    if (dynamic) {
        const uint4 *xv = static_cast<const uint4 *>(x_raw);
        const int64_t words = static_cast<int64_t>(p.M) * p.K / 8;  // 8 16-bit values per word
        // eight loads in flight per thread before any is used: a few tens of
        // KB are then read in one or two L2 round trips
        uint32_t m = 0;
        for (int64_t w0 = threadIdx.x; w0 < words; w0 += 8 * kSqThreads) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t w = w0 + static_cast<int64_t>(u) * kSqThreads;
                v[u] = make_uint4(0, 0, 0, 0);
                if (w < words)
                    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                                 : "l"(xv + w));
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) m = word_mag_max<XDT>(v[u], m);
        }
        m = block_max_u32(fold_mag<XDT>(m), red);
        sa = scale_from_amax(mag_bits_to_float<XDT>(m));
        if (blockIdx.x == 0 && threadIdx.x == 0) *a_scale_out = sa;
    } else {
        sa = ld_f32(a_scale_out);
    }

    if (warp == 0) {
        if (lane == 0) {
            const int w_row = tile * SW_BM;
            uint32_t issued = (1u << pre) - 1u;
            uint32_t issued_parity = 0;
            int stage = pre == S ? 0 : pre;
            uint32_t phase = pre == S ? 1u : 0u;
            for (int i = pre; i < nkb; ++i) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_cycles)) break;
                mbar_expect_tx(full_bar(stage), kSwWBytes);
                tma_load_2d(sbase + stage * sb, &tmap_w, (kb_begin + i) * SW_BK, w_row, full_bar(stage));
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s)) mbar_wait_drain(full_bar(s), (issued_parity >> s) & 1u, p.status);
        }
        __syncwarp();
    } else if (warp == 4) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            for (int i = 0; i < nkb; ++i) {
                if (!mbar_wait(xempty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_cycles)) break;
                const uint32_t dst = xbase + static_cast<uint32_t>(stage) * xsb;
                const int kx = (kb_begin + i) * SW_BK;
                mbar_expect_tx(xfull_bar(stage), xsb);
                tma_load_2d(dst, &tmap_x, kx, 0, xfull_bar(stage));
                tma_load_2d(dst + xsb / 2, &tmap_x, kx + 64, 0, xfull_bar(stage));
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == SX) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            for (int s = 0; s < SX; ++s)
                if (issued & (1u << s)) mbar_wait_drain(xfull_bar(s), (issued_parity >> s) & 1u, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(p.T >> 3) << 17) |
                                   (static_cast<uint32_t>(SW_BM >> 4) << 24);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            if (p.stall & kStallMma) ok = mbar_wait(done_bar, 0, abort_flag, p.status, p.wait_cycles);
            for (int i = 0; ok && i < nkb; ++i) {
                if (!mbar_wait_fast(full_bar(stage), phase, abort_flag, p.status, p.wait_cycles) ||
                    !mbar_wait_fast(bready_bar(stage), phase, abort_flag, p.status, p.wait_cycles))
                    break;
                tc_fence_after();
                const uint32_t st = sbase + stage * sb;
                const uint64_t dw = sw128_desc(st), da = sw128_desc(st + kSwWBytes);
#pragma unroll
                for (int k = 0; k < SW_BK / SW_UMMA_K; ++k)
                    mma_f8_n(tmem_base, dw + 2 * k, da + 2 * k, idesc, (i | k) != 0 ? 1u : 0u);
                mma_commit(empty_bar(stage));
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            mma_commit(done_bar);
        }
        __syncwarp();
    } else {
        // converters: rows M .. T-1 of every stage's code tile are zero once
        const int ct = static_cast<int>(threadIdx.x) - 64;
        for (int s = 0; s < S; ++s)
            for (int o = ct * 16 + p.M * 128; o < p.T * 128; o += kSqConvThreads * 16)
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sbase + s * sb + kSwWBytes +
                                                                             static_cast<uint32_t>(o)),
                             "r"(0u)
                             : "memory");
        const Quot d = Quot::make<XDT>(sa);
        int stage = 0, xs = 0;
        uint32_t phase = 0, xphase = 0;
        for (int i = 0; i < nkb; ++i) {
            // the token block has landed, and the stage's code tile is free
            // (the MMAs of its previous round have retired)
            if (!mbar_wait(xfull_bar(xs), xphase, abort_flag, p.status, p.wait_cycles) ||
                !mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_cycles))
                break;
            const uint32_t xst = xbase + static_cast<uint32_t>(xs) * xsb;
            const uint32_t bst = sbase + stage * sb + kSwWBytes;
            // task (row r, 16-code piece j): x values 16 j .. 16 j + 15 of row r
            for (int task = ct; task < p.M * 8; task += kSqConvThreads) {
                const int r = task >> 3, j = task & 7;
                // the stage holds two M x 64 boxes (k 0-63, 64-127) of 128-byte rows
                const uint32_t src = xst + static_cast<uint32_t>((j >> 2) * (xsb / 2) + r * 128 + (j & 3) * 32);
                const uint4 v0 = ld_shared_v4u(src), v1 = ld_shared_v4u(src + 16);
                const uint2 c0 = dynamic ? codes_of_word<XDT, false>(v0, d) : codes_of_word<XDT, true>(v0, d);
                const uint2 c1 = dynamic ? codes_of_word<XDT, false>(v1, d) : codes_of_word<XDT, true>(v1, d);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 bst + static_cast<uint32_t>(r * 128 + ((j ^ (r & 7)) * 16))),
                             "r"(c0.x), "r"(c0.y), "r"(c1.x), "r"(c1.y)
                             : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // codes visible to the MMAs
            mbar_arrive(bready_bar(stage));
            mbar_arrive(xempty_bar(xs));
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
            if (++xs == SX) {
                xs = 0;
                xphase ^= 1u;
            }
        }
    }

    // ---- epilogue (as in gemm_f8_swapab, with this CTA's own scale;
    // warps 0-3 own the TMEM lane quarters)
    const bool done_ok = mbar_wait(done_bar, 0, abort_flag, p.status, p.wait_cycles);
    tc_fence_after();
    const int row = warp * 32 + lane;
    if (warp < 4 && done_ok && !*abort_flag) {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
        for (int c = 0; c < p.T; c += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + static_cast<uint32_t>(c), r);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                st_shared_f32(sbase + static_cast<uint32_t>(((c + j) * kSwPitch + row) * 4), r[j]);
        }
    }
    tc_fence_before();
    if (split > 1)
        cluster_sync_all();
    else
        __syncthreads();
    const bool ok = !*abort_flag;
    const int items = p.M * (SW_BM / 4);
    const int i0 = static_cast<int>((static_cast<long long>(items) * rank) / split);
    const int i1 = static_cast<int>((static_cast<long long>(items) * (rank + 1)) / split);
    const float sw0 = ld_f32(p.w_scale);
    const OutDiv od = OutDiv::make(p.out_dtype == FP8L_E4M3 ? ld_f32(p.out_scale) : 1.0f);
    for (int i = i0 + static_cast<int>(threadIdx.x); ok && i < i1; i += kSqThreads) {
        const int t = i >> 5;
        const int c4 = (i & 31) * 4;
        const int n = tile * SW_BM + c4;
        if (n >= p.N) continue;
        const uint32_t off = sbase + static_cast<uint32_t>((t * kSwPitch + c4) * 4);
        float4 acc;
        if (split == 1) {
            acc = ld_shared_v4(off);
        } else {
            float4 part[kSwMaxSplit];
#pragma unroll
            for (int q = 0; q < kSwMaxSplit; ++q)
                if (q < split) part[q] = ld_cluster_v4(off, static_cast<uint32_t>(q));
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < kSwMaxSplit; ++q) {  // the same order in every run
                if (q < split) {
                    acc.x += part[q].x;
                    acc.y += part[q].y;
                    acc.z += part[q].z;
                    acc.w += part[q].w;
                }
            }
        }
        float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] *= sa * (p.w_per_channel ? ld_f32(p.w_scale + n + j) : sw0);
        const size_t o = static_cast<size_t>(t) * p.N + n;
        if (p.out_dtype == FP8L_E4M3) {
            const uint32_t lo = out_e4m3x2(od.quot(v[0]), od.quot(v[1]));
            const uint32_t hi = out_e4m3x2(od.quot(v[2]), od.quot(v[3]));
            *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(p.y) + o) = lo | (hi << 16);
        } else {
            *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.y) + o) =
                make_uint2(pack_out16(v[0], v[1], p.out_dtype), pack_out16(v[2], v[3], p.out_dtype));
        }
    }
    if (split > 1) cluster_sync_all();

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(tmem_cols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- W8A16 on tcgen05
//
// ("Marlin fp8": weight-only FP8 for decode; 16-bit activations, E4M3
// weights with per-channel scales.)
//
//   y[m, n] = w_scale[n] * sum_k x[m,k] dec(w[n,k])   (fp32 accumulation,
//             rounded to nearest in x's type)
//
// The same swapped operands as above, with kind::f16 MMAs: A and B of one
// MMA have one 16-bit type, so the E4M3 weights are widened to the
// activations' type first.  That is exact (every E4M3 value is a normal f16
// or zero, and its 3-bit significand fits bf16's 7), done by converter
// warps, and the widened weights go to TMEM as the MMA's A operand; the
// tokens are the B operand in shared memory.
//   warp 0         weight producer: per 128-element k-block the raw 128 x
//                  128-byte block (rows of the [N, K] matrix with the
//                  128-byte swizzle, or 8 groups x 2 chunks of the packed
//                  layout read as 2 KB runs).
//   warp 10        token producer: two T x 64 blocks (128-byte swizzle) per
//                  k-block.
//   warp 1         TMEM (256 columns: two 64-column A buffers, then the
//                  T <= 64 accumulator columns); lane 0 issues
//                  tcgen05.mma.cta_group::1.kind::f16 [d], [a], b (M = 128,
//                  N = T, K = 16), eight per k-block.
//   warps 2-9      two converter warpgroups taking alternate k-blocks, lane
//                  = weight row (warp w owns TMEM lanes 32 (w mod 4) ..):
//                  the row's 128 bytes from shared memory (laid out or read
//                  so that a wavefront has no bank conflicts), release of
//                  the weight stage, cvt e4m3x2 -> f16x2 (bf16 by exponent
//                  rebasing), two tcgen05.st of 32 columns into the free A
//                  buffer; then the first group moves the accumulator to the
//                  fp32 tile for the owner loop.
// Weights and tokens have separate rings, so a weight stage is free as soon
// as its converters have read it (the tokens' stage waits for the MMAs).
// Measured (graph replay over rotating copies): 0.40-0.50 of HBM whatever
// the token count, against 0.45-0.82 for the CUDA-core kernel up to 16
// tokens and 0.15-0.33 for it at 32-64, so the automatic choice takes this
// kernel from 17 to 64 tokens.  Neither twice the converter warps, six A
// buffers, conflict-free shared-memory reads, more weight stages, nor one
// barrier operation per warp instead of per thread moved it; with the TMEM
// stores and the MMAs both removed (a timing copy) the rest of the pipeline
// reached 0.6.
constexpr int W16_BK = 128;                    // k-block, elements
constexpr int W16_UMMA_K = 16;                 // K of one kind::f16 MMA
constexpr int kW16Groups = 2;                  // converter warpgroups, alternate k-blocks
constexpr int kW16XWarp = 2 + 4 * kW16Groups;  // the token producer's own warp
constexpr int kW16Threads = 32 * (kW16XWarp + 1);
constexpr int kW16WBytes = SW_BM * W16_BK;     // 16 KB of E4M3 weights per stage
constexpr int kW16MaxT = 64;
constexpr int kW16ABufCols = W16_BK / 2;       // two 16-bit values per TMEM column
// One A buffer per converter group, and a weight ring whose stage count is a
// multiple of the groups: every stage and buffer then always has the same
// consumer, so no waiter can run two phases ahead of a barrier and mistake
// an older completion of the same parity for the one it waits for (with
// five stages for two groups, consecutive rounds of a stage alternated
// between the groups and that happened).
constexpr int kW16ABufs = kW16Groups;
constexpr int kW16DCol = kW16ABufs * kW16ABufCols;  // accumulator after the A buffers
constexpr uint32_t kW16TmemCols = 256;
constexpr int kW16ConvThreads = 128;
constexpr int kW16MaxWStages = 8;
static_assert(kW16MaxWStages % kW16Groups == 0, "weight stages are dealt to the converter groups");

struct W16Params {
    int M, N, K;
    int T, w_stages, x_stages, x_stage_bytes, num_k_blocks, split, prefetch, packed;
    const float *w_scale;
    void *y;
    unsigned *status;
    long long wait_cycles;
    unsigned stall;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// D (TMEM) += A (TMEM) * B (shared memory descriptor), kind::f16
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Two E4M3 codes (low byte first) to the f16 pair of the same values (the
// hardware conversion; exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    uint32_t r;
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
        : "=r"(r)
        : "r"(two_codes));
    return r;
}

// An f16 pair holding E4M3 values to the bf16 pair of the same values: a
// nonzero E4M3 value is a normal f16 whose significand's low 7 bits are
// zero, so its bf16 bits are the magnitude shifted right by 3 with the
// exponent rebased from bias 15 to 127 (+112 << 7); zero stays zero.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_e4m3(uint32_t h) {
    const uint32_t mag = h & 0x7FFF7FFFu;
    const uint32_t rebased = ((mag >> 3) & 0x0FFF0FFFu) + 0x38003800u;
    return (rebased & __vcmpne2(mag, 0u)) | (h & 0x80008000u);
}

// 16 E4M3 codes to 8 words of 16-bit pairs of x's type
template <int XDT>
__device__ __forceinline__ void widen_codes16(const uint4 &u, uint32_t *h) {
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        uint32_t lo = e4m3x2_to_f16x2(w4[e] & 0xFFFFu);
        uint32_t hi = e4m3x2_to_f16x2(w4[e] >> 16);
        if (XDT == FP8L_BF16) {
            lo = f16x2_to_bf16x2_e4m3(lo);
            hi = f16x2_to_bf16x2_e4m3(hi);
        }
        h[2 * e] = lo;
        h[2 * e + 1] = hi;
    }
}

template <int XDT>
__global__ void __launch_bounds__(kW16Threads, 2)
gemm_w8a16_tc(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
              const W16Params p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw);
    const int SW = p.w_stages, SX = p.x_stages;
    const uint32_t xsb = static_cast<uint32_t>(p.x_stage_bytes);
    const uint32_t xbase = sbase + static_cast<uint32_t>(SW) * kW16WBytes;  // token ring after the weights
    const uint32_t ring_bytes = static_cast<uint32_t>(SW) * kW16WBytes + static_cast<uint32_t>(SX) * xsb;
    const uint32_t bar0 = sbase + ring_bytes;
    auto wfull_bar = [&](int s) { return bar0 + 8u * s; };
    auto wempty_bar = [&](int s) { return bar0 + 8u * (SW + s); };
    auto xfull_bar = [&](int s) { return bar0 + 8u * (2 * SW + s); };
    auto xempty_bar = [&](int s) { return bar0 + 8u * (2 * SW + SX + s); };
    auto afull_bar = [&](int b) { return bar0 + 8u * (2 * SW + 2 * SX + b); };
    auto aempty_bar = [&](int b) { return bar0 + 8u * (2 * SW + 2 * SX + kW16ABufs + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * SW + 2 * SX + 2 * kW16ABufs);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(
        gbase + ring_bytes + (2 * SW + 2 * SX + 2 * kW16ABufs + 1) * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = p.split;
    const int rank = split > 1 ? static_cast<int>(blockIdx.x) % split : 0;
    const int tile = static_cast<int>(blockIdx.x) / split;
    const int base = p.num_k_blocks / split, rem = p.num_k_blocks % split;
    const int kb_begin = rank * base + (rank < rem ? rank : rem);
    const int nkb = base + (rank < rem ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SW; ++s) {
            mbar_init(wfull_bar(s), 1);
            mbar_init(wempty_bar(s), kW16ConvThreads);
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(xfull_bar(s), 1);
            mbar_init(xempty_bar(s), 1);
        }
        for (int b = 0; b < kW16ABufs; ++b) {
            mbar_init(afull_bar(b), kW16ConvThreads);
            mbar_init(aempty_bar(b), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kW16TmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // weights: stable (no wait for the preceding kernel)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
            if (!p.prefetch) asm volatile("griddepcontrol.wait;" ::: "memory");
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            for (int i = 0; i < nkb; ++i) {
                if (!mbar_wait(wempty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_cycles)) break;
                const uint32_t dst = sbase + static_cast<uint32_t>(stage) * kW16WBytes;
                const int kb = kb_begin + i;
                mbar_expect_tx(wfull_bar(stage), kW16WBytes);
                if (p.packed)  // 128 u64 (1 KB: 16 rows x 64 bytes) x 2 chunks x 8 groups
                    tma_load_3d(dst, &tmap_w, 0, 2 * kb, tile * (SW_BM / 16), wfull_bar(stage));
                else
                    tma_load_2d(dst, &tmap_w, kb * W16_BK, tile * SW_BM, wfull_bar(stage));
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == SW) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            for (int s = 0; s < SW; ++s)
                if (issued & (1u << s)) mbar_wait_drain(wfull_bar(s), (issued_parity >> s) & 1u, p.status);
        }
        __syncwarp();
    } else if (warp == kW16XWarp) {
        if (lane == 0) {
            // tokens: written by the preceding kernel
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
            asm volatile("griddepcontrol.wait;" ::: "memory");
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            for (int i = 0; i < nkb; ++i) {
                if (!mbar_wait(xempty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_cycles)) break;
                const uint32_t dst = xbase + static_cast<uint32_t>(stage) * xsb;
                const int kx = (kb_begin + i) * W16_BK;
                mbar_expect_tx(xfull_bar(stage), xsb);
                tma_load_2d(dst, &tmap_x, kx, 0, xfull_bar(stage));
                tma_load_2d(dst + xsb / 2, &tmap_x, kx + 64, 0, xfull_bar(stage));
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == SX) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            for (int s = 0; s < SX; ++s)
                if (issued & (1u << s)) mbar_wait_drain(xfull_bar(s), (issued_parity >> s) & 1u, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // kind::f16: D f32; A and B f16 (0) or bf16 (1), K-major; N = T, M = 128
            const uint32_t fmt = XDT == FP8L_BF16 ? 1u : 0u;
            const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) |
                                   (static_cast<uint32_t>(p.T >> 3) << 17) |
                                   (static_cast<uint32_t>(SW_BM >> 4) << 24);
            int xs = 0, buf = 0;
            uint32_t xphase = 0, aphase = 0;
            bool ok = true;
            if (p.stall & kStallMma) ok = mbar_wait(done_bar, 0, abort_flag, p.status, p.wait_cycles);
            for (int i = 0; ok && i < nkb; ++i) {
                if (!mbar_wait_fast(xfull_bar(xs), xphase, abort_flag, p.status, p.wait_cycles) ||
                    !mbar_wait_fast(afull_bar(buf), aphase, abort_flag, p.status, p.wait_cycles))
                    break;
                tc_fence_after();
                const uint32_t xst = xbase + static_cast<uint32_t>(xs) * xsb;
                const uint64_t dx0 = sw128_desc(xst), dx1 = sw128_desc(xst + xsb / 2);
                const uint32_t a0 = tmem_base + static_cast<uint32_t>(buf * kW16ABufCols);
#pragma unroll
                for (int k = 0; k < W16_BK / W16_UMMA_K; ++k)
                    mma_f16_ta(tmem_base + kW16DCol, a0 + 8u * k, (k < 4 ? dx0 : dx1) + 2 * (k & 3), idesc,
                               (i | k) != 0 ? 1u : 0u);
                mma_commit(aempty_bar(buf));  // A buffer free once these MMAs retire
                mma_commit(xempty_bar(xs));   // and the stage's tokens
                if (++xs == SX) {
                    xs = 0;
                    xphase ^= 1u;
                }
                if (++buf == kW16ABufs) {
                    buf = 0;
                    aphase ^= 1u;
                }
            }
            mma_commit(done_bar);
        }
        __syncwarp();
    } else {
        // converters: this thread's weight row, TMEM lane quarter of the warp;
        // group g takes the k-blocks g, g + kW16Groups, ...
        const int q = warp & 3;
        const int grp = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        // 16-byte piece j of the row (k = 16j ..) in the stage.  Row-major:
        // 128-byte rows written with the 128-byte swizzle, piece j of row r
        // at r * 128 + 16 (j ^ (r mod 8)): the eight lanes of one shared-
        // memory wavefront (rows r .. r+7) then hit different banks.  Packed:
        // 1 KB blocks [group][chunk] of 16 rows x 64 bytes, piece j of row r
        // at (r / 16) * 2048 + (j / 4) * 1024 + (r mod 16) * 64 + 16 (j mod 4);
        // lanes read the four pieces of a chunk in the order
        // (jj + rot) mod 4, rot = (r / 2) mod 4, for the same reason.
        const bool packed = p.packed != 0;
        const uint32_t row_off = packed ? static_cast<uint32_t>((row >> 4) * 2048 + (row & 15) * 64)
                                        : static_cast<uint32_t>(row * W16_BK);
        const int rot = packed ? ((row >> 1) & 3) : 0;
        int stage = grp, buf = grp;
        uint32_t phase = 0, aphase = 0;
        for (int i = grp; i < nkb; i += kW16Groups) {
            if (!mbar_wait(wfull_bar(stage), phase, abort_flag, p.status, p.wait_cycles)) break;
            const uint32_t wrow = sbase + static_cast<uint32_t>(stage) * kW16WBytes + row_off;
            uint4 v[8];
            if (packed) {
                // v[4 h + c'] = piece 4 h + (c' + rot) mod 4
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    v[jj] = ld_shared_u4(wrow + static_cast<uint32_t>((jj >> 2) * 1024 + (((jj & 3) + rot) & 3) * 16));
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    v[j] = ld_shared_u4(wrow + static_cast<uint32_t>((j ^ (row & 7)) * 16));
            }
            mbar_arrive(wempty_bar(stage));  // this row's weights are in registers
            // the buffer's previous k-block must be through the MMAs before it
            // is overwritten (the loads above overlap that wait)
            if (!mbar_wait(aempty_bar(buf), aphase ^ 1u, abort_flag, p.status, p.wait_cycles)) break;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t h[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 u = v[4 * half + c];
                    if (packed) {
                        // piece 4 half + c was loaded as v[4 half + (c - rot) mod 4]
                        const int src = (c - rot) & 3;
                        u = v[4 * half];
                        u = src == 1 ? v[4 * half + 1] : u;
                        u = src == 2 ? v[4 * half + 2] : u;
                        u = src == 3 ? v[4 * half + 3] : u;
                    }
                    widen_codes16<XDT>(u, h + 8 * c);
                }
                tmem_st32(tmem_base + lane_addr + static_cast<uint32_t>(buf * kW16ABufCols + 32 * half), h);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            mbar_arrive(afull_bar(buf));
            stage += kW16Groups;  // SW is a multiple of kW16Groups
            if (stage >= SW) {
                stage -= SW;
                phase ^= 1u;
            }
            aphase ^= 1u;  // kW16ABufs == kW16Groups: this group's buffer, next round
        }
    }

    // ---- epilogue: every thread joins the barriers; the first converter
    // group (which owns every TMEM lane quarter) moves the accumulator
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const bool done_ok = mbar_wait(done_bar, 0, abort_flag, p.status, p.wait_cycles);
    tc_fence_after();
    if (warp >= 2 && warp < 6 && done_ok && !*abort_flag) {
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kW16DCol;
        for (int c = 0; c < p.T; c += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + static_cast<uint32_t>(c), r);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                st_shared_f32(sbase + static_cast<uint32_t>(((c + j) * kSwPitch + row) * 4), r[j]);
        }
    }
    tc_fence_before();
    if (split > 1)
        cluster_sync_all();
    else
        __syncthreads();
    const bool ok = !*abort_flag;
    const int items = p.M * (SW_BM / 4);
    const int i0 = static_cast<int>((static_cast<long long>(items) * rank) / split);
    const int i1 = static_cast<int>((static_cast<long long>(items) * (rank + 1)) / split);
    for (int i = i0 + static_cast<int>(threadIdx.x); ok && i < i1; i += kW16Threads) {
        const int t = i >> 5;
        const int c4 = (i & 31) * 4;
        const int n = tile * SW_BM + c4;
        if (n >= p.N) continue;
        const uint32_t off = sbase + static_cast<uint32_t>((t * kSwPitch + c4) * 4);
        float4 acc;
        if (split == 1) {
            acc = ld_shared_v4(off);
        } else {
            float4 part[kSwMaxSplit];
#pragma unroll
            for (int qq = 0; qq < kSwMaxSplit; ++qq)
                if (qq < split) part[qq] = ld_cluster_v4(off, static_cast<uint32_t>(qq));
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int qq = 0; qq < kSwMaxSplit; ++qq) {  // the same order in every run
                if (qq < split) {
                    acc.x += part[qq].x;
                    acc.y += part[qq].y;
                    acc.z += part[qq].z;
                    acc.w += part[qq].w;
                }
            }
        }
        const float v0 = acc.x * ld_f32(p.w_scale + n), v1 = acc.y * ld_f32(p.w_scale + n + 1);
        const float v2 = acc.z * ld_f32(p.w_scale + n + 2), v3 = acc.w * ld_f32(p.w_scale + n + 3);
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.y) + static_cast<size_t>(t) * p.N + n) =
            make_uint2(pack_out16(v0, v1, XDT), pack_out16(v2, v3, XDT));
    }
    if (split > 1) cluster_sync_all();

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kW16TmemCols)
                     : "memory");
    }
}

// Stand-in for gemm_f8_swapab in the occupancy queries: same block size and
// shared memory, no TMEM.  For the product kernel itself the occupancy API
// answers one CTA per SM at any shared-memory size (it cannot know how many
// TMEM columns a CTA will allocate), while the GPU runs as many side by side
// as shared memory allows (two at 112 KB, seen by ncu).
// (The W8A16 kernel has its own twin with its block size.)
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 1) swapab_occupancy_twin() {}

constexpr int kMaxDevices = 64;
std::atomic<int> g_attr_set[kMaxDevices];
std::atomic<int> g_smem_per_sm[kMaxDevices];    // shared memory per SM (bytes)
std::atomic<int> g_smem_reserved[kMaxDevices];  // reserved per CTA (bytes)

size_t swap_smem_bytes(int stages, int stage_bytes) {
    return 1024 + size_t(stages) * stage_bytes + size_t(2 * stages + 1) * 8 + 16;
}

// The largest ring used: kSwSmemTarget or the floor for kSwMaxT; the
// attribute is set once per device to cover every launch, with the
// shared-memory carveout at its maximum so that the CTAs the launcher counts
// on fit side by side.
constexpr size_t kSwSmemMax = kSwSmemTarget + 32 * 1024;

int ensure_attr(int dev) {
    if (g_attr_set[dev].load(std::memory_order_acquire)) return FP8L_OK;
    int per_sm = 0, reserved = 0;
    if (cudaFuncSetAttribute(gemm_f8_swapab, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSwSmemMax)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_f8_swapab, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_f8_swapab_q<FP8L_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSqSmemMax)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_f8_swapab_q<FP8L_F16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_f8_swapab_q<FP8L_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSqSmemMax)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_f8_swapab_q<FP8L_BF16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_w8a16_tc<FP8L_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSwSmemMax)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_w8a16_tc<FP8L_F16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_w8a16_tc<FP8L_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSwSmemMax)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_w8a16_tc<FP8L_BF16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(swapab_occupancy_twin<kSwThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSqSmemMax)) != cudaSuccess ||
        cudaFuncSetAttribute(swapab_occupancy_twin<kSwThreads>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(swapab_occupancy_twin<kSqThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSqSmemMax)) != cudaSuccess ||
        cudaFuncSetAttribute(swapab_occupancy_twin<kSqThreads>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(swapab_occupancy_twin<kW16Threads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSwSmemMax)) != cudaSuccess ||
        cudaFuncSetAttribute(swapab_occupancy_twin<kW16Threads>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
        return FP8L_ECUDA;
    g_smem_per_sm[dev].store(per_sm, std::memory_order_relaxed);
    g_smem_reserved[dev].store(reserved, std::memory_order_relaxed);
    g_attr_set[dev].store(1, std::memory_order_release);
    return FP8L_OK;
}

// Clusters of `split` CTAs of this block size and ring size that the GPU
// holds at once (cudaOccupancyMaxActiveClusters of the twin kernel: clusters
// sit within one GPC), cached per device, kernel (0: W8A8, 1: W8A16, 2: W8A8
// with the quantization fused), token tile and split.
std::atomic<int> g_max_clusters[kMaxDevices][3][kSwMaxT / 16][kSwMaxSplit + 1];

int max_clusters(int dev, int kernel, int T, size_t smem, int split) {
    std::atomic<int> &slot = g_max_clusters[dev][kernel][T / 16 - 1][split];
    int n = slot.load(std::memory_order_relaxed);
    if (n > 0) return n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split), 1, 1);
    cfg.blockDim = dim3(kernel == 1 ? kW16Threads : (kernel == 2 ? kSqThreads : kSwThreads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e =
        kernel == 1   ? cudaOccupancyMaxActiveClusters(&n, swapab_occupancy_twin<kW16Threads>, &cfg)
        : kernel == 2 ? cudaOccupancyMaxActiveClusters(&n, swapab_occupancy_twin<kSqThreads>, &cfg)
                      : cudaOccupancyMaxActiveClusters(&n, swapab_occupancy_twin<kSwThreads>, &cfg);
    if (e != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    slot.store(n, std::memory_order_relaxed);
    return n;
}

// The largest cluster whose launch runs in one wave (see launch_swapab).
int pick_split(int dev, int kernel, int T, size_t smem, int tiles, int num_k_blocks, int sms) {
    int slots = g_smem_per_sm[dev].load(std::memory_order_relaxed) /
                static_cast<int>(smem + size_t(g_smem_reserved[dev].load(std::memory_order_relaxed)));
    if (slots < 1) slots = 1;
    if (slots > 8) slots = 8;
    int split = kSwMaxSplit < num_k_blocks ? kSwMaxSplit : num_k_blocks;
    while (split > 1 && (int64_t(tiles) * split > int64_t(sms) * slots ||
                         tiles > max_clusters(dev, kernel, T, smem, split)))
        --split;
    return split < 1 ? 1 : split;
}

}  // namespace

// Swapped-operand product for 1 <= M <= 128 (fp8_scaled_mm).  Stages: as
// many as fit kSwSmemTarget (at least 3, so the fp32 tile fits the ring);
// split: CTAs per tile so that the CTA slots of the GPU share the weight
// stream, at most kSwMaxSplit and at most the k-blocks.
int launch_swapab(const uint8_t *a, const uint8_t *w, int M, int N, int K, const float *a_scale,
                  int a_per_token, const float *w_scale, int w_per_channel,
                  const float *out_scale, void *y, int out_dtype, unsigned *status, int sms,
                  bool stable, cudaStream_t stream) {
    if (M < 1 || M > kSwMaxT) return FP8L_ESHAPE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8L_ECUDA;
    if (ensure_attr(dev) != FP8L_OK) return FP8L_ECUDA;
    SwapParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.T = (M + 15) & ~15;
    p.stage_bytes = kSwWBytes + p.T * SW_BK;
    int stages = static_cast<int>((kSwSmemTarget - 1024 - 24) / (p.stage_bytes + 16));
    if (stages > kSwMaxStages) stages = kSwMaxStages;
    if (stages < 3) stages = 3;
    p.stages = stages;
    const size_t smem = swap_smem_bytes(stages, p.stage_bytes);
    if (smem > kSwSmemMax || size_t(p.T) * kSwPitch * 4 > size_t(stages) * p.stage_bytes)
        return FP8L_ESHAPE;
    p.num_k_blocks = (K + SW_BK - 1) / SW_BK;
    p.a_scale = a_scale;
    p.w_scale = w_scale;
    p.w_per_channel = w_per_channel;
    p.a_per_token = a_per_token;
    p.out_scale = out_scale;
    p.y = y;
    p.out_dtype = out_dtype;
    p.status = status;
    const WaitConfig wc = wait_config();
    p.wait_cycles = wc.cycles;
    p.stall = wc.stall;
    p.prefetch = stable ? 1 : 0;
    p.x_stages = 0;

    // split: the largest cluster whose launch runs in one wave (a cluster
    // sits in one GPC, so fewer clusters of s CTAs fit than slots / s: at
    // two CTAs per SM 97 of 3, 46 of 6, 36 of 8; a second wave measured up
    // to 1.5x slower)
    const int tiles = (N + SW_BM - 1) / SW_BM;
    const int split = pick_split(dev, 0, p.T, smem, tiles, p.num_k_blocks, sms);
    p.split = split;

    CUtensorMap mw, ma;
    if (make_kmajor_map(&mw, w, N, K, SW_BK, SW_BM) != FP8L_OK) return FP8L_ECUDA;
    if (make_kmajor_map(&ma, a, M, K, SW_BK, p.T) != FP8L_OK) return FP8L_ECUDA;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(int64_t(tiles) * split), 1, 1);
    cfg.blockDim = dim3(kSwThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    if (split > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = static_cast<unsigned>(split);
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    if (stable) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    if (cudaLaunchKernelEx(&cfg, gemm_f8_swapab, mw, ma, p) != cudaSuccess) return FP8L_ECUDA;
    return launch_status();
}

// W8A16 product on tcgen05 for 1 <= M <= 64 (fp8_w8a16_mm).  A token ring
// of two stages (2 T x 128 bytes each) and as many 16 KB weight stages as
// then fit kSwSmemTarget, a multiple of the converter groups (at most
// kW16MaxWStages); split as for the W8A8 product.
int launch_w8a16_tc(const void *x, int x_dtype, const uint8_t *w, bool packed, const float *w_scale,
                    int M, int N, int K, void *y, unsigned *status, int sms, bool stable,
                    cudaStream_t stream) {
    if (M < 1 || M > kW16MaxT) return FP8L_ESHAPE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8L_ECUDA;
    if (ensure_attr(dev) != FP8L_OK) return FP8L_ECUDA;
    W16Params p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.T = (M + 15) & ~15;
    p.x_stage_bytes = 2 * p.T * 128;
    p.x_stages = 2;  // tokens come from L2; the shared memory goes to weights in flight
    const size_t fixed = 1024 + 16 + size_t(2 * kW16MaxWStages + 2 * 4 + 2 * kW16ABufs + 1) * 8 +
                         size_t(p.x_stages) * p.x_stage_bytes;
    int wst = static_cast<int>((size_t(kSwSmemTarget) - fixed) / kW16WBytes);
    if (wst > kW16MaxWStages) wst = kW16MaxWStages;
    wst -= wst % kW16Groups;  // each stage always consumed by the same group
    if (wst < 2 * kW16Groups) wst = 2 * kW16Groups;
    p.w_stages = wst;
    const size_t ring = size_t(wst) * kW16WBytes + size_t(p.x_stages) * p.x_stage_bytes;
    const size_t smem = 1024 + ring + size_t(2 * wst + 2 * p.x_stages + 2 * kW16ABufs + 1) * 8 + 16;
    if (smem > kSwSmemMax || size_t(p.T) * kSwPitch * 4 > ring) return FP8L_ESHAPE;
    p.num_k_blocks = (K + W16_BK - 1) / W16_BK;
    p.packed = packed ? 1 : 0;
    p.w_scale = w_scale;
    p.y = y;
    p.status = status;
    const WaitConfig wc = wait_config();
    p.wait_cycles = wc.cycles;
    p.stall = wc.stall;
    p.prefetch = stable ? 1 : 0;
    const int tiles = (N + SW_BM - 1) / SW_BM;
    p.split = pick_split(dev, 1, p.T, smem, tiles, p.num_k_blocks, sms);

    CUtensorMap mw, mx;
    if (packed) {
        // [N/16 groups][C chunks][1 KB = 16 rows x 64 bytes] as 8-byte elements:
        // box of 8 groups x 2 chunks x 128 elements
        const uint64_t C = static_cast<uint64_t>((K + 63) / 64);
        const uint64_t dims[3] = {128, C, static_cast<uint64_t>(N / 16)};
        const uint64_t strides[2] = {1024, C * 1024};
        const uint32_t box[3] = {128, 2, SW_BM / 16};
        if (make_tile_map(&mw, w, 8, 3, dims, strides, box, false) != FP8L_OK) return FP8L_ECUDA;
    } else {
        const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
        const uint64_t strides[1] = {static_cast<uint64_t>(K)};
        const uint32_t box[2] = {W16_BK, SW_BM};
        if (make_tile_map(&mw, w, 1, 2, dims, strides, box, true) != FP8L_OK) return FP8L_ECUDA;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
        const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
        const uint32_t box[2] = {64, static_cast<uint32_t>(p.T)};
        if (make_tile_map(&mx, x, 2, 2, dims, strides, box, true) != FP8L_OK) return FP8L_ECUDA;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(int64_t(tiles) * p.split), 1, 1);
    cfg.blockDim = dim3(kW16Threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    if (p.split > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = static_cast<unsigned>(p.split);
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    if (stable) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    const cudaError_t e = x_dtype == FP8L_BF16
                              ? cudaLaunchKernelEx(&cfg, gemm_w8a16_tc<FP8L_BF16>, mw, mx, p)
                              : cudaLaunchKernelEx(&cfg, gemm_w8a16_tc<FP8L_F16>, mw, mx, p);
    if (e != cudaSuccess) return FP8L_ECUDA;
    return launch_status();
}

// Swapped-operand product with the activation quantization fused
// (fp8_quant_scaled_mm): 1 <= M <= 128, dynamic mode up to
// FP8L_FUSED_DYNAMIC_MAX_BYTES of x.  Weight stages as in launch_swapab, less
// the two 16-bit token stages.
int launch_swapab_q(const void *x, int x_dtype, const uint8_t *w, int M, int N, int K, float *a_scale,
                    int dynamic, const float *w_scale, int w_per_channel, const float *out_scale, void *y,
                    int out_dtype, unsigned *status, int sms, bool stable, cudaStream_t stream) {
    if (M < 1 || M > kSwMaxT) return FP8L_ESHAPE;
    if (dynamic && int64_t(M) * K * 2 > FP8L_FUSED_DYNAMIC_MAX_BYTES) return FP8L_ESHAPE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8L_ECUDA;
    if (ensure_attr(dev) != FP8L_OK) return FP8L_ECUDA;
    SwapParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.T = (M + 15) & ~15;
    p.stage_bytes = kSwWBytes + p.T * SW_BK;
    const size_t xsb = size_t(M) * 256;
    // token ring first (kSqXRingBytes, 2 to kSqMaxXStages stages), weight
    // stages in the rest of kSqSmemTarget; then, if that is fewer weight
    // stages than the plain swapped product keeps in flight, the token ring
    // gives up stages to match it as long as kSqMinXStagesTrade remain
    const size_t fixed = 1024 + 64;
    const size_t per_w = p.stage_bytes + 24, per_x = xsb + 16;
    int xst = static_cast<int>(kSqXRingBytes / xsb);
    if (xst > kSqMaxXStages) xst = kSqMaxXStages;
    if (xst < 2) xst = 2;
    auto w_room = [&](int xs) {
        const size_t used = fixed + size_t(xs) * per_x;
        return used >= kSqSmemTarget ? 0 : static_cast<int>((kSqSmemTarget - used) / per_w);
    };
    int stages = w_room(xst);
    int plain = static_cast<int>((kSwSmemTarget - 1024 - 24) / (p.stage_bytes + 16));
    if (plain > kSwMaxStages) plain = kSwMaxStages;
    if (stages < plain) {
        const size_t need = fixed + size_t(plain) * per_w;
        const int xs = need >= kSqSmemTarget ? 0 : static_cast<int>((kSqSmemTarget - need) / per_x);
        if (xs >= kSqMinXStagesTrade && xs < xst) {
            xst = xs;
            stages = plain;
        }
    }
    if (stages > kSwMaxStages) stages = kSwMaxStages;
    if (stages < 3) stages = 3;
    p.x_stages = xst;
    const size_t xring = size_t(xst) * xsb;
    p.stages = stages;
    const size_t ring = size_t(stages) * p.stage_bytes + xring;
    const size_t smem = 1024 + ((ring + 7) & ~size_t(7)) + size_t(3 * stages + 2 * xst + 1) * 8 + 16;
    if (smem > kSqSmemMax || size_t(p.T) * kSwPitch * 4 > size_t(stages) * p.stage_bytes)
        return FP8L_ESHAPE;
    p.num_k_blocks = (K + SW_BK - 1) / SW_BK;
    p.a_scale = a_scale;
    p.w_scale = w_scale;
    p.w_per_channel = w_per_channel;
    p.a_per_token = 0;
    p.out_scale = out_scale;
    p.y = y;
    p.out_dtype = out_dtype;
    p.status = status;
    const WaitConfig wc = wait_config();
    p.wait_cycles = wc.cycles;
    p.stall = wc.stall;
    p.prefetch = stable ? 1 : 0;
    const int tiles = (N + SW_BM - 1) / SW_BM;
    p.split = pick_split(dev, 2, p.T, smem, tiles, p.num_k_blocks, sms);

    CUtensorMap mw, mx;
    if (make_kmajor_map(&mw, w, N, K, SW_BK, SW_BM) != FP8L_OK) return FP8L_ECUDA;
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
        const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
        const uint32_t box[2] = {64, static_cast<uint32_t>(M)};
        if (make_tile_map(&mx, x, 2, 2, dims, strides, box, false) != FP8L_OK) return FP8L_ECUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(int64_t(tiles) * p.split), 1, 1);
    cfg.blockDim = dim3(kSqThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    if (p.split > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = static_cast<unsigned>(p.split);
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    if (stable) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    const cudaError_t e =
        x_dtype == FP8L_BF16
            ? cudaLaunchKernelEx(&cfg, gemm_f8_swapab_q<FP8L_BF16>, mw, mx, p, a_scale, dynamic, x)
            : cudaLaunchKernelEx(&cfg, gemm_f8_swapab_q<FP8L_F16>, mw, mx, p, a_scale, dynamic, x);
    if (e != cudaSuccess) return FP8L_ECUDA;
    return launch_status();
}

}  // namespace fp8l

// Weight blocks (128 rows) up to which the fused product was measured
// faster than quantizer + product on a 152-SM GB300: up to 8 tokens while
// every block has a CTA in the first wave (2 per SM), 9-16 tokens while the
// blocks are few enough for clusters to split K (one per SM or fewer).
// Beyond that the fused kernel's CTAs, with fewer weight stages and a
// conversion step in each stage's round trip, stream too slowly alone
// (M = 1 at 57344 x 8192: 88 us against 80; M = 16 at 28672 x 4096: 29.3
// against 27.3; M = 32 at 6144 x 4096: 14.3 against 13.5).
constexpr int64_t kFusedPreferBlocks = 152;
constexpr int64_t kFusedPreferStreamElems = 16384;

extern "C" int fp8_quant_scaled_mm_preferred(int64_t M, int64_t N, int64_t K, int dynamic) {
    using namespace fp8l;
    if (M < 1 || M > 16 || N <= 0 || K <= 0 || N > (1 << 20) || K > (1 << 20) || N % 16 != 0 || K % 16 != 0)
        return 0;
    if (dynamic && M * K * 2 > FP8L_FUSED_DYNAMIC_MAX_BYTES) return 0;
    if (fp8_scaled_mm_kernel(M, N, K, 0u) == FP8L_KERNEL_STREAM)
        // the weight stream with the codes made in the kernel: up to 8 tokens
        // (one token tile), or short rows (the tiny 16 x 512 layer: 2.6 us
        // against 6.0); 16 tokens of 4096 took 11.9 us against 11.7
        return (M <= 8 || M * K <= kFusedPreferStreamElems) ? 1 : 0;
    const int64_t blocks = (N + SW_BM - 1) / SW_BM;
    return blocks <= (M <= 8 ? 2 : 1) * kFusedPreferBlocks ? 1 : 0;
}

extern "C" int fp8_quant_scaled_mm(const void *x, int x_dtype, const uint8_t *w, int64_t M, int64_t N,
                                   int64_t K, float *a_scale, int dynamic, const float *w_scale,
                                   int w_per_channel, const float *out_scale, void *y, int out_dtype,
                                   void *workspace, unsigned flags, void *stream) {
    using namespace fp8l;
    if (x_dtype != FP8L_F16 && x_dtype != FP8L_BF16) return FP8L_EINVAL;
    if (out_dtype != FP8L_F16 && out_dtype != FP8L_BF16 && out_dtype != FP8L_E4M3) return FP8L_EINVAL;
    if ((flags & ~(FP8L_WEIGHTS_STABLE | FP8L_KERNEL_MASK)) != 0u) return FP8L_EINVAL;
    unsigned kernel = flags & FP8L_KERNEL_MASK;
    if (kernel == FP8L_KERNEL_TILED) return FP8L_EINVAL;
    if (a_scale == nullptr || w_scale == nullptr || workspace == nullptr || w == nullptr) return FP8L_EINVAL;
    if (out_dtype == FP8L_E4M3 && out_scale == nullptr) return FP8L_EINVAL;
    if (M < 0 || M > 128 || N <= 0 || K <= 0 || N > (1 << 20) || K > (1 << 20) || N % 16 != 0 ||
        K % 16 != 0)
        return FP8L_ESHAPE;
    if (dynamic && M * K * 2 > FP8L_FUSED_DYNAMIC_MAX_BYTES) return FP8L_ESHAPE;
    // the kernel fp8_scaled_mm would run the codes through (its tile kernel
    // excepted): the same MMAs, so the same result
    if (kernel == FP8L_KERNEL_AUTO)
        kernel = fp8_scaled_mm_kernel(M, N, K, 0u) == FP8L_KERNEL_STREAM ? FP8L_KERNEL_STREAM
                                                                        : FP8L_KERNEL_SWAPPED;
    if (kernel == FP8L_KERNEL_STREAM && M > 16) return FP8L_ESHAPE;
    if (M > 0 && (x == nullptr || y == nullptr)) return FP8L_EINVAL;
    auto misaligned4 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) != 0; };
    if (!aligned16(w) || !aligned16(workspace) || (M > 0 && (!aligned16(x) || !aligned16(y))) ||
        misaligned4(a_scale) || misaligned4(w_scale) || (out_dtype == FP8L_E4M3 && misaligned4(out_scale)))
        return FP8L_EALIGN;
    int sms = 0;
    int st = check_device(&sms);
    if (st != FP8L_OK) return st;
    if (M == 0) return FP8L_OK;
    if (kernel == FP8L_KERNEL_STREAM)
        return launch_skinny_quant(x, x_dtype, w, static_cast<int>(M), static_cast<int>(N),
                                   static_cast<int>(K), a_scale, dynamic ? 1 : 0, w_scale,
                                   w_per_channel ? 1 : 0, out_scale, y, out_dtype,
                                   (flags & FP8L_WEIGHTS_STABLE) != 0u, as_stream(stream));
    return launch_swapab_q(x, x_dtype, w, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                           a_scale, dynamic ? 1 : 0, w_scale, w_per_channel ? 1 : 0, out_scale, y, out_dtype,
                           status_word(workspace), sms, (flags & FP8L_WEIGHTS_STABLE) != 0u, as_stream(stream));
}

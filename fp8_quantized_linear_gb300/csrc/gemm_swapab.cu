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
// shared memory per CTA aimed at: two CTAs per SM, or four with a token
// tile of at most 32 rows (stages of 18 or 20 KB)
constexpr int kSwSmemTarget = 112 * 1024;
constexpr int kSwSmemTargetFewTokens = 112 * 1024;

struct SwapParams {
    int M, N, K;
    int T;            // MMA N: M rounded up to 16
    int stages;       // ring depth
    int stage_bytes;  // kSwWBytes + T * SW_BK
    int num_k_blocks;
    int split;        // CTAs of a cluster sharing a tile (1: no cluster)
    int prefetch;     // stable weights: weight blocks issued before griddepcontrol.wait
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
            const uint32_t lo = e4m3x2(od.quot(v[0]), od.quot(v[1]));
            const uint32_t hi = e4m3x2(od.quot(v[2]), od.quot(v[3]));
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

// Stand-in for gemm_f8_swapab in the occupancy queries: same block size and
// shared memory, no TMEM.  For the product kernel itself the occupancy API
// answers one CTA per SM at any shared-memory size (it cannot know how many
// TMEM columns a CTA will allocate), while the GPU runs as many side by side
// as shared memory allows (two at 112 KB, seen by ncu).
__global__ void __launch_bounds__(kSwThreads, 1) swapab_occupancy_twin() {}

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
        cudaFuncSetAttribute(swapab_occupancy_twin, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSwSmemMax)) != cudaSuccess ||
        cudaFuncSetAttribute(swapab_occupancy_twin, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
        return FP8L_ECUDA;
    g_smem_per_sm[dev].store(per_sm, std::memory_order_relaxed);
    g_smem_reserved[dev].store(reserved, std::memory_order_relaxed);
    g_attr_set[dev].store(1, std::memory_order_release);
    return FP8L_OK;
}

// Clusters of `split` CTAs of this ring size that the GPU holds at once
// (cudaOccupancyMaxActiveClusters of the twin kernel: clusters sit within
// one GPC), cached per device, token tile and split.
std::atomic<int> g_max_clusters[kMaxDevices][kSwMaxT / 16][kSwMaxSplit + 1];

int max_clusters(int dev, int T, size_t smem, int split) {
    std::atomic<int> &slot = g_max_clusters[dev][T / 16 - 1][split];
    int n = slot.load(std::memory_order_relaxed);
    if (n > 0) return n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split), 1, 1);
    cfg.blockDim = dim3(kSwThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, swapab_occupancy_twin, &cfg) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    slot.store(n, std::memory_order_relaxed);
    return n;
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
    const int target = p.T <= 32 ? kSwSmemTargetFewTokens : kSwSmemTarget;
    int stages = static_cast<int>((target - 1024 - 24) / (p.stage_bytes + 16));
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

    // CTAs of this ring size side by side on an SM (shared memory is the
    // only limit: 128 threads of 72 registers)
    int slots = g_smem_per_sm[dev].load(std::memory_order_relaxed) /
                static_cast<int>(smem + size_t(g_smem_reserved[dev].load(std::memory_order_relaxed)));
    if (slots < 1) slots = 1;
    if (slots > 8) slots = 8;
    // split: the largest cluster whose launch runs in one wave (a cluster
    // sits in one GPC, so fewer clusters of s CTAs fit than slots / s: at
    // two CTAs per SM 97 of 3, 46 of 6, 36 of 8; a second wave measured up
    // to 1.5x slower)
    const int tiles = (N + SW_BM - 1) / SW_BM;
    int split = kSwMaxSplit < p.num_k_blocks ? kSwMaxSplit : p.num_k_blocks;
    while (split > 1 && (int64_t(tiles) * split > int64_t(sms) * slots ||
                         tiles > max_clusters(dev, p.T, smem, split)))
        --split;
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

}  // namespace fp8l

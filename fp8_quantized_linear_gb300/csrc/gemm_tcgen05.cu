// W8A8 scaled product on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// ("[Kernel][FP8] Initial support with dynamic per-tensor scaling": the
// forward pass is torch._scaled_mm of the E4M3 activations and weights with
// their scales; "Marlin fp8": per-output-channel weight scales; "RFC: FP8
// Quantization Schema in vLLM": output_scale for an E4M3 result.)
//
//   y[m, n] = cast( sum_k dec(a[m,k]) dec(w[n,k]) * a_scale(m) * w_scale(n) )
//   (a_scale(m) = a_scale[m] with per-token activation scales, else a_scale[0])
//
// Structure (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: 128x128 A tile and 256x128 W tile per k-block
//               (E4M3 bytes, 128-byte swizzle) into a STAGES-deep ring of
//               shared-memory stages guarded by full/empty mbarriers.
//   warp 1      owns the TMEM allocation (2 x 256 fp32 columns: a double
//               buffered 128x256 accumulator) and one lane issues
//               tcgen05.mma.cta_group::1.kind::f8f6f4 (M=128, N=256, K=32),
//               four per k-block; tcgen05.commit frees a stage when its
//               MMAs retire and publishes a finished accumulator.
//   warps 2-9   epilogue, two warps per TMEM lane quarter (warp % 4), each
//               over half of the columns: tcgen05.ld of their 32 TMEM lanes
//               (= tile rows), scale by a_scale * w_scale(n), round to bf16/fp16 or divide
//               by output_scale and cast to E4M3, 16-byte stores.  With two
//               accumulators the epilogue of tile i overlaps the MMAs of
//               tile i+1.
// Tiles are visited M-block fastest, so the CTAs working at one time share a
// few W column blocks and all of A in L2.  Out-of-range rows / K columns of
// a tile are zero-filled by TMA and masked in the epilogue.
// Every mbarrier wait is bounded: on time-out the CTA raises an abort flag,
// records FP8L_ETIMEOUT in the workspace status word, lets the other roles
// drop out, waits (bounded) for its own copies and MMAs, frees TMEM, returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "tc_device.cuh"

namespace fp8l {
namespace {

constexpr int BM = 128;           // tile rows (tokens)      = MMA M
constexpr int BN = 256;           // tile columns (channels) = MMA N
constexpr int BK = 128;           // k-block, bytes = E4M3 elements = swizzle span
constexpr int UMMA_K = 32;        // K of one kind::f8f6f4 MMA
constexpr int STAGES = 4;
constexpr int kABytes = BM * BK;  // 16 KB
constexpr int kBBytes = BN * BK;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kTmemCols = 2 * BN;  // two accumulators
// 8 epilogue warps: two per TMEM lane quarter (warp % 4), each taking half of
// the tile's 32-column chunks.  With one per quarter the epilogue, one warp
// per scheduler working through each row's chunks in sequence, was
// latency-bound and held the main loop back: a one-round 1024 x 4096 x 4096
// product with E4M3 output and per-channel scales took 25.0 us against 17.6
// us for bf16 output and a per-tensor scale (21.2 us with 8 warps), 8192 x
// 28672 x 4096 737 us against 554.
constexpr int kEpiWarps = 8;
constexpr int kEpiGroups = kEpiWarps / 4;  // warps sharing one TMEM lane quarter
static_assert(kEpiWarps % 4 == 0, "whole groups of four epilogue warps");
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kNumBarriers = 2 * STAGES + 2 + 2 + 1;
constexpr int kMaxGroups = 256;  // grouped mode: experts
// shared memory: alignment slack, stages, barriers, TMEM slot and abort flag
// (16 bytes), then the grouped mode's row ranges and m-block prefix sums
constexpr size_t kGroupSmemBytes = 3 * (kMaxGroups + 1) * sizeof(int);
constexpr size_t kSmemBytes =
    1024 + size_t(STAGES) * kStageBytes + kNumBarriers * 8 + 16 + kGroupSmemBytes;

struct GemmParams {
    int M, N, K;
    int num_m_blocks, num_n_blocks, num_k_blocks;
    const float *a_scale;
    const float *w_scale;
    int w_per_channel;
    int a_per_token;  // a_scale has M entries
    const float *out_scale;
    void *y;
    int out_dtype;
    unsigned *status;
    const int *group_offs;  // grouped mode: [num_groups + 1] row offsets in device memory
    int num_groups;         // 0: one product; > 0: expert e takes rows offs[e] .. offs[e+1]-1
                            // and the weight rows e*N .. e*N + N-1 (w is [num_groups, N, K])
    long long wait_cycles;  // limit of the main waits (kDefaultWaitCycles unless a test shortened it)
    unsigned stall;         // kStallMma: testing the time-out path
    int split;  // > 1: a cluster of `split` CTAs shares one tile and splits its k-blocks
    // CTA-pair kernel: 256 x 256 tiles over the columns [0, pair_n_main)
    // (pair_main_tiles of them), then pair_tail_n columns of tiles
    // pair_tail_w wide over [pair_n_main, N) so that the last round of tiles
    // spreads over the SM pairs (pair_tail_n = 0: 256-wide tiles throughout)
    int pair_main_tiles, pair_n_main, pair_tail_w, pair_tail_n;
    uint32_t idesc_tail;  // instruction descriptor of the tail tiles (N = pair_tail_w)
};

// Instruction descriptor, kind::f8f6f4: D f32 (bits 4-5 = 1), A and B E4M3
// (format 0, bits 7-9 and 10-12), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// Scales and stores 32 accumulator columns [n0, n0+32) of row m; sa is the
// row's activation scale, sa_sw = sa * (per-tensor weight scale) and wsc the
// per-channel weight scales of the tile's weights (w_scale, or the expert's).
__device__ __forceinline__ void store_row_chunk(const GemmParams &p, const uint32_t (&r)[32],
                                                int m, int n0, float sa, float sa_sw,
                                                const float *wsc) {
    const bool full32 = n0 + 32 <= p.N;  // N % 16 == 0: else exactly 16 columns remain
    float v[32];
    if (p.w_per_channel && full32 && (reinterpret_cast<uintptr_t>(wsc) & 15u) == 0) {
        // n0 is a multiple of 32: the chunk's 32 scales in eight 16-byte loads
        const float4 *s4 = reinterpret_cast<const float4 *>(wsc + n0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 sw = __ldg(s4 + q);
            v[4 * q] = __uint_as_float(r[4 * q]) * (sa * sw.x);
            v[4 * q + 1] = __uint_as_float(r[4 * q + 1]) * (sa * sw.y);
            v[4 * q + 2] = __uint_as_float(r[4 * q + 2]) * (sa * sw.z);
            v[4 * q + 3] = __uint_as_float(r[4 * q + 3]) * (sa * sw.w);
        }
    } else if (p.w_per_channel) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float sw = (j < 16 || full32) ? __ldg(wsc + n0 + j) : 0.0f;
            v[j] = __uint_as_float(r[j]) * (sa * sw);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * sa_sw;
    }
    if (p.out_dtype == FP8L_E4M3) {
        const OutDiv d = OutDiv::make(__ldg(p.out_scale));
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = out_e4m3x2(d.quot(v[4 * i]), d.quot(v[4 * i + 1]));
            const uint32_t hi = out_e4m3x2(d.quot(v[4 * i + 2]), d.quot(v[4 * i + 3]));
            w[i] = lo | (hi << 16);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.y) +
                                               static_cast<size_t>(m) * p.N + n0);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        if (full32) dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_out16(v[2 * i], v[2 * i + 1], p.out_dtype);
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.y) +
                                               static_cast<size_t>(m) * p.N + n0);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        if (full32) {
            dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
            dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
        }
    }
}

// Where a tile sits: rows [row0, row_end) of A and Y (row_end bounds the
// valid rows), weight rows from w_row0, output columns from n0, expert e.
struct TileInfo {
    int row0, row_end, w_row0, n0, e;
};

// Grouped mode: per expert the valid row range [lo, hi) (offsets clamped to
// [0, M] and made non-decreasing) and the prefix sum of its 128-row blocks.
struct GroupTable {
    const int *lo, *hi, *prefix;  // shared memory; prefix has num_groups + 1 entries
};

__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, const GroupTable &g, int tile,
                                              int total_mb) {
    TileInfo t;
    const int mbg = tile % total_mb;
    const int nb = tile / total_mb;
    t.n0 = nb * BN;
    if (p.num_groups == 0) {
        t.row0 = mbg * BM;
        t.row_end = p.M;
        t.w_row0 = nb * BN;
        t.e = 0;
        return t;
    }
    // last expert whose first block is <= mbg (empty experts are skipped:
    // their prefix equals the next one's)
    int lo = 0, hi = p.num_groups;  // prefix[lo] <= mbg < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (g.prefix[mid] <= mbg) lo = mid; else hi = mid;
    }
    t.e = lo;
    t.row0 = g.lo[lo] + (mbg - g.prefix[lo]) * BM;
    t.row_end = g.hi[lo];
    t.w_row0 = lo * p.N + nb * BN;
    return t;
}

// Split mode: every CTA of the cluster writes its fp32 partial tile into its
// own (idle) stage ring, row pitch kPartPitch floats; after a cluster
// barrier CTA `rank` adds the `split` partials of its rows [rank*rows_per,
// ...) read through distributed shared memory (all `split` loads of a group
// of four columns issued before any is used), scales, casts and stores: four
// columns per thread, consecutive threads on consecutive columns.
constexpr int kPartPitch = BN + 4;  // floats per partial-tile row (conflict-free v4 stores)
constexpr int kMaxSplit = 4;  // clusters of 8 at this shared-memory size ran 1.4-1.7x slower
static_assert(BM * kPartPitch * 4 <= STAGES * kStageBytes, "partial tile fits in the ring");

__device__ void split_reduce_store(const GemmParams &p, int tile, int rank, uint32_t sbase) {
    const int mb = tile % p.num_m_blocks;
    const int nb = tile / p.num_m_blocks;
    const int rows_per = (BM + p.split - 1) / p.split;
    const int r0 = rank * rows_per;
    const int r1 = r0 + rows_per < BM ? r0 + rows_per : BM;
    const int items = (r1 - r0) * (BN / 4);
    const float sa0 = __ldg(p.a_scale);
    const float sw0 = __ldg(p.w_scale);
    for (int i = threadIdx.x; i < items; i += blockDim.x) {
        const int row = r0 + i / (BN / 4);
        const int col = 4 * (i % (BN / 4));
        const int m = mb * BM + row;
        const int n = nb * BN + col;
        if (m >= p.M || n >= p.N) continue;
        const uint32_t off = sbase + static_cast<uint32_t>((row * kPartPitch + col) * 4);
        float4 part[kMaxSplit];
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q)
            if (q < p.split) part[q] = ld_cluster_v4(off, static_cast<uint32_t>(q));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q) {  // the same order in every run
            if (q < p.split) {
                acc.x += part[q].x;
                acc.y += part[q].y;
                acc.z += part[q].z;
                acc.w += part[q].w;
            }
        }
        float v[4] = {acc.x, acc.y, acc.z, acc.w};
        const float sa = p.a_per_token ? __ldg(p.a_scale + m) : sa0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[j] *= sa * (p.w_per_channel ? __ldg(p.w_scale + n + j) : sw0);
        if (p.out_dtype == FP8L_E4M3) {
            const OutDiv d = OutDiv::make(__ldg(p.out_scale));
            const uint32_t lo = out_e4m3x2(d.quot(v[0]), d.quot(v[1]));
            const uint32_t hi = out_e4m3x2(d.quot(v[2]), d.quot(v[3]));
            *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(p.y) + static_cast<size_t>(m) * p.N + n) =
                lo | (hi << 16);
        } else {
            const uint32_t a = pack_out16(v[0], v[1], p.out_dtype);
            const uint32_t b = pack_out16(v[2], v[3], p.out_dtype);
            *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.y) + static_cast<size_t>(m) * p.N + n) =
                make_uint2(a, b);
        }
    }
}

// ---------------------------------------------------------------- kernel

__global__ void __launch_bounds__(kThreads, 1)
gemm_f8_tcgen05(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
    // launched as a programmatic dependent (stable weights), the kernel is
    // resident before the preceding kernel ends; it touches no global memory
    // until that kernel's writes are visible (a no-op otherwise)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
    uint8_t *gbase = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + STAGES * kStageBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + STAGES * kStageBytes + kNumBarriers * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *g_lo = reinterpret_cast<int *>(gbase + STAGES * kStageBytes + kNumBarriers * 8 + 16);
    int *g_hi = g_lo + (kMaxGroups + 1);
    int *g_prefix = g_hi + (kMaxGroups + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (p.num_groups > 0) {
        // expert row ranges from the device offsets, then the prefix sums of
        // their 128-row blocks (one thread; at most kMaxGroups experts)
        for (int e = threadIdx.x; e <= p.num_groups; e += blockDim.x) {
            const int v = p.group_offs[e];
            g_lo[e] = v < 0 ? 0 : (v > p.M ? p.M : v);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int run = 0, prev = 0;
            for (int e = 0; e < p.num_groups; ++e) {
                const int lo = g_lo[e] > prev ? g_lo[e] : prev;
                int hi = g_lo[e + 1];
                hi = hi > lo ? hi : lo;
                g_prefix[e] = run;
                run += (hi - lo + BM - 1) / BM;
                g_lo[e] = lo;
                g_hi[e] = hi;
                prev = hi;
            }
            g_prefix[p.num_groups] = run;
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), kEpiWarps);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const GroupTable gt{g_lo, g_hi, g_prefix};
    const int total_mb = p.num_groups > 0 ? g_prefix[p.num_groups] : p.num_m_blocks;
    const int num_tiles = total_mb * p.num_n_blocks;
    // persistent mode: tiles blockIdx.x, +gridDim.x, ...; split mode: the
    // cluster's one tile and this CTA's share of its k-blocks
    const bool split = p.split > 1;
    const int rank = split ? static_cast<int>(blockIdx.x) % p.split : 0;
    const int tile_begin = split ? static_cast<int>(blockIdx.x) / p.split : static_cast<int>(blockIdx.x);
    const int tile_step = split ? num_tiles : static_cast<int>(gridDim.x);
    int kb_begin = 0, kb_end = p.num_k_blocks;
    if (split) {
        const int base = p.num_k_blocks / p.split, rem = p.num_k_blocks % p.split;
        kb_begin = rank * base + (rank < rem ? rank : rem);
        kb_end = kb_begin + base + (rank < rem ? 1 : 0);
    }

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;  // per stage: load in flight, its parity
            bool ok = true;
            for (int tile = tile_begin; ok && tile < num_tiles; tile += tile_step) {
                const TileInfo ti = tile_info(p, gt, tile, total_mb);
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_cycles)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + stage * kStageBytes;
                    mbar_expect_tx(full_bar(stage), kStageBytes);
                    tma_load_2d(sa, &tmap_a, kb * BK, ti.row0, full_bar(stage));
                    tma_load_2d(sa + kABytes, &tmap_b, kb * BK, ti.w_row0, full_bar(stage));
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every load this thread issued must land before the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s)) mbar_wait_drain(full_bar(s), (issued_parity >> s) & 1u, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            // testing the time-out path: wait for a barrier that nothing
            // completes before this role's own commit below
            if (p.stall & kStallMma) ok = mbar_wait(done_bar, 0, abort_flag, p.status, p.wait_cycles);
            for (int tile = tile_begin; ok && tile < num_tiles; tile += tile_step) {
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status, p.wait_cycles)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!mbar_wait_fast(full_bar(stage), phase, abort_flag, p.status, p.wait_cycles)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + stage * kStageBytes;
                    // descriptors of the stage's operands; k step: +32 bytes = +2
                    // in the start-address field (addresses >> 4)
                    const uint64_t da = sw128_desc(sa), db = sw128_desc(sa + kABytes);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        mma_f8(d_tmem, da + 2 * k, db + 2 * k, ((kb - kb_begin) | k) != 0 ? 1u : 0u);
                    mma_commit(empty_bar(stage));  // stage reusable once these MMAs retire
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(tfull_bar(acc));  // accumulator ready once all MMAs retire
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // all MMAs of this CTA retire before TMEM is freed
            mma_commit(done_bar);
            mbar_wait_drain(done_bar, 0, p.status);
        }
        __syncwarp();
    } else {
        const int quarter = warp & 3;  // TMEM lanes this warp may read: 32*quarter ..
        const int grp = (warp - 2) >> 2;  // its share of the tile's 32-column chunks
        const int c_begin = grp * (BN / 32) / kEpiGroups, c_end = (grp + 1) * (BN / 32) / kEpiGroups;
        const int row = quarter * 32 + lane;
        const float sa0 = __ldg(p.a_scale);
        const float sw0 = __ldg(p.w_scale);
        int acc = 0;
        uint32_t acc_phase = 0;
        if (split) {
            // fp32 partial tile into the (now idle) stage ring: part[row][col]
            if (mbar_wait(tfull_bar(0), 0, abort_flag, p.status, p.wait_cycles)) {
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
                const uint32_t prow = sbase + static_cast<uint32_t>(row * kPartPitch * 4);
#pragma unroll 1
                for (int c = c_begin; c < c_end; ++c) {
                    uint32_t r[32];
                    tmem_ld32(taddr + static_cast<uint32_t>(c * 32), r);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(prow + static_cast<uint32_t>((c * 32 + 4 * j) * 4), r[4 * j],
                                     r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                }
                tc_fence_before();
            }
        }
        for (int tile = split ? num_tiles : tile_begin; tile < num_tiles; tile += tile_step) {
            const TileInfo ti = tile_info(p, gt, tile, total_mb);
            if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.status, p.wait_cycles)) break;
            tc_fence_after();
            const int m = ti.row0 + row;
            const bool row_ok = m < ti.row_end;
            const float sa = p.a_per_token ? (row_ok ? __ldg(p.a_scale + m) : 0.0f) : sa0;
            // grouped: the expert's scales (one, or N)
            const float *wsc = p.w_scale + (p.w_per_channel ? static_cast<size_t>(ti.e) * p.N : ti.e);
            const float sa_sw = sa * (p.num_groups > 0 && !p.w_per_channel ? __ldg(wsc) : sw0);
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = c_begin; c < c_end; ++c) {
                uint32_t r[32];
                tmem_ld32(taddr + static_cast<uint32_t>(c * 32), r);
                const int n0 = ti.n0 + c * 32;
                if (row_ok && n0 < p.N) store_row_chunk(p, r, m, n0, sa, sa_sw, wsc);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    if (split) {
        // every CTA of the cluster has its partial tile in shared memory; CTA
        // `rank` adds the `split` partials of its rows and stores them
        cluster_sync_all();
        split_reduce_store(p, tile_begin, rank, sbase);
        cluster_sync_all();  // peers may still be reading this CTA's partials
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
    }
}


// ---------------------------------------------------------------- CTA-pair kernel
//
// The same product with the tile split over a pair of SMs (a cluster of two
// CTAs): tcgen05.mma.cta_group::2 computes a 256 x 256 tile per k-step, each
// CTA staging 128 rows of A and 128 rows (half of the tile's columns) of W;
// the MMA reads the peer's operand halves from its shared memory, and each
// CTA's TMEM receives its 128 rows of the accumulator.  Per SM and k-block
// that is 32 KB of operands for the same 128 x 256 x 128 of MMA work that
// costs 48 KB in the single-SM kernel, so six stages fit where four did and
// the loads run further ahead of the tensor pipe.
//   warp 0     TMA producer in each CTA: its own A and W halves; both CTAs'
//              copies complete on the even CTA's full barrier, armed by the
//              even CTA for the bytes of both.
//   warp 1     TMEM (512 columns, allocated by both CTAs together); in the
//              even CTA one lane issues the MMAs, and its commits arrive on
//              the stage-empty and accumulator-full barriers of both CTAs.
//   warps 2-9  epilogue in each CTA over its 128 rows, two warps per TMEM
//              lane quarter splitting the columns; the accumulator-empty
//              barrier in the even CTA collects the 16 epilogue warps of the
//              pair.
// Waits are bounded as in the single-SM kernel; a time-out also raises the
// peer's abort flag, and both CTAs meet at a cluster barrier before TMEM is
// released.
constexpr int P_BM = 128;                            // rows per CTA; a pair covers 256
constexpr int P_BN = 256;                            // MMA N; each CTA stages half of it
constexpr int P_STAGES = 6;
constexpr int kPABytes = P_BM * BK;                  // 16 KB
constexpr int kPBBytes = (P_BN / 2) * BK;            // 16 KB
constexpr int kPStageBytes = kPABytes + kPBBytes;    // 32 KB
constexpr int kPNumBarriers = 2 * P_STAGES + 2 + 2 + 1;
constexpr size_t kPSmemBytes = 1024 + size_t(P_STAGES) * kPStageBytes + kPNumBarriers * 8 + 16;
// kind::f8f6f4, D f32, A and B E4M3 K-major, N = 256, M = 256 (pair)
constexpr uint32_t kIdescPair = (1u << 4) | (uint32_t(P_BN >> 3) << 17) | (uint32_t(256 >> 4) << 24);

// TMA load into this CTA's shared memory, completing on an mbarrier of
// either CTA of the pair (bar: shared::cluster address)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Where a pair tile sits: 256-row block mt, first column n0, width w (256,
// or the tail width).
struct PairTile {
    int mt, n0, w;
};

__device__ __forceinline__ PairTile pair_tile(const GemmParams &p, int tile, int tiles_m) {
    PairTile t;
    if (tile < p.pair_main_tiles) {
        t.mt = tile % tiles_m;
        t.n0 = (tile / tiles_m) * P_BN;
        t.w = P_BN;
    } else {
        const int u = tile - p.pair_main_tiles;
        t.mt = u % tiles_m;
        t.n0 = p.pair_n_main + (u / tiles_m) * p.pair_tail_w;
        t.w = p.pair_tail_w;
    }
    return t;
}

// arrive on the barrier at this offset in both CTAs once the MMAs issued so
// far have retired
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_f8_pair(const __grid_constant__ CUtensorMap tmap_a,
             const __grid_constant__ CUtensorMap tmap_b,
             const __grid_constant__ CUtensorMap tmap_bt, const GemmParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // see gemm_f8_tcgen05
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + P_STAGES * kPStageBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (P_STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * P_STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * P_STAGES + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * P_STAGES + 4);
    uint32_t *tmem_slot =
        reinterpret_cast<uint32_t *>(gbase + P_STAGES * kPStageBytes + kPNumBarriers * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(full_bar(s), 1);   // the even CTA's arming arrival (+ both CTAs' bytes)
            mbar_init(empty_bar(s), 1);  // the MMA commit, multicast to both CTAs
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 2 * kEpiWarps);  // the pair's epilogue warps
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before either touches the other's
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t peer_abort = map_to_rank(smem_u32(const_cast<int *>(abort_flag)), rank ^ 1u);

    const int pair = static_cast<int>(blockIdx.x) >> 1;
    const int num_pairs = static_cast<int>(gridDim.x) >> 1;
    const int tiles_m = (p.M + 2 * P_BM - 1) / (2 * P_BM);
    const int num_tiles = p.pair_main_tiles + tiles_m * p.pair_tail_n;

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
            if (p.pair_tail_n > 0)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_bt)) : "memory");
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;  // even CTA: stages armed, their parity
            bool ok = true;
            for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
                const PairTile t = pair_tile(p, tile, tiles_m);
                const bool tail = t.w != P_BN;
                // bytes of one stage in each CTA: its A rows and its half of the tile's columns
                const uint32_t stage_tx = kPABytes + static_cast<uint32_t>(t.w / 2) * BK;
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.wait_cycles,
                                   peer_abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + stage * kPStageBytes;
                    if (leader) {
                        mbar_expect_tx(full_bar(stage), 2 * stage_tx);
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    }
                    const uint32_t fb = map_to_rank(full_bar(stage), 0);
                    tma_load_2d_pair(sa, &tmap_a, kb * BK, t.mt * 2 * P_BM + static_cast<int>(rank) * P_BM, fb);
                    tma_load_2d_pair(sa + kPABytes, tail ? &tmap_bt : &tmap_b, kb * BK,
                                     t.n0 + static_cast<int>(rank) * (t.w / 2), fb);
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // the even CTA's full barriers count both CTAs' copies: every
            // armed stage lands before either CTA passes the final cluster
            // barrier
            for (int s = 0; s < P_STAGES; ++s)
                if (armed & (1u << s)) mbar_wait_drain(full_bar(s), (armed_parity >> s) & 1u, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            if (p.stall & kStallMma)
                ok = mbar_wait(done_bar, 0, abort_flag, p.status, p.wait_cycles, peer_abort);
            for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status, p.wait_cycles,
                               peer_abort))
                    break;
                tc_fence_after();
                const uint32_t idesc = tile < p.pair_main_tiles ? kIdescPair : p.idesc_tail;
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * P_BN);
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!mbar_wait_fast(full_bar(stage), phase, abort_flag, p.status, p.wait_cycles,
                                        peer_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + stage * kPStageBytes;
                    const uint64_t da = sw128_desc(sa), db = sw128_desc(sa + kPABytes);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        mma_f8_pair(d_tmem, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    commit_pair(empty_bar(stage));
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                commit_pair(tfull_bar(acc));
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // every MMA issued has retired (all tcgen05 operations of this
            // kernel use the pair form; the peer's copy of the barrier is unused)
            commit_pair(done_bar);
            mbar_wait_drain(done_bar, 0, p.status);
        }
        __syncwarp();
    } else {
        const int quarter = warp & 3;  // the TMEM lanes this warp may read
        const int grp = (warp - 2) >> 2;  // its share of each tile's 32-column chunks
        const int row = static_cast<int>(rank) * P_BM + quarter * 32 + lane;  // row in the pair tile
        const float sa0 = __ldg(p.a_scale);
        const float sw0 = __ldg(p.w_scale);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = pair; tile < num_tiles; tile += num_pairs) {
            const PairTile t = pair_tile(p, tile, tiles_m);
            if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.status, p.wait_cycles, peer_abort))
                break;
            tc_fence_after();
            const int m = t.mt * 2 * P_BM + row;
            const bool row_ok = m < p.M;
            const float sa = p.a_per_token ? (row_ok ? __ldg(p.a_scale + m) : 0.0f) : sa0;
            const float sa_sw = sa * sw0;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * P_BN);
            const int chunks = t.w / 32;
#pragma unroll 1
            for (int c = grp * chunks / kEpiGroups; c < (grp + 1) * chunks / kEpiGroups; ++c) {
                uint32_t r[32];
                tmem_ld32(taddr + static_cast<uint32_t>(c * 32), r);
                const int n0 = t.n0 + c * 32;
                if (row_ok && n0 < p.N) store_row_chunk(p, r, m, n0, sa, sa_sw, p.w_scale);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(tempty_bar(acc));
                else
                    mbar_arrive_remote(map_to_rank(tempty_bar(acc), 0));
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    // every copy, MMA and TMEM read of the pair is finished before TMEM is
    // released and before either CTA's shared memory goes away
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

// 2-D map over a row-major [rows, K] uint8 matrix, box BK x box_rows, 128B swizzle
int make_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows) {
    return make_kmajor_map(map, ptr, rows, K, BK, box_rows);
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_smem_set[kMaxDevices];

int ensure_smem_attr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8L_ECUDA;
    if (g_smem_set[dev].load(std::memory_order_acquire)) return FP8L_OK;
    if (cudaFuncSetAttribute(gemm_f8_tcgen05, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_f8_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPSmemBytes)) != cudaSuccess)
        return FP8L_ECUDA;
    g_smem_set[dev].store(1, std::memory_order_release);
    return FP8L_OK;
}

// Tile plan of the CTA-pair kernel.  256 x 256 tiles fill whole rounds of
// the SM pairs; the columns left over become tiles a multiple of 32 narrower
// so that the last round spreads over the pairs instead of leaving most of
// them idle (M = 1024, N = 10240: 160 tiles on 76 pairs would take three
// rounds, the third with 8 tiles).  Cost model: a tile w columns wide costs
// max(w, kTailFloor) / 256 of a full tile (its A tile is loaded whatever its
// width); the plan minimises the most loaded pair's cost, widest tail first
// among equals, and keeps 256-wide tiles throughout unless that is beaten.
constexpr int kTailFloor = 96;

struct PairPlan {
    int main_tiles, n_main, tail_w, tail_n;
};

PairPlan plan_pair(int tiles_m, int N, int pairs) {
    const int nb = (N + P_BN - 1) / P_BN;
    const int total = tiles_m * nb;
    PairPlan best{total, nb * P_BN, 0, 0};
    auto cost = [&](int main_tiles, int tail_tiles, int w) {
        const int mr = main_tiles % pairs, tr = tail_tiles % pairs;
        const int wc = w > kTailFloor ? w : kTailFloor;
        int worst = 0;  // in 1/256 of a full tile
        for (int q = 0; q < pairs; ++q) {
            const int mc = main_tiles / pairs + (q < mr ? 1 : 0);
            const int d = (q - mr + pairs) % pairs;  // tail tiles start after the last main one
            const int tc = tail_tiles / pairs + (d < tr ? 1 : 0);
            const int c = mc * P_BN + tc * wc;
            worst = c > worst ? c : worst;
        }
        return worst;
    };
    if (pairs < 1 || total % pairs == 0) return best;
    int best_cost = cost(total, 0, P_BN);
    const int rounds = total / pairs;
    int c = (rounds * pairs) / tiles_m;  // whole 256-column blocks before the tail
    if (c > nb) c = nb;
    const int rem = N - c * P_BN;
    if (rem <= 0) return best;
    for (int w = P_BN - 32; w >= 32; w -= 32) {
        const int tail_n = (rem + w - 1) / w;
        const int cst = cost(c * tiles_m, tail_n * tiles_m, w);
        if (cst < best_cost) {
            best_cost = cst;
            best = PairPlan{c * tiles_m, c * P_BN, w, tail_n};
        }
    }
    return best;
}

// groups == 0: one product of w [N, K]; groups > 0: w is [groups, N, K] and
// group_offs the device row offsets of the experts (grouped mode).  Products
// with enough tiles to fill the SMs run the CTA-pair kernel unless
// single_sm; grouped products and small-M split-K run the single-SM kernel.
int launch_tcgen05(const uint8_t *a, const uint8_t *w, int M, int N, int K, const float *a_scale,
                   int a_per_token, const float *w_scale, int w_per_channel,
                   const float *out_scale, void *y,
                   int out_dtype, unsigned *status, int sms, cudaStream_t stream,
                   const int *group_offs = nullptr, int groups = 0, bool single_sm = false,
                   bool pdl = false) {
    CUtensorMap ma, mb;
    const bool pair_ok = groups == 0 && !single_sm && sms >= 2 &&
                         int64_t((M + BM - 1) / BM) * ((N + BN - 1) / BN) * 2 > sms;
    if (make_map(&ma, a, M, K, BM) != FP8L_OK) return FP8L_ECUDA;
    if (make_map(&mb, w, int64_t(groups > 0 ? groups : 1) * N, K, pair_ok ? P_BN / 2 : BN) != FP8L_OK)
        return FP8L_ECUDA;
    if (ensure_smem_attr() != FP8L_OK) return FP8L_ECUDA;
    GemmParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_m_blocks = (M + BM - 1) / BM;
    p.num_n_blocks = (N + BN - 1) / BN;
    p.num_k_blocks = (K + BK - 1) / BK;
    p.a_scale = a_scale;
    p.w_scale = w_scale;
    p.w_per_channel = w_per_channel;
    p.a_per_token = a_per_token;
    p.out_scale = out_scale;
    p.y = y;
    p.out_dtype = out_dtype;
    p.status = status;
    p.group_offs = group_offs;
    p.num_groups = groups;
    const WaitConfig wc = wait_config();
    p.wait_cycles = wc.cycles;
    p.stall = wc.stall;
    p.pair_main_tiles = 0;
    p.pair_n_main = 0;
    p.pair_tail_w = 0;
    p.pair_tail_n = 0;
    p.idesc_tail = 0;
    if (pair_ok) {
        const int tiles_m = (M + 2 * P_BM - 1) / (2 * P_BM);
        const PairPlan plan = plan_pair(tiles_m, N, sms / 2);
        p.pair_main_tiles = plan.main_tiles;
        p.pair_n_main = plan.n_main;
        p.pair_tail_w = plan.tail_w;
        p.pair_tail_n = plan.tail_n;
        // kind::f8f6f4, D f32, E4M3 K-major operands, N = tail width, M = 256
        p.idesc_tail = (1u << 4) | (static_cast<uint32_t>(plan.tail_w >> 3) << 17) |
                       (static_cast<uint32_t>(256 >> 4) << 24);
        CUtensorMap mbt = mb;
        if (plan.tail_n > 0 && make_map(&mbt, w, N, K, plan.tail_w / 2) != FP8L_OK) return FP8L_ECUDA;
        const int64_t pair_tiles = int64_t(plan.main_tiles) + int64_t(tiles_m) * plan.tail_n;
        const int64_t pairs = pair_tiles < sms / 2 ? pair_tiles : sms / 2;
        p.split = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kPSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 2 : 1;
        if (cudaLaunchKernelEx(&cfg, gemm_f8_pair, ma, mb, mbt, p) != cudaSuccess) return FP8L_ECUDA;
        return launch_status();
    }
    // grouped: each expert adds at most one partial block to ceil(M / BM)
    const int64_t tiles = (int64_t(p.num_m_blocks) + groups) * p.num_n_blocks;
    // Few tiles (small M): a cluster of `split` CTAs per tile splits K so
    // that most SMs stream weights; otherwise one persistent CTA per SM.
    int split = 1;
    if (groups == 0 && tiles * 2 <= sms) {
        split = static_cast<int>(sms / tiles);
        if (split > kMaxSplit) split = kMaxSplit;
        if (split > p.num_k_blocks) split = p.num_k_blocks;
        if (split < 1) split = 1;
    }
    p.split = split;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split > 1 ? tiles * split : (tiles < sms ? tiles : sms)), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
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
    if (pdl) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    if (cudaLaunchKernelEx(&cfg, gemm_f8_tcgen05, ma, mb, p) != cudaSuccess) return FP8L_ECUDA;
    return launch_status();
}

}  // namespace
}  // namespace fp8l

namespace fp8l {
namespace {

// The kernel fp8_scaled_mm runs for FP8L_KERNEL_AUTO (per-shape times of the
// three kernels on GB300, each product alone over rotating operand copies):
//   - weight streaming on the CUDA cores for few tokens and small weights
//     (16 MiB at up to 16 tokens, 24 MiB at up to 4), where its shorter
//     start-up wins (4096 x 4096: 4.9 us against 6.4 us at M = 1);
//   - the swapped-operand tcgen05 product up to 128 tokens (M = 16 at
//     28672 x 4096: 21.5 us against 31.6 us streamed on the CUDA cores and
//     31.8 us on token x channel tiles), except above 64 tokens with 256 MiB
//     or more of weights, where the token x channel tiles read the
//     activations from L2 half as often (M = 128, 57344 x 8192: 87.7 us
//     against 93.1 us);
//   - token x channel tiles otherwise.
unsigned choose_kernel(int64_t M, int64_t N, int64_t K) {
    const int64_t wbytes = N * K;
    if ((M <= 4 && wbytes <= (int64_t(24) << 20)) || (M <= 16 && wbytes <= (int64_t(16) << 20)))
        return FP8L_KERNEL_STREAM;
    if (M <= 128 && !(M > 64 && wbytes >= (int64_t(256) << 20))) return FP8L_KERNEL_SWAPPED;
    return FP8L_KERNEL_TILED;
}

}  // namespace
}  // namespace fp8l

extern "C" unsigned fp8_scaled_mm_kernel(int64_t M, int64_t N, int64_t K, unsigned flags) {
    const unsigned k = flags & FP8L_KERNEL_MASK;
    if (k != FP8L_KERNEL_AUTO) return k;
    return fp8l::choose_kernel(M, N, K);
}

extern "C" int fp8_scaled_mm(const uint8_t *a, const uint8_t *w, int64_t M, int64_t N, int64_t K,
                             const float *a_scale, const float *w_scale, int w_per_channel,
                             const float *out_scale, void *y, int out_dtype, void *workspace,
                             unsigned flags, void *stream) {
    using namespace fp8l;
    if (out_dtype != FP8L_F16 && out_dtype != FP8L_BF16 && out_dtype != FP8L_E4M3)
        return FP8L_EINVAL;
    if ((flags & ~(FP8L_WEIGHTS_STABLE | FP8L_A_PER_TOKEN | FP8L_SINGLE_SM_TILES | FP8L_KERNEL_MASK)) != 0u)
        return FP8L_EINVAL;
    unsigned kernel = flags & FP8L_KERNEL_MASK;
    if (kernel == FP8L_KERNEL_SWAPPED && M > 128) return FP8L_ESHAPE;
    if (a_scale == nullptr || w_scale == nullptr || workspace == nullptr || w == nullptr)
        return FP8L_EINVAL;
    if (out_dtype == FP8L_E4M3 && out_scale == nullptr) return FP8L_EINVAL;
    if (M < 0 || M > 0x7FFFFFFF || N <= 0 || K <= 0 || N > (1 << 20) || K > (1 << 20) ||
        N % 16 != 0 || K % 16 != 0)
        return FP8L_ESHAPE;
    if (M > 0 && (a == nullptr || y == nullptr)) return FP8L_EINVAL;
    auto misaligned4 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) != 0; };
    if (!aligned16(w) || !aligned16(workspace) || (M > 0 && (!aligned16(a) || !aligned16(y))) ||
        misaligned4(a_scale) || misaligned4(w_scale) ||
        (out_dtype == FP8L_E4M3 && misaligned4(out_scale)))
        return FP8L_EALIGN;
    int sms = 0;
    int st = check_device(&sms);
    if (st != FP8L_OK) return st;
    if (M == 0) return FP8L_OK;
    cudaStream_t s = as_stream(stream);
    const int pc = w_per_channel ? 1 : 0;
    const int pt = (flags & FP8L_A_PER_TOKEN) != 0u ? 1 : 0;
    const bool stable = (flags & FP8L_WEIGHTS_STABLE) != 0u;
    if (kernel == FP8L_KERNEL_AUTO) kernel = choose_kernel(M, N, K);
    if (kernel == FP8L_KERNEL_STREAM)
        return launch_skinny_e4m3(a, w, static_cast<int>(M), static_cast<int>(N),
                                  static_cast<int>(K), a_scale, pt, w_scale, pc, out_scale, y,
                                  out_dtype, stable, s);
    if (kernel == FP8L_KERNEL_SWAPPED)
        return launch_swapab(a, w, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                             a_scale, pt, w_scale, pc, out_scale, y, out_dtype,
                             status_word(workspace), sms, stable, s);
    return launch_tcgen05(a, w, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                          a_scale, pt, w_scale, pc, out_scale, y, out_dtype,
                          status_word(workspace), sms, s, nullptr, 0,
                          (flags & FP8L_SINGLE_SM_TILES) != 0u, stable);
}

extern "C" int fp8_grouped_mm(const uint8_t *a, const uint8_t *w, const int32_t *group_offsets,
                              int64_t num_groups, int64_t M, int64_t N, int64_t K,
                              const float *a_scale, const float *w_scale, int w_per_channel,
                              const float *out_scale, void *y, int out_dtype, void *workspace,
                              unsigned flags, void *stream) {
    using namespace fp8l;
    if (out_dtype != FP8L_F16 && out_dtype != FP8L_BF16 && out_dtype != FP8L_E4M3)
        return FP8L_EINVAL;
    if ((flags & ~(FP8L_WEIGHTS_STABLE | FP8L_A_PER_TOKEN)) != 0u) return FP8L_EINVAL;
    if (a_scale == nullptr || w_scale == nullptr || workspace == nullptr || w == nullptr ||
        group_offsets == nullptr)
        return FP8L_EINVAL;
    if (out_dtype == FP8L_E4M3 && out_scale == nullptr) return FP8L_EINVAL;
    if (num_groups < 1 || num_groups > kMaxGroups || M < 0 || M > 0x7FFFFFFF || N <= 0 ||
        K <= 0 || N > (1 << 20) || K > (1 << 20) || N % 16 != 0 || K % 16 != 0 ||
        num_groups * N > 0x7FFFFFFF)
        return FP8L_ESHAPE;
    if (M > 0 && (a == nullptr || y == nullptr)) return FP8L_EINVAL;
    auto misaligned4 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) != 0; };
    if (!aligned16(w) || !aligned16(workspace) || (M > 0 && (!aligned16(a) || !aligned16(y))) ||
        misaligned4(a_scale) || misaligned4(w_scale) || misaligned4(group_offsets) ||
        (out_dtype == FP8L_E4M3 && misaligned4(out_scale)))
        return FP8L_EALIGN;
    int sms = 0;
    int st = check_device(&sms);
    if (st != FP8L_OK) return st;
    if (M == 0) return FP8L_OK;
    return launch_tcgen05(a, w, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                          a_scale, (flags & FP8L_A_PER_TOKEN) != 0u ? 1 : 0, w_scale,
                          w_per_channel ? 1 : 0, out_scale, y, out_dtype, status_word(workspace),
                          sms, as_stream(stream), group_offsets, static_cast<int>(num_groups), false,
                          (flags & FP8L_WEIGHTS_STABLE) != 0u);
}

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

#include "quant_device.cuh"

namespace fp8l {
namespace {

constexpr int kThreads = 256;

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


template <int DT, bool DYN>
__global__ void __launch_bounds__(kTThreads, 1)
quant_tma_kernel(const void *__restrict__ x, int64_t numel, uint8_t *__restrict__ q,
                 float *__restrict__ scale, unsigned *epoch, unsigned *arrive, unsigned *amax,
                 unsigned *status, int piece_words, int total_pieces, int stages, int keep_pieces,
                 long long wait_cycles, unsigned stall) {
    extern __shared__ __align__(128) uint4 stage_mem[];
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ uint32_t red[33];
    __shared__ int abort_sh;
    __shared__ unsigned epoch_sh;
    constexpr int EB = Elt<DT>::kBytes;
    constexpr int EPW = 16 / EB;  // elements per 16-byte word
    // a product launched as a programmatic dependent may be scheduled now;
    // it waits for this grid's writes itself
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
            if (q_mbar_wait(smem_u32(&full[s]), (par >> s) & 1u, wait_cycles))
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
        uint32_t mm = m;
        // a single block has the maximum already and skips the barrier words
        // (testing the time-out path: one arrival more than the grid has)
        const bool barrier = G > 1 || (stall & kStallGrid) != 0u;
        const unsigned expect = gridDim.x + ((stall & kStallGrid) ? 1u : 0u);
        if (barrier && !grid_max(arrive + pair, amax + pair, m, status, &mm, expect, wait_cycles))
            return;  // no copy in flight here
        sc = scale_from_amax(mag_bits_to_float<DT>(mm));
        if (blockIdx.x == 0 && tid == 0) {
            *scale = sc;
            if (barrier) *epoch = epoch_sh + 1u;  // every block read the counter before arriving
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
            if (pending & (1u << i)) q_mbar_wait(smem_u32(&full[i]), (par >> i) & 1u, kDefaultWaitCycles);
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
    const WaitConfig wc = wait_config();
    cudaError_t e;
    if (dynamic)
        e = cudaLaunchKernelEx(&cfg, quant_tma_kernel<DT, true>, x, numel, q, scale, epoch_word(workspace),
                               arrive_words(workspace), amax_words(workspace), status_word(workspace),
                               p.piece_words, static_cast<int>(p.total_pieces), p.stages, p.keep_pieces,
                               wc.cycles, wc.stall);
    else
        e = cudaLaunchKernelEx(&cfg, quant_tma_kernel<DT, false>, x, numel, q, scale,
                               static_cast<unsigned *>(nullptr), static_cast<unsigned *>(nullptr),
                               static_cast<unsigned *>(nullptr),
                               workspace ? status_word(workspace) : static_cast<unsigned *>(nullptr),
                               p.piece_words, static_cast<int>(p.total_pieces), p.stages, 0,
                               wc.cycles, wc.stall);
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
#include <mutex>

namespace fp8l {
namespace {

// 2048 partial maxima, then one ticket word that is zero between calls (zero
// at load, and every call leaves it at zero)
constexpr int kNoallocMaxPartials = 2048;
static __device__ __align__(256) float g_noalloc_partials[kNoallocMaxPartials + 64];

constexpr int kNoallocMaxDevices = 64;
struct NoallocSlot {
    std::mutex mu;
    unsigned long long ctx_id = 0;  // context the address below belongs to
    float *ptr = nullptr;
};
NoallocSlot g_noalloc[kNoallocMaxDevices];

// Device address of g_noalloc_partials in the context current on this
// thread.  In host code the array's name is only a host-side stand-in, so the
// address comes from cudaGetSymbolAddress, with the device current.  It is
// kept per device together with the id of the context it was taken in and
// looked up again when another context is current (a context created after
// cudaDeviceReset, or a caller's own context on that device).
int noalloc_scratch(float **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8L_ECUDA;
    if (dev < 0 || dev >= kNoallocMaxDevices) return FP8L_EUNSUPPORTED;
    NoallocSlot &slot = g_noalloc[dev];
    std::lock_guard<std::mutex> lock(slot.mu);
    unsigned long long id = 0;
    if (current_context_id(&id) != FP8L_OK) return FP8L_ECUDA;
    if (slot.ptr == nullptr || id == 0 || id != slot.ctx_id) {
        void *addr = nullptr;  // the lookup makes the device's context current if none is
        if (cudaGetSymbolAddress(&addr, g_noalloc_partials) != cudaSuccess || addr == nullptr)
            return FP8L_ECUDA;
        if (current_context_id(&id) != FP8L_OK || id == 0) return FP8L_ECUDA;
        slot.ptr = static_cast<float *>(addr);
        slot.ctx_id = id;
    }
    *out = slot.ptr;
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

// Entry points that are not tied to one kernel: workspace size, status word,
// error strings, device check; the tensor-map encoder of the TMA kernels.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace fp8l {

namespace {
std::atomic<long long> g_wait_cycles{0};
std::atomic<unsigned> g_stall{0};
}  // namespace

WaitConfig wait_config() {
    const long long c = g_wait_cycles.load(std::memory_order_relaxed);
    return WaitConfig{c > 0 ? c : kDefaultWaitCycles, g_stall.load(std::memory_order_relaxed)};
}

namespace {
constexpr int kMaxDevices = 64;
// 0 = unknown, 1 = supported, 2 = unsupported; SM count beside it
std::atomic<int> g_dev_state[kMaxDevices];
std::atomic<int> g_dev_sms[kMaxDevices];
}  // namespace

int check_device(int *sm_count_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8L_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return FP8L_EUNSUPPORTED;
    int state = g_dev_state[dev].load(std::memory_order_acquire);
    if (state == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FP8L_ECUDA;
        g_dev_sms[dev].store(sms, std::memory_order_relaxed);
        state = (major == 10 && minor == 3) ? 1 : 2;
        g_dev_state[dev].store(state, std::memory_order_release);
    }
    if (sm_count_out) *sm_count_out = g_dev_sms[dev].load(std::memory_order_relaxed);
    return state == 1 ? FP8L_OK : FP8L_EUNSUPPORTED;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}
}  // namespace

int make_kmajor_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_k,
                    int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) return FP8L_ECUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8L_OK : FP8L_ECUDA;
}

namespace {
// Status word of the calls that take no workspace (fp8_w8a16_mm's
// tensor-core kernel): time-outs are recorded here and reported, then
// cleared, by fp8l_read_status together with the workspace's word.
__device__ unsigned g_library_status;

struct StatusSlot {
    std::mutex mu;
    unsigned long long ctx_id = 0;  // context the address below belongs to
    unsigned *ptr = nullptr;
};
constexpr int kStatusMaxDevices = 64;
StatusSlot g_status_slots[kStatusMaxDevices];
}  // namespace

// Device address of g_library_status in the context current on this thread
// (taken with cudaGetSymbolAddress, kept per device with the id of its
// context and looked up again when another context is current).
int library_status_word(unsigned **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8L_ECUDA;
    if (dev < 0 || dev >= kStatusMaxDevices) return FP8L_EUNSUPPORTED;
    StatusSlot &slot = g_status_slots[dev];
    std::lock_guard<std::mutex> lock(slot.mu);
    unsigned long long id = 0;
    if (current_context_id(&id) != FP8L_OK) return FP8L_ECUDA;
    if (slot.ptr == nullptr || id == 0 || id != slot.ctx_id) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_library_status) != cudaSuccess || addr == nullptr)
            return FP8L_ECUDA;
        if (current_context_id(&id) != FP8L_OK || id == 0) return FP8L_ECUDA;
        slot.ptr = static_cast<unsigned *>(addr);
        slot.ctx_id = id;
    }
    *out = slot.ptr;
    return FP8L_OK;
}

int make_tile_map(CUtensorMap *map, const void *ptr, int elem_bytes, int rank, const uint64_t *dims,
                  const uint64_t *strides, const uint32_t *box, bool swizzle128) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr || rank < 1 || rank > 5 || (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 8))
        return FP8L_ECUDA;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = static_cast<cuuint64_t>(dims[i]);
        b[i] = static_cast<cuuint32_t>(box[i]);
        estr[i] = 1;
        if (i + 1 < rank) st[i] = static_cast<cuuint64_t>(strides[i]);
    }
    const CUtensorMapDataType type = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_UINT64;
    CUresult r = enc(map, type,
                     static_cast<cuuint32_t>(rank), const_cast<void *>(ptr), d, st, b, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8L_OK : FP8L_ECUDA;
}

int current_context_id(unsigned long long *id) {
    static std::atomic<PFN_cuCtxGetCurrent_v4000> get_cur{nullptr};
    static std::atomic<PFN_cuCtxGetId_v12000> get_id{nullptr};
    PFN_cuCtxGetCurrent_v4000 fc = get_cur.load(std::memory_order_acquire);
    PFN_cuCtxGetId_v12000 fi = get_id.load(std::memory_order_acquire);
    if (fc == nullptr || fi == nullptr) {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &r1) !=
                cudaSuccess ||
            r1 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) !=
                cudaSuccess ||
            r2 != cudaDriverEntryPointSuccess)
            return FP8L_ECUDA;
        fc = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        fi = reinterpret_cast<PFN_cuCtxGetId_v12000>(q);
        get_cur.store(fc, std::memory_order_release);
        get_id.store(fi, std::memory_order_release);
    }
    CUcontext ctx = nullptr;
    if (fc(&ctx) != CUDA_SUCCESS) return FP8L_ECUDA;
    if (ctx == nullptr) {
        *id = 0;
        return FP8L_OK;
    }
    return fi(ctx, id) == CUDA_SUCCESS ? FP8L_OK : FP8L_ECUDA;
}

namespace {
// Waits for `s` and reads the status word at the start of workspace `ws`.
// A set word is cleared; after a time-out the whole barrier area [0, 32) is
// zeroed too (ticket, call counter, arrival counts, maximum words), since the
// call that gave up may have left them part-way through a grid barrier.
int read_and_clear(void *ws, cudaStream_t s) {
    unsigned host[2] = {0u, 0u};
    unsigned *dev = status_word(ws);
    unsigned *lib = nullptr;
    if (library_status_word(&lib) != FP8L_OK) return FP8L_ECUDA;
    if (cudaMemcpyAsync(&host[0], dev, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&host[1], lib, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return FP8L_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FP8L_ECUDA;
    if (host[0] != 0u) {
        const size_t bytes = (host[0] & kStatusTimeout) ? kBarrierAreaBytes : sizeof(unsigned);
        if (cudaMemsetAsync(ws, 0, bytes, s) != cudaSuccess) return FP8L_ECUDA;
    }
    if (host[1] != 0u && cudaMemsetAsync(lib, 0, sizeof(unsigned), s) != cudaSuccess) return FP8L_ECUDA;
    if ((host[0] | host[1]) != 0u && cudaStreamSynchronize(s) != cudaSuccess) return FP8L_ECUDA;
    return ((host[0] | host[1]) & kStatusTimeout) ? FP8L_ETIMEOUT : FP8L_OK;
}
}  // namespace

}  // namespace fp8l

extern "C" {

size_t fp8l_workspace_bytes(void) { return fp8l::kWorkspaceBytes; }

int fp8l_abi_version(void) { return FP8L_ABI_VERSION; }

const char *fp8l_strerror(int status) {
    switch (status) {
        case FP8L_OK: return "ok";
        case FP8L_EINVAL: return "invalid argument (null pointer, dtype or flag)";
        case FP8L_ESHAPE: return "invalid shape (negative, too large, or not a multiple of 16)";
        case FP8L_EALIGN: return "tensor pointer not 16-byte aligned";
        case FP8L_ECUDA: return "CUDA call or kernel launch failed";
        case FP8L_ETIMEOUT: return "a device-side wait timed out";
        case FP8L_EUNSUPPORTED: return "unsupported device or dtype combination";
        default: return "unknown status";
    }
}

int fp8l_debug_waits(long long wait_cycles, unsigned stall_mask) {
    if (wait_cycles < 0 || (stall_mask & ~(fp8l::kStallMma | fp8l::kStallGrid)) != 0u)
        return FP8L_EINVAL;
    fp8l::g_wait_cycles.store(wait_cycles, std::memory_order_relaxed);
    fp8l::g_stall.store(stall_mask, std::memory_order_relaxed);
    return FP8L_OK;
}

int fp8l_read_status(void *workspace, void *stream) {
    if (workspace == nullptr) return FP8L_EINVAL;
    if (!fp8l::aligned16(workspace)) return FP8L_EALIGN;
    return fp8l::read_and_clear(workspace, fp8l::as_stream(stream));
}

}  // extern "C"

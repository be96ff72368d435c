// Entry points that are not tied to one kernel: workspace size, status word,
// error strings, device check.
#include <atomic>

#include "common.cuh"

namespace fp8l {

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

int fp8l_read_status(void *workspace, void *stream) {
    if (workspace == nullptr) return FP8L_EINVAL;
    if (!fp8l::aligned16(workspace)) return FP8L_EALIGN;
    cudaStream_t s = fp8l::as_stream(stream);
    unsigned host = 0;
    unsigned *dev = fp8l::status_word(workspace);
    if (cudaMemcpyAsync(&host, dev, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return FP8L_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FP8L_ECUDA;
    if (host != 0u) {
        if (cudaMemsetAsync(dev, 0, sizeof(unsigned), s) != cudaSuccess) return FP8L_ECUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return FP8L_ECUDA;
    }
    return (host & fp8l::kStatusTimeout) ? FP8L_ETIMEOUT : FP8L_OK;
}

}  // extern "C"

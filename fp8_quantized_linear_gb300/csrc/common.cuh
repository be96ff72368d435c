// Shared host and device helpers of the FP8 linear library (sm_103a only).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8linear.h"

namespace fp8l {

// ---------------------------------------------------------------------------
// Workspace layout (fp8l_workspace_bytes bytes, zero-filled by the caller once)
//   [0, 4)                   uint32 status word (bit flags below)
//   [4, 8)                   uint32 two-launch quantizer ticket (zero between calls)
//   [8, 12)                  uint32 single-launch quantizer call counter (any value)
//   [16, 24)                 uint32[2] its grid-barrier arrival counts
//   [24, 32)                 uint32[2] its maximum-magnitude words
//                            (the pair of index `counter & 1` is zero when a
//                            call starts; that call clears the other pair)
//   [256, 256 + 4*kMaxParts) float per-block partial maxima (two-launch quantizer)
constexpr size_t kStatusOffset = 0;
constexpr size_t kBarrierAreaBytes = 32;  // [0, 32): status and barrier words
constexpr size_t kPartialsOffset = 256;
constexpr int kMaxPartials = 2048;
constexpr size_t kWorkspaceBytes = kPartialsOffset + sizeof(float) * kMaxPartials;

constexpr unsigned kStatusTimeout = 1u;  // a bounded device-side wait gave up

// Limits of the bounded device-side waits, in SM clock cycles.  The default
// is ~2 s at 2 GHz (a healthy wait takes microseconds).  fp8l_debug_waits may
// shorten the limit of the main waits and make one wait target a barrier
// that nothing completes (testing the time-out path); waits that drain
// copies in flight before a block exits always keep the default.
constexpr long long kDefaultWaitCycles = 4LL << 30;
constexpr unsigned kStallMma = 1u;   // product: the MMA role's first wait never completes
constexpr unsigned kStallGrid = 2u;  // quantizer: the grid barrier waits for one block too many
struct WaitConfig {
    long long cycles;  // limit of the main waits
    unsigned stall;    // kStall* bits
};
WaitConfig wait_config();

// Largest magnitude of OCP E4M3.
constexpr float kE4M3Max = 448.0f;

// ---------------------------------------------------------------------------
// host helpers

inline bool aligned16(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline unsigned *status_word(void *workspace) {
    return reinterpret_cast<unsigned *>(static_cast<char *>(workspace) + kStatusOffset);
}

inline unsigned *ticket_word(void *workspace) {
    return reinterpret_cast<unsigned *>(static_cast<char *>(workspace) + 4);
}

inline unsigned *epoch_word(void *workspace) {
    return reinterpret_cast<unsigned *>(static_cast<char *>(workspace) + 8);
}

inline unsigned *arrive_words(void *workspace) {
    return reinterpret_cast<unsigned *>(static_cast<char *>(workspace) + 16);
}

inline unsigned *amax_words(void *workspace) {
    return reinterpret_cast<unsigned *>(static_cast<char *>(workspace) + 24);
}

inline float *partials(void *workspace) {
    return reinterpret_cast<float *>(static_cast<char *>(workspace) + kPartialsOffset);
}

// FP8L_OK when the current device is compute capability 10.3; caches the
// answer and the SM count per device ordinal.
int check_device(int *sm_count_out);

// Unique id of the CUDA context current on this thread (0 when none is):
// the driver's cuCtxGetId, which never repeats within a process, so a
// context created after cudaDeviceReset gets a new id.
int current_context_id(unsigned long long *id);

// 2-D TMA map over a row-major [rows, K] byte matrix: box box_k x box_rows,
// 128-byte swizzle, zero fill outside the matrix.
int make_kmajor_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_k,
                    int box_rows);

// Device address (in the current context) of the library's own status word,
// where kernels of calls without a workspace record time-outs;
// fp8l_read_status reports and clears it with the workspace's word.
int library_status_word(unsigned **out);

// N-D TMA map (rank <= 5) over 1-, 2- or 8-byte elements: dims and box
// innermost first, strides[i] = bytes between consecutive indices of
// dimension i + 1 (multiples of 16); optional 128-byte swizzle; zero fill
// outside the tensor.
int make_tile_map(CUtensorMap *map, const void *ptr, int elem_bytes, int rank, const uint64_t *dims,
                  const uint64_t *strides, const uint32_t *box, bool swizzle128);

// FP8L_ECUDA if the last launch failed, else FP8L_OK.
inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? FP8L_OK : FP8L_ECUDA;
}

// Launchers shared between translation units.
int launch_skinny_e4m3(const uint8_t *a, const uint8_t *w, int M, int N, int K,
                       const float *a_scale, int a_per_token, const float *w_scale,
                       int w_per_channel, const float *out_scale, void *y, int out_dtype,
                       bool stable_weights, cudaStream_t stream);
// W8A8 for up to 16 tokens of 16-bit x, the per-tensor quantization (static
// a_scale read, or dynamic a_scale written) in the weight-streaming kernel
int launch_skinny_quant(const void *x, int x_dtype, const uint8_t *w, int M, int N, int K,
                        float *a_scale, int dynamic, const float *w_scale, int w_per_channel,
                        const float *out_scale, void *y, int out_dtype, bool stable_weights,
                        cudaStream_t stream);
int launch_w8a16_tc(const void *x, int x_dtype, const uint8_t *w, bool packed, const float *w_scale,
                    int M, int N, int K, void *y, unsigned *status, int sms, bool stable,
                    cudaStream_t stream);
int launch_swapab(const uint8_t *a, const uint8_t *w, int M, int N, int K, const float *a_scale,
                  int a_per_token, const float *w_scale, int w_per_channel,
                  const float *out_scale, void *y, int out_dtype, unsigned *status, int sms,
                  bool stable, cudaStream_t stream);

// ---------------------------------------------------------------------------
// device helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte load of streamed weights: bypasses L1 and has L2 fetch the whole
// 256-byte segment around it (the neighbouring chunks of the row are read by
// other warps moments later).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

}  // namespace fp8l

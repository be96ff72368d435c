// Device helpers of the weight-streaming kernels (skinny.cu, skinny_quant.cu).
#pragma once

#include <stdint.h>

namespace fp8l {

// E4M3 x E4M3 tensor-core step with fp32 accumulation: A 16 x 32 (rows of
// W), B 32 x 8 (tokens)
__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Loads of data the preceding kernel on the stream may write (activations,
// activation and output scales).  Coherent loads in volatile asm: they stay
// after griddepcontrol.wait, and the non-coherent read-only path (whose
// loads the compiler may treat as invariant and move ahead of the wait) is
// only for data no kernel in flight writes, such as the stable weights.
__device__ __forceinline__ uint4 ld_act16(const void *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_act_f32(const float *p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

}  // namespace fp8l

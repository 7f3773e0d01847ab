// kivi_device.cuh -- device helpers shared by the KIVI sm_103a kernels.
//
// Nothing here is shared with the CPU oracle: the conversions use the
// hardware's IEEE fp16/fp32 instructions and every rounding step is an
// explicit __f*_rn intrinsic, so the compiler can neither fuse a multiply
// into an add nor reassociate.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "kivi_launch.h"

namespace kivi {

constexpr float kMagic = 8388608.0f;  // 2^23

// Number of representable codes minus one: 2^bits - 1.
template <int BITS>
struct Levels {
    static constexpr uint32_t value = (1u << BITS) - 1u;
};

// --- packed fp32x2 arithmetic (sm_100+): two IEEE round-to-nearest ops per
// instruction, each lane rounded exactly like the scalar __f*_rn intrinsic.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pk(float a, float b) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 upk(f32x2 v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// --- programmatic dependent launch. Every kernel calls pdl_wait() before its
// first global access, so it may be launched while the previous kernel on
// the stream is still running; pdl_trigger() lets the next one be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace kivi

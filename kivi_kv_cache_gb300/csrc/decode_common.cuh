// decode_common.cuh -- PTX helpers shared by the decode kernels: cp.async
// staging, ldmatrix, the m16n8k16 fp16 MMA, the units of code operands
// (fp16 subnormals by masking), the fp16 hi/lo split of fp32 operands, and
// thread-block cluster access.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "kivi_device.cuh"

namespace kivi {
namespace dec {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy; with fill == false nothing is read and 16 zero bytes land.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool fill) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(fill ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp16 hi (lo == false) or lo (lo == true) part of the pair (x, y):
// hi = fp16(x), lo = fp16(x - hi) (x - hi is exact in fp32). One mixed-
// precision fma per element, x + hi * m with the fp16 m = -1 (lo) or 0 (hi),
// gives x - hi or x itself, and one conversion rounds either to fp16.
__device__ __forceinline__ uint32_t split_pair(float x, float y, bool lo) {
    const unsigned short m = lo ? 0xbc00 : 0;  // fp16 -1 or +0
    uint32_t r;
    asm("{\n\t.reg .b32 h;\n\t.reg .b16 hl, hh;\n\t.reg .f32 rx, ry;\n\t"
        "cvt.rn.f16x2.f32 h, %2, %1;\n\t"
        "mov.b32 {hl, hh}, h;\n\t"
        "fma.rn.f32.f16 rx, hl, %3, %1;\n\t"
        "fma.rn.f32.f16 ry, hh, %3, %2;\n\t"
        "cvt.rn.f16x2.f32 %0, ry, rx;\n\t}"
        : "=r"(r)
        : "f"(x), "f"(y), "h"(m));
    return r;
}

// Code operands of the decode MMAs: a code masked in place within a 16-bit
// half is an fp16 subnormal, exact as an MMA operand: a nibble at bit 4j is
// c 16^j 2^-24, a crumb at bit 2j is c 4^j 2^-24. The per-position factor
// 16^j or 4^j is folded into the other operand (scores) or into the units of
// the accumulator (P.V): kOUnit4[u] for nibble position u, kOUnit2[k] for
// crumb position k.
__device__ constexpr float kOUnit4[2] = {0x1p-24f, 0x1p-20f};
__device__ constexpr float kOUnit2[4] = {0x1p-24f, 0x1p-22f, 0x1p-20f, 0x1p-18f};

// 2^e as fp32 for e in [-126, 127]
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

// exponent E with m * 2^E < 2^14 (m >= 0); 0 for m == 0, clamped
__device__ __forceinline__ int safe_exp(float m) {
    if (!(m > 0.f)) return 0;
    const int ex = ((__float_as_int(m) >> 23) & 0xff) - 127;  // floor(log2 m) for normal m
    const int e = 13 - ex;
    return e < -100 ? -100 : (e > 100 ? 100 : e);
}

// thread-block cluster: rank of this CTA, the cluster-wide barrier (release /
// acquire: shared-memory writes before it are visible to every CTA of the
// cluster after it), and a load from another CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster(const float* p, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// barrier over `threads` threads (a multiple of 32) with named barrier `id`
// (1..15; 0 is the CTA-wide __syncthreads barrier)
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace dec
}  // namespace kivi

// decode_merge.cuh -- the split merge shared by the decode kernels.
//
// The cached tokens of one (batch, KV head) are split over n_split CTAs
// (VeloxQuant-MLX benchmarks page, "KV-Cache Kernel Roofline": one CTA per
// head leaves the GPU idle). Each CTA leaves a partial (o, m, l) in the
// workspace and takes a ticket from the head's counter. The CTA with the last
// ticket sets the counter back to zero, so the workspace is ready for the
// next call, and merges the partials:
//     M = max_s m_s,  out = sum_s o_s 2^(m_s - M) / sum_s l_s 2^(m_s - M).
// The merge runs inside the decode launch, so no second kernel is needed.
#pragma once

#include <math.h>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

// Ticket add with acquire-release semantics at GPU scope: the release half
// publishes every write this thread has observed (the CTA's partial stores,
// ordered before it by the CTA barrier); the acquire half makes the writes
// published by earlier tickets visible to the ticket holder.
__device__ __forceinline__ unsigned ticket_add_acq_rel(unsigned* p) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
    return old;
}

// Called by all threads of the CTA after its partials are written. Returns
// true in the CTA that must merge; *flag is a shared-memory int.
__device__ __forceinline__ bool take_last_ticket(const DecodeArgs& a, int bh, int* flag) {
    __syncthreads();  // every thread's partial stores precede thread 0's ticket
    if (threadIdx.x == 0) {
        const unsigned ticket = ticket_add_acq_rel(a.counters + bh);
        const bool last = ticket == (unsigned)(a.n_split - 1);
        if (last) atomicExch(a.counters + bh, 0u);  // ready for the next call
        *flag = last;
    }
    __syncthreads();  // the ticket holder's acquire covers its CTA's reads after this barrier
    return *flag != 0;
}

// VW consecutive floats (1, 2, 4 or 8; 4 VW-byte aligned) read through L2
// (ld.global.cg: other CTAs of this launch wrote them), or zeros.
template <int VW>
__device__ __forceinline__ void ldcg_vec(float (&v)[VW], const float* p, bool on) {
    if constexpr (VW == 1) {
        v[0] = on ? __ldcg(p) : 0.f;
    } else if constexpr (VW == 2) {
        const float2 x = on ? __ldcg(reinterpret_cast<const float2*>(p)) : make_float2(0.f, 0.f);
        v[0] = x.x, v[1] = x.y;
    } else {
#pragma unroll
        for (int e = 0; e < VW / 4; ++e) {
            const float4 x = on ? __ldcg(reinterpret_cast<const float4*>(p) + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[4 * e] = x.x, v[4 * e + 1] = x.y, v[4 * e + 2] = x.z, v[4 * e + 3] = x.w;
        }
    }
}

// One head of the merge below: warp-level, channel slice sl of the row.
template <int NW, int D>
__device__ __forceinline__ void merge_one(const DecodeArgs& a, long long bq, int sl, int lane) {
    constexpr int SL = NW >= 4 ? NW / 4 : 1;  // channel slices per row
    constexpr int CW = D / SL;       // channels per slice
    constexpr int VW = CW / 32;      // channels per lane
    static_assert(VW >= 1 && VW <= 8 && CW % 32 == 0, "a slice is 32 to 256 channels");
    constexpr int CHUNK = VW <= 2 ? 40 : (VW == 4 ? 16 : 8);  // rows of the first round trip
    constexpr int BLK = VW <= 2 ? 32 : CHUNK;                  // rows per later round trip
    const int n = a.n_split;
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + bq * n;
    const float* po = a.part_o + bq * n * D + sl * CW + lane * VW;
    float v[CHUNK][VW];
#pragma unroll
    for (int k = 0; k < CHUNK; ++k) ldcg_vec<VW>(v[k], po + (long long)k * D, k < n);
    const float2 x0 = lane < n ? __ldcg(ml + lane) : make_float2(-INFINITY, 0.f);
    const float2 x1 = lane + 32 < n ? __ldcg(ml + lane + 32) : make_float2(-INFINITY, 0.f);
    float M = fmaxf(x0.x, x1.x);
    for (int s = lane + 64; s < n; s += 32) M = fmaxf(M, __ldcg(ml + s).x);
    M = warp_max(M);
    const float w0 = x0.x == -INFINITY ? 0.f : exp2f(x0.x - M);  // 0 past the last split
    const float w1 = x1.x == -INFINITY ? 0.f : exp2f(x1.x - M);
    float L = fmaf(x0.y, w0, x1.y * w1);
    float acc[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) acc[e] = 0.f;
#pragma unroll
    for (int k = 0; k < CHUNK; ++k) {
        const float wk = __shfl_sync(0xffffffffu, k < 32 ? w0 : w1, k & 31);
#pragma unroll
        for (int e = 0; e < VW; ++e) acc[e] = fmaf(v[k][e], wk, acc[e]);
    }
    for (int s0 = CHUNK; s0 < n; s0 += BLK) {
        // splits s0 .. s0 + BLK - 1: rows, and the weights in lanes 0 .. BLK - 1
        const int s = s0 + lane;
        float2 x = lane < BLK && s < n ? __ldcg(ml + s) : make_float2(-INFINITY, 0.f);
        const float wt = x.x == -INFINITY ? 0.f : exp2f(x.x - M);
        if (s >= 64) L = fmaf(x.y, wt, L);  // splits below 64 are in w0, w1 already
#pragma unroll
        for (int k = 0; k < BLK; ++k) ldcg_vec<VW>(v[k], po + (long long)(s0 + k) * D, s0 + k < n);
#pragma unroll
        for (int k = 0; k < BLK; ++k) {
            const float wk = __shfl_sync(0xffffffffu, wt, k);
#pragma unroll
            for (int e = 0; e < VW; ++e) acc[e] = fmaf(v[k][e], wk, acc[e]);
        }
    }
    L = warp_sum(L);
    const float r = 1.0f / L;
    float* out = a.out + bq * D + sl * CW + lane * VW;
    if constexpr (VW == 1) {
        out[0] = acc[0] * r;
    } else if constexpr (VW == 2) {
        *reinterpret_cast<float2*>(out) = make_float2(acc[0] * r, acc[1] * r);
    } else {
#pragma unroll
        for (int e = 0; e < VW / 4; ++e)
            reinterpret_cast<float4*>(out)[e] =
                make_float4(acc[4 * e] * r, acc[4 * e + 1] * r, acc[4 * e + 2] * r, acc[4 * e + 3] * r);
    }
}

// Merge of the n_split partials of query heads bq0 .. bq0 + nheads - 1
// (nheads <= 4) by the NW warps (2, 4 or 8) of the CTA holding the last
// ticket: with 4 or 8 warps, warp w takes head w % 4 and channel slice w / 4
// of the NW / 4 slices of a row; with 2 warps, warp w takes heads w and
// w + 2 in turn, whole rows. A lane holds VW consecutive channels of the
// slice.
// The first CHUNK partial rows (up to 80 registers' worth: 40 rows at
// VW <= 2) are requested together with the (m, l) pairs of splits lane and
// lane + 32, so up to CHUNK splits cost one L2 round trip; row s takes its
// weight 2^(m_s - M) from lane s % 32 by shuffle. Splits past CHUNK follow in
// blocks of 32. No barrier inside.
template <int NW, int D>
__device__ __forceinline__ void merge_splits(const DecodeArgs& a, long long bq0, int nheads, int warp, int lane) {
    static_assert(NW == 2 || NW == 4 || NW == 8, "2, 4 or 8 warps");
    if (NW == 2) {  // each warp merges two heads in turn
        for (int h = warp; h < nheads; h += 2) merge_one<NW, D>(a, bq0 + h, 0, lane);
        return;
    }
    const int h = warp & 3, sl = warp >> 2;
    if (h >= nheads) return;
    merge_one<NW, D>(a, bq0 + h, sl, lane);
}

}  // namespace kivi

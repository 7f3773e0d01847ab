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

// Float4 vectors of a head-dim-D row per lane: lane l holds channels
// 4 (l + 32 v) .. + 3 for v < kMergeVec; at D = 64 only lanes 0..15 hold one.
template <int D>
struct MergeShape {
    static constexpr int kVec = D >= 128 ? D / 128 : 1;
    __device__ static bool active(int lane) { return D >= 128 || lane < D / 4; }
};

// Log-sum-exp sum of the partials lo .. hi-1 of one query head: *M = their
// largest running max, *L = sum_s l_s 2^(m_s - M), and acc = sum_s o_s
// 2^(m_s - M) for this lane's channels (M = -inf, L = 0, 0 for an empty
// range). Partials are read through L2 (ld.global.cg): other CTAs of this
// launch wrote them. The first CHUNK partial rows are requested together with
// the (m, l) pairs, so up to CHUNK splits cost one L2 round trip.
template <int CHUNK, int D>
__device__ __forceinline__ void merge_range(const float2* ml, const float4* po, int lo, int hi, int lane,
                                            float* M_out, float* L_out, float4 (&acc)[MergeShape<D>::kVec]) {
    static_assert(CHUNK == 4 || CHUNK == 8 || CHUNK == 16, "chunk of partial rows");
    constexpr int NV = MergeShape<D>::kVec;
    const bool on = MergeShape<D>::active(lane);
    const int n = hi - lo;
    ml += lo;
    po += (long long)lo * (D / 4);
    float4 v[CHUNK][NV];
#pragma unroll
    for (int k = 0; k < CHUNK; ++k)
#pragma unroll
        for (int e = 0; e < NV; ++e)
            v[k][e] = on && k < n ? __ldcg(po + (long long)k * (D / 4) + 32 * e) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float2 x0 = lane < n ? __ldcg(&ml[lane]) : make_float2(-INFINITY, 0.f);
    float M = x0.x;
    for (int s = lane + 32; s < n; s += 32) M = fmaxf(M, __ldcg(&ml[s]).x);
    M = warp_max(M);
    float L = 0.f;
#pragma unroll
    for (int e = 0; e < NV; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n; s0 += 32) {
        float2 x = x0;
        if (s0 > 0) x = s0 + lane < n ? __ldcg(&ml[s0 + lane]) : make_float2(-INFINITY, 0.f);
        const float wt = x.x == -INFINITY ? 0.f : exp2f(x.x - M);
        L = fmaf(x.y, wt, L);
        for (int k0 = 0; k0 < 32 && s0 + k0 < n; k0 += CHUNK) {
            if (s0 + k0 > 0) {
#pragma unroll
                for (int k = 0; k < CHUNK; ++k)
#pragma unroll
                    for (int e = 0; e < NV; ++e)
                        v[k][e] = on && s0 + k0 + k < n ? __ldcg(po + (long long)(s0 + k0 + k) * (D / 4) + 32 * e)
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < CHUNK; ++k) {
                const float wk = __shfl_sync(0xffffffffu, wt, k0 + k);  // 0 past the last split
#pragma unroll
                for (int e = 0; e < NV; ++e) {
                    acc[e].x = fmaf(v[k][e].x, wk, acc[e].x);
                    acc[e].y = fmaf(v[k][e].y, wk, acc[e].y);
                    acc[e].z = fmaf(v[k][e].z, wk, acc[e].z);
                    acc[e].w = fmaf(v[k][e].w, wk, acc[e].w);
                }
            }
        }
    }
    *M_out = M;
    *L_out = warp_sum(L);
}

// Shared-memory row of one head's share in the multi-warp merge: o[D], m, l,
// padded to a multiple of 4 floats so float4 rows stay aligned.
template <int D>
__host__ __device__ constexpr int scratch_row() { return D + 4; }

// Merge of the partials of query heads bq0 .. bq0 + nheads - 1 (nheads <= 4)
// by a CTA of nwarps (4, 8 or 16) warps: warp w takes head w % 4 and the w / 4-th
// of the splits, so more warps cut the L2 round trips; the shares meet in
// `scratch` (16-byte aligned shared memory, nwarps * scratch_row<D>() floats).
// Every thread of the CTA must call it (it holds a CTA barrier when nwarps > 4).
// CHUNK partial rows per L2 round trip: CHUNK / kVec of them at D = 256.
template <int CHUNK, int D>
__device__ __forceinline__ void merge_splits(const DecodeArgs& a, long long bq0, int nheads, int warp,
                                             int nwarps, int lane, float* scratch) {
    constexpr int NV = MergeShape<D>::kVec;
    constexpr int RC = CHUNK / NV;  // rows per request at this width
    constexpr int kRow = scratch_row<D>();
    const bool on = MergeShape<D>::active(lane);
    const int n = a.n_split;
    const int h = warp & 3, sub = warp >> 2, nsub = nwarps >> 2;
    const int per = (n + nsub - 1) / nsub;
    const int lo = min(n, sub * per), hi = min(n, lo + per);
    const long long bq = bq0 + h;
    float M = -INFINITY, L = 0.f;
    float4 acc[NV];
#pragma unroll
    for (int e = 0; e < NV; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h < nheads)
        merge_range<RC, D>(reinterpret_cast<const float2*>(a.part_ml) + bq * n,
                           reinterpret_cast<const float4*>(a.part_o + bq * n * D) + lane, lo, hi, lane, &M, &L, acc);
    if (nsub > 1) {
        float* mine = scratch + (sub * 4 + h) * kRow;
        if (sub > 0 && h < nheads) {
            if (on) {
#pragma unroll
                for (int e = 0; e < NV; ++e) reinterpret_cast<float4*>(mine)[lane + 32 * e] = acc[e];
            }
            if (lane == 0) {
                mine[D] = M;
                mine[D + 1] = L;
            }
        }
        __syncthreads();
        if (sub > 0 || h >= nheads) return;
        for (int t = 1; t < nsub; ++t) {
            const float* other = scratch + (t * 4 + h) * kRow;
            const float Mo = other[D];
            if (Mo == -INFINITY) continue;  // an empty share of the splits
            const float Mn = fmaxf(M, Mo);
            const float fa = M == -INFINITY ? 0.f : exp2f(M - Mn), fb = exp2f(Mo - Mn);
            if (on) {
#pragma unroll
                for (int e = 0; e < NV; ++e) {
                    const float4 ob = reinterpret_cast<const float4*>(other)[lane + 32 * e];
                    acc[e] = make_float4(fmaf(acc[e].x, fa, ob.x * fb), fmaf(acc[e].y, fa, ob.y * fb),
                                         fmaf(acc[e].z, fa, ob.z * fb), fmaf(acc[e].w, fa, ob.w * fb));
                }
            }
            L = fmaf(L, fa, other[D + 1] * fb);
            M = Mn;
        }
    }
    if (h < nheads && on) {
#pragma unroll
        for (int e = 0; e < NV; ++e)
            reinterpret_cast<float4*>(a.out + bq * D)[lane + 32 * e] =
                make_float4(acc[e].x / L, acc[e].y / L, acc[e].z / L, acc[e].w / L);
    }
}

}  // namespace kivi

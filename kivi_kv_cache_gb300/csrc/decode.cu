// decode.cu -- fused dequantize-and-attend single-token decode over the
// packed KIVI store plus the fp16 residual window.
//
// Method: VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly
// 0% Faster", "So why does the kernel ship?" (attention reads the packed
// codes and expands them in registers, never materialising fp16 K/V), and the
// VeloxQuant-MLX benchmarks page, "KV-Cache Kernel Roofline" (one query token
// per head; a single threadgroup per (batch, head) leaves the GPU idle).
//
// GB300 design:
//  * split over the cached tokens: grid = (n_split, Hkv, B). Each CTA takes a
//    contiguous run of 32-token tiles (store tiles first, then residual
//    tiles), keeps a running max / sum per query head (online softmax) and
//    writes unnormalised partials; decode_combine merges the splits with
//    log-sum-exp weights. The split count is chosen so B*Hkv*n_split fills
//    every SM even at B = 1, Hkv = 8.
//  * grouped-query attention: one CTA serves all Hq/Hkv query heads of its KV
//    head, so each packed K/V byte is read from HBM once per group.
//  * the affine dequant is folded out of the inner loops. A key group (32
//    tokens) shares scale s_d and zero z_d per channel, so
//        q . khat_t = sum_d (q_d s_d) c_td + sum_d q_d z_d ;
//    a value row shares (s_j, z_j) per 32-channel group j, so
//        sum_t p_t vhat_td = sum_t (p_t s_tj) c_td + sum_t p_t z_tj .
//    The inner loops are then one FMA per (code, head).
//  * scores are kept in the exp2 domain (sm_scale * log2 e folded into q).
#include <math.h>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

namespace {

constexpr int kThreads = 128;  // = D: one thread per channel in the PV pass
constexpr int kTile = 32;      // tokens per tile (= G, one key group)

template <int BITS, int GQ>
struct DecodeSmem {
    static constexpr int ROWB = kD * BITS / 8;
    float q[GQ][kD];                       // q * sm_scale * log2 e
    union {
        struct {
            uint8_t kc[kTile][ROWB];
            uint8_t vc[kTile][ROWB];
            float ksc[kD];
            float kz[kD];
            float vsc[kTile][kD / kG];
            float vz[kTile][kD / kG];
        } st;
        struct {
            __half k[kTile][kD];
            __half v[kTile][kD];
        } rs;
    } tile;
    float qs[4][kTile * GQ + 4];           // q*s per channel quarter (padded)
    float qz[4][GQ];                       // per-warp partial of sum_d q_d z_d
    float sc[GQ][kTile];                   // tile scores
    float pst[kTile][kD / kG][GQ];         // p * vscale (store) or p (residual)
    float pz[kD / kG][GQ];                 // sum_t p_t * vzero_tj
    float corr[GQ];                        // rescale of the running output
};

template <int BITS, int GQ>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecodeArgs a) {
    constexpr int ROWB = kD * BITS / 8;
    constexpr uint32_t CM = Levels<BITS>::value;
    __shared__ __align__(16) DecodeSmem<BITS, GQ> sm;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int split = blockIdx.x;
    const int hk = blockIdx.y;
    const int b = blockIdx.z;
    const int bh = b * a.Hkv + hk;
    const int h0 = hk * GQ;  // first query head of this KV group

    pdl_wait();
    for (int h = 0; h < GQ; ++h)
        sm.q[h][tid] = __half2float(a.q[((long long)b * a.Hq + h0 + h) * kD + tid]) * a.score_scale;

    float o[GQ];
    float m_run[GQ], l_run[GQ];  // meaningful in warp 0
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        o[h] = 0.f;
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
    }

    const int tile_begin = split * a.tiles_per_split;
    const int tile_end = min(tile_begin + a.tiles_per_split, a.n_tiles);
    for (int tile = tile_begin; tile < tile_end; ++tile) {
        const bool is_store = tile < a.n_store_tiles;
        const int tok0 = is_store ? tile * kTile : (tile - a.n_store_tiles) * kTile;
        const int nvalid = is_store ? min(kTile, a.S_q - tok0) : min(kTile, a.n_res - tok0);

        __syncthreads();  // previous tile fully consumed (and q staged)
        // ---- 1. stage the tile in shared memory ----
        if (is_store) {
            constexpr int VPR = ROWB / 16;  // 16-byte vectors per code row
            const uint4* kc = reinterpret_cast<const uint4*>(a.kcodes + ((long long)bh * a.s_cap + tok0) * ROWB);
            const uint4* vc = reinterpret_cast<const uint4*>(a.vcodes + ((long long)bh * a.s_cap + tok0) * ROWB);
            for (int i = tid; i < kTile * VPR; i += kThreads) {
                const int row = i / VPR;
                uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
                if (row < nvalid) {
                    kv = __ldg(kc + i);
                    vv = __ldg(vc + i);
                }
                reinterpret_cast<uint4*>(&sm.tile.st.kc[0][0])[i] = kv;
                reinterpret_cast<uint4*>(&sm.tile.st.vc[0][0])[i] = vv;
            }
            const long long km = ((long long)bh * (a.s_cap / kG) + tile) * kD + tid;
            sm.tile.st.ksc[tid] = __ldg(a.kscale + km);
            sm.tile.st.kz[tid] = __half2float(a.kzero[km]);
            {
                const int row = tid >> 2, j = tid & 3;
                float s = 0.f, z = 0.f;
                if (row < nvalid) {
                    const long long vm = ((long long)bh * a.s_cap + tok0 + row) * (kD / kG) + j;
                    s = __ldg(a.vscale + vm);
                    z = __half2float(a.vzero[vm]);
                }
                sm.tile.st.vsc[row][j] = s;
                sm.tile.st.vz[row][j] = z;
            }
        } else {
            const uint4* kr = reinterpret_cast<const uint4*>(a.k_res + ((long long)bh * a.res_cap + tok0) * kD);
            const uint4* vr = reinterpret_cast<const uint4*>(a.v_res + ((long long)bh * a.res_cap + tok0) * kD);
            for (int i = tid; i < kTile * (kD / 8); i += kThreads) {
                const int row = i / (kD / 8);
                uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
                if (row < nvalid) {
                    kv = __ldg(kr + i);
                    vv = __ldg(vr + i);
                }
                reinterpret_cast<uint4*>(&sm.tile.rs.k[0][0])[i] = kv;
                reinterpret_cast<uint4*>(&sm.tile.rs.v[0][0])[i] = vv;
            }
        }
        __syncthreads();

        // ---- 2. per-tile query folding (store tiles): qs_d = q_d * s_d ----
        if (is_store) {
            const float s = sm.tile.st.ksc[tid];
            const float z = sm.tile.st.kz[tid];
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                const float qv = sm.q[h][tid];
                sm.qs[tid >> 5][(tid & 31) * GQ + h] = qv * s;
                const float part = warp_sum(qv * z);
                if (lane == 0) sm.qz[warp][h] = part;
            }
            __syncthreads();
        }

        // ---- 3. scores: thread (token t, channel quarter cq) ----
        {
            const int t = tid >> 2, cq = tid & 3;
            float acc[GQ];
#pragma unroll
            for (int h = 0; h < GQ; ++h) acc[h] = 0.f;
            if (is_store) {
                // 32 channels [32cq, 32cq + 32) of token t: 16 (4-bit) or 8 (2-bit) bytes
                const uint32_t* cw = reinterpret_cast<const uint32_t*>(&sm.tile.st.kc[t][cq * 32 * BITS / 8]);
#pragma unroll
                for (int wi = 0; wi < 32 * BITS / 32; ++wi) {
                    const uint32_t w = cw[wi];
#pragma unroll
                    for (int k = 0; k < 32 / BITS; ++k) {
                        const float c = code_to_float((w >> (k * BITS)) & CM);
                        const int d = wi * (32 / BITS) + k;
#pragma unroll
                        for (int h = 0; h < GQ; ++h) acc[h] = fmaf(sm.qs[cq][d * GQ + h], c, acc[h]);
                    }
                }
            } else {
                const __half2* kr = reinterpret_cast<const __half2*>(&sm.tile.rs.k[t][cq * 32]);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 kv = __half22float2(kr[i]);
#pragma unroll
                    for (int h = 0; h < GQ; ++h) {
                        acc[h] = fmaf(sm.q[h][cq * 32 + 2 * i], kv.x, acc[h]);
                        acc[h] = fmaf(sm.q[h][cq * 32 + 2 * i + 1], kv.y, acc[h]);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
                acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 2);
            }
            if (cq == 0) {
#pragma unroll
                for (int h = 0; h < GQ; ++h) {
                    float s = acc[h];
                    if (is_store) s += sm.qz[0][h] + sm.qz[1][h] + sm.qz[2][h] + sm.qz[3][h];
                    sm.sc[h][t] = t < nvalid ? s : -INFINITY;
                }
            }
        }
        __syncthreads();

        // ---- 4. online softmax over the tile (warp 0, lane = token) ----
        if (warp == 0) {
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                const float s = sm.sc[h][lane];
                const float m_new = fmaxf(m_run[h], warp_max(s));
                const float p = lane < nvalid ? exp2f(s - m_new) : 0.f;
                const float corr = exp2f(m_run[h] - m_new);  // 0 on the first tile
                l_run[h] = l_run[h] * corr + warp_sum(p);
                m_run[h] = m_new;
                if (lane == 0) sm.corr[h] = corr;
                if (is_store) {
#pragma unroll
                    for (int j = 0; j < kD / kG; ++j) {
                        sm.pst[lane][j][h] = p * sm.tile.st.vsc[lane][j];
                        const float pzj = warp_sum(p * sm.tile.st.vz[lane][j]);
                        if (lane == 0) sm.pz[j][h] = pzj;
                    }
                } else {
                    sm.pst[lane][0][h] = p;
                }
            }
        }
        __syncthreads();

        // ---- 5. P.V: thread = channel d, group j = d / 32 = warp ----
        {
            const int d = tid, j = warp;
#pragma unroll
            for (int h = 0; h < GQ; ++h) o[h] *= sm.corr[h];
            if (is_store) {
                const int byte = d * BITS / 8, shift = (d * BITS) & 7;
#pragma unroll 8
                for (int t = 0; t < kTile; ++t) {
                    const float c = code_to_float((sm.tile.st.vc[t][byte] >> shift) & CM);
#pragma unroll
                    for (int h = 0; h < GQ; ++h) o[h] = fmaf(sm.pst[t][j][h], c, o[h]);
                }
#pragma unroll
                for (int h = 0; h < GQ; ++h) o[h] += sm.pz[j][h];
            } else {
#pragma unroll 8
                for (int t = 0; t < kTile; ++t) {
                    const float v = __half2float(sm.tile.rs.v[t][d]);
#pragma unroll
                    for (int h = 0; h < GQ; ++h) o[h] = fmaf(sm.pst[t][0][h], v, o[h]);
                }
            }
        }
    }

    // ---- partials (or the final output when there is a single split) ----
    pdl_trigger();
    __syncthreads();
    if (warp == 0 && lane == 0) {
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            sm.corr[h] = l_run[h];
            sm.pz[0][h] = m_run[h];
        }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        const long long bq = (long long)b * a.Hq + h0 + h;
        if (a.n_split == 1) {
            a.out[bq * kD + tid] = o[h] / sm.corr[h];
        } else {
            a.part_o[(bq * a.n_split + split) * kD + tid] = o[h];
            if (tid == 0) {
                a.part_ml[(bq * a.n_split + split) * 2 + 0] = sm.pz[0][h];
                a.part_ml[(bq * a.n_split + split) * 2 + 1] = sm.corr[h];
            }
        }
    }
}

// out[b, h, :] = sum_i o_i 2^(m_i - M) / sum_i l_i 2^(m_i - M), M = max_i m_i.
// One pass with a running maximum; the loads of 8 splits are issued together
// so a merge of n splits waits on about n/8 memory round trips.
__global__ void __launch_bounds__(kThreads) decode_combine_kernel(DecodeArgs a) {
    pdl_wait();
    const long long bq = blockIdx.x;
    const int n = a.n_split;
    const float* ml = a.part_ml + bq * n * 2;
    const float* po = a.part_o + bq * n * kD + threadIdx.x;
    float M = -INFINITY, L = 0.f, acc = 0.f;
    for (int i0 = 0; i0 < n; i0 += 8) {
        float m[8], l[8], o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const bool ok = i0 + k < n;
            m[k] = ok ? ml[2 * (i0 + k)] : -INFINITY;
            l[k] = ok ? ml[2 * (i0 + k) + 1] : 0.f;
            o[k] = ok ? po[(long long)(i0 + k) * kD] : 0.f;
        }
        float mc = m[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) mc = fmaxf(mc, m[k]);
        const float Mn = fmaxf(M, mc);
        const float r = Mn == -INFINITY ? 0.f : exp2f(M - Mn);
        L *= r;
        acc *= r;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float w = m[k] == -INFINITY ? 0.f : exp2f(m[k] - Mn);
            L = fmaf(l[k], w, L);
            acc = fmaf(o[k], w, acc);
        }
        M = Mn;
    }
    a.out[bq * kD + threadIdx.x] = acc / L;
}

template <int BITS, int GQ>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
    dim3 grid(a.n_split, a.Hkv, a.B);
    cudaError_t e = launch_pdl(decode_split_kernel<BITS, GQ>, grid, kThreads, 0, stream, a);
    if (e != cudaSuccess || a.n_split == 1) return e;
    e = launch_pdl(decode_combine_kernel, dim3(a.B * a.Hq), kThreads, 0, stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_bits(const DecodeArgs& a, int gq, cudaStream_t stream) {
    switch (gq) {
        case 1: return launch_typed<BITS, 1>(a, stream);
        case 2: return launch_typed<BITS, 2>(a, stream);
        case 4: return launch_typed<BITS, 4>(a, stream);
        case 8: return launch_typed<BITS, 8>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t stream) {
    if (a.n_split == 1) return cudaSuccess;
    cudaError_t e = launch_pdl(decode_combine_kernel, dim3(a.B * a.Hq), kThreads, 0, stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    return bits == 4 ? launch_bits<4>(a, gq, stream) : launch_bits<2>(a, gq, stream);
}

}  // namespace kivi

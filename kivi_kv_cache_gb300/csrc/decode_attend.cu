// decode_attend.cu -- fused dequantize-and-attend single-token decode over the
// packed KIVI store plus the fp16 residual window, on the tensor cores
// (mma.sync m16n8k16, fp16 operands, fp32 accumulation), with the channels of
// each tile split over the CTA's warps. It serves any grouped-query group of
// up to 8 query heads per KV head; groups of 1, 2 or 4 heads run the
// one-warp-per-tile kernel of decode_mma.cu, which executes fewer instructions
// per tile.
//
// Method: VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly
// 0% Faster", "So why does the kernel ship?" (attention reads the packed
// codes and expands them in registers), and the VeloxQuant-MLX benchmarks
// page, "KV-Cache Kernel Roofline" (one query token per head; too few
// threadgroups per (batch, head) leave the GPU idle, so the cached tokens are
// split across CTAs and merged by a log-sum-exp combine).
//
// The dequant is folded out of the contraction. A key group shares s_d, z_d
// per channel, and a value row shares s_j, z_j per 32-channel group:
//     q . khat_t  = sum_d (q_d s_d) c_td + sum_d q_d z_d
//     sum_t p_t vhat_td = sum_t (p_t s_tj) c_td + sum_t p_t z_tj
// The codes c are one MMA operand, exact in fp16. The fp32 products
// q_d s_d and p_t s_tj form the other operand:
//   * a code nibble (or 2-bit crumb) alone in a byte, read as fp8 e4m3, is
//     c * 2^-9 exactly, so cvt.rn.f16x2.e4m3x2 turns two codes into fp16;
//   * each fp32 operand is split into fp16 hi + lo (hi = fp16(x), lo =
//     fp16(x - hi)) and carried as two MMA columns per query head, n = 2h +
//     part. The pair keeps about 22 significant bits;
//   * a power-of-two factor per tile and warp keeps every hi below 2^14, so
//     no fp16 overflows for any finite input. It is divided out exactly
//     afterwards.
// The sums over z are plain fp32 FMAs.
//
// Work split: the grid is (n_split, Hkv, B). A CTA owns a contiguous run of
// tiles of one (batch, KV head): 32-token tiles of the packed store, then
// 16-token tiles of the residual window. Its 4 warps work on the same tile
// together, split by channels:
//   * warp w computes the partial q.k over channels 32w..32w+31;
//   * warp w computes p.v for value group w, channels 32w..32w+31.
// One CTA barrier per tile exchanges the partial scores. Every warp then runs
// the same online softmax on the full scores, bit-identical in all four, so no
// softmax states need merging inside the CTA: each warp owns a quarter of the
// output channels.
// Tiles are staged by all 128 threads with cp.async in a 4-deep ring, with
// layouts chosen so that the fragment loads are free of bank conflicts.
// Splits of one (batch, KV head) meet in the workspace:
//   * each CTA writes its partial (o, m, l) and takes a ticket from a per-head
//     counter;
//   * the CTA with the last ticket sets the counter back to zero and merges
//     the partials into the output with log-sum-exp weights.
//
// MMA fragment layouts (m16n8k16, row.col), lane = 4 g + c:
//   * A regs: (row g, k 2c..2c+1), (row g+8, same k), (row g, k 2c+8..9),
//     (row g+8, k 2c+8..9);
//   * B regs: (k 2c..2c+1, n g), (k 2c+8..9, n g);
//   * C regs: (row g, n 2c..2c+1), (row g+8, n 2c..2c+1).
#include <math.h>

#include "decode_common.cuh"
#include "decode_merge.cuh"
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

namespace {

using namespace dec;

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 4;
constexpr int kStage = 8192;  // bytes per ring stage
constexpr int kResTok = kResTileTokensSplit;  // tokens per residual tile
// Store tile inside a stage.
//   KC, VC: codes as [16-byte column][32 rows][16 B].
//   KS: key scales [128] f32.   KZ: key zeros [128] f16.
//   VS: value scales [32][4] f32.   VZ: value zeros [32][4] f16.
constexpr int kKC = 0, kVC = 2048, kKS = 4096, kKZ = 4608, kVS = 4864, kVZ = 5376;
// Residual tile: K rows [16][256 B] at 0 and V rows at kRV. The 16-byte chunk
// c of row r sits at position c ^ (r & 7).
constexpr int kRV = 4096;
constexpr int kOwStride = 33;  // epilogue rows, padded

template <int NB>
struct Smem {
    uint8_t stage[kStages][kStage];
    float psc[2][32][4 * NB][kWarps];      // partial scores [buffer][token][head][warp]
    float pbuf[kWarps][32][4 * NB];        // this tile's p, per warp [token][head]
    float ow[kWarps][4 * NB][kOwStride];   // epilogue: each warp's 32 channels per head
    int last;
};

// ---------------------------------------------------------------------------
// tile staging (all 128 threads)
// ---------------------------------------------------------------------------

template <int BITS>
__device__ __forceinline__ void fetch_tile(const DecodeArgs& a, int bh, int tile, uint8_t* st, int tid) {
    if (tile < a.n_store_tiles) {
        constexpr int ROWB = kD * BITS / 8;  // 64 or 32 bytes per token row
        constexpr int CPR = ROWB / 16;       // 16-byte chunks per row
        constexpr int NC = 32 * CPR;         // chunks per code tile
        const long long row0 = (long long)bh * a.s_cap + (long long)tile * 32;
        const long long grp = (long long)bh * (a.s_cap / kG) + tile;
#pragma unroll
        for (int i = tid; i < 2 * NC + 96; i += kThreads) {
            const uint8_t* src;
            int off;
            if (i < 2 * NC) {
                const bool v = i >= NC;
                const int j = v ? i - NC : i, row = j / CPR, col = j % CPR;
                src = (v ? a.vcodes : a.kcodes) + (row0 + row) * ROWB + col * 16;
                off = (v ? kVC : kKC) + col * 512 + row * 16;
            } else {
                const int j = i - 2 * NC;
                if (j < 32) {
                    src = reinterpret_cast<const uint8_t*>(a.kscale + grp * kD) + j * 16;
                    off = kKS + j * 16;
                } else if (j < 48) {
                    src = reinterpret_cast<const uint8_t*>(a.kzero + grp * kD) + (j - 32) * 16;
                    off = kKZ + (j - 32) * 16;
                } else if (j < 80) {
                    src = reinterpret_cast<const uint8_t*>(a.vscale + row0 * (kD / kG)) + (j - 48) * 16;
                    off = kVS + (j - 48) * 16;
                } else {
                    src = reinterpret_cast<const uint8_t*>(a.vzero + row0 * (kD / kG)) + (j - 80) * 16;
                    off = kVZ + (j - 80) * 16;
                }
            }
            cp_async16(st + off, src, true);
        }
    } else {
        const int rt = tile - a.n_store_tiles;
        const int nvalid = min(kResTok, a.n_res - rt * kResTok);
        const long long row0 = (long long)bh * a.res_cap + (long long)rt * kResTok;
#pragma unroll
        for (int i = tid; i < 2 * kResTok * 16; i += kThreads) {
            const bool v = i >= kResTok * 16;
            const int j = v ? i - kResTok * 16 : i, row = j >> 4, col = j & 15;
            const __half* base = v ? a.v_res : a.k_res;
            const bool ok = row < nvalid;
            const __half* src = ok ? base + (row0 + row) * kD + col * 8 : base;
            cp_async16(st + (v ? kRV : 0) + row * 256 + ((col ^ (row & 7)) << 4), src, ok);
        }
    }
}

// ---------------------------------------------------------------------------
// per-tile pieces (one warp, its 32 channels)
// ---------------------------------------------------------------------------

// Partial scores of a store tile over channels 32w..32w+31. Lane (g, c) holds
// q8[nb][i] = q_(4nb + g/2), channel 32w + 8c + i, times the softmax scale.
// sc[nb][i]: token g + 8i, head 4nb + c.
template <int BITS, int NB>
__device__ __forceinline__ void qk_store(const uint8_t* S, int w, int g, int c, bool lo_part,
                                         const float (&q8)[NB][8], float qmax, float (&sc)[NB][4]) {
    const float* KS = reinterpret_cast<const float*>(S + kKS) + 32 * w + 8 * c;
    const float4 sa = *reinterpret_cast<const float4*>(KS);
    const float4 sb = *reinterpret_cast<const float4*>(KS + 4);
    const float s8[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
    float smax = fmaxf(fmaxf(fmaxf(sa.x, sa.y), fmaxf(sa.z, sa.w)), fmaxf(fmaxf(sb.x, sb.y), fmaxf(sb.z, sb.w)));
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 1));
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 2));  // scales are >= 0
    const int E = safe_exp(qmax * smax);
    const float fB = pow2i(E);      // B operand = q s 2^E
    const float fC = pow2i(9 - E);  // codes enter as c 2^-9
    const uint4 zw = *reinterpret_cast<const uint4*>(S + kKZ + (32 * w + 8 * c) * 2);
    const uint32_t zz[4] = {zw.x, zw.y, zw.z, zw.w};
    float z8[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(u32_as_h2(zz[k]));
        z8[2 * k] = f.x;
        z8[2 * k + 1] = f.y;
    }

    uint32_t bq[NB][2][2];
    float qzc[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = q8[nb][i] * s8[i] * fB;
        if (BITS == 4) {  // K-step 0: channels 8c + {0,2 | 4,6}; K-step 1: {1,3 | 5,7}
            bq[nb][0][0] = split_pair(v[0], v[2], lo_part);
            bq[nb][0][1] = split_pair(v[4], v[6], lo_part);
            bq[nb][1][0] = split_pair(v[1], v[3], lo_part);
            bq[nb][1][1] = split_pair(v[5], v[7], lo_part);
        } else {          // K-step 0: channels 8c + {0,4 | 1,5}; K-step 1: {2,6 | 3,7}
            bq[nb][0][0] = split_pair(v[0], v[4], lo_part);
            bq[nb][0][1] = split_pair(v[1], v[5], lo_part);
            bq[nb][1][0] = split_pair(v[2], v[6], lo_part);
            bq[nb][1][1] = split_pair(v[3], v[7], lo_part);
        }
        float t = 0.f;  // sum_d q_d z_d of head 4nb + g/2 over this lane's 8 channels
#pragma unroll
        for (int i = 0; i < 8; ++i) t = fmaf(q8[nb][i], z8[i], t);
        t += __shfl_xor_sync(0xffffffffu, t, 1);
        t += __shfl_xor_sync(0xffffffffu, t, 2);
        qzc[nb] = __shfl_sync(0xffffffffu, t, 8 * c);  // lane 8c has g = 2c: head 4nb + c
    }

#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        const int r0 = 16 * mt + g, r1 = r0 + 8;
        uint32_t A[2][4];  // [K-step][a0..a3]
        if (BITS == 4) {
            const uint8_t* KC = S + kKC + w * 512 + 4 * c;
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(KC + r0 * 16);
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(KC + r1 * 16);
            e4m3x4_to_f16(w0 & 0x0f0f0f0fu, A[0][0], A[0][2]);
            e4m3x4_to_f16(w1 & 0x0f0f0f0fu, A[0][1], A[0][3]);
            e4m3x4_to_f16((w0 >> 4) & 0x0f0f0f0fu, A[1][0], A[1][2]);
            e4m3x4_to_f16((w1 >> 4) & 0x0f0f0f0fu, A[1][1], A[1][3]);
        } else {
            const uint8_t* KC = S + kKC + (w >> 1) * 512 + 8 * (w & 1) + 2 * c;
            const uint32_t p0 = *reinterpret_cast<const uint16_t*>(KC + r0 * 16);
            const uint32_t p1 = *reinterpret_cast<const uint16_t*>(KC + r1 * 16);
            const uint32_t x = p0 | (p1 << 16);  // crumb k: channel 8c + k (byte 0/2), 8c + 4 + k (byte 1/3)
            e4m3x4_to_f16(x & 0x03030303u, A[0][0], A[0][1]);
            e4m3x4_to_f16((x >> 2) & 0x03030303u, A[0][2], A[0][3]);
            e4m3x4_to_f16((x >> 4) & 0x03030303u, A[1][0], A[1][1]);
            e4m3x4_to_f16((x >> 6) & 0x03030303u, A[1][2], A[1][3]);
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(acc, A[0][0], A[0][1], A[0][2], A[0][3], bq[nb][0][0], bq[nb][0][1]);
            mma16816(acc, A[1][0], A[1][1], A[1][2], A[1][3], bq[nb][1][0], bq[nb][1][1]);
            sc[nb][2 * mt] = fmaf(acc[0] + acc[1], fC, qzc[nb]);
            sc[nb][2 * mt + 1] = fmaf(acc[2] + acc[3], fC, qzc[nb]);
        }
    }
}

// Partial scores of a residual tile (fp16 K rows) over channels 32w..32w+31.
// br: q 2^Er hi or lo in natural channel order. sc[nb][0..1]: tokens g, g+8.
template <int NB>
__device__ __forceinline__ void qk_res(const uint8_t* S, int w, int lane, const uint32_t (&br)[NB][2][2],
                                       float fCr, float (&sc)[NB][4]) {
    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
    const int q = lane >> 3, r = lane & 7;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int row = (q & 1) * 8 + r, chunk = 4 * w + 2 * s + (q >> 1);
        uint32_t A[4];
        ldsm_x4(A, S + row * 256 + ((chunk ^ (row & 7)) << 4));
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) mma16816(acc[nb], A[0], A[1], A[2], A[3], br[nb][s][0], br[nb][s][1]);
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        sc[nb][0] = (acc[nb][0] + acc[nb][1]) * fCr;
        sc[nb][1] = (acc[nb][2] + acc[nb][3]) * fCr;
        sc[nb][2] = sc[nb][3] = 0.f;
    }
}

// P.V of a store tile for value group w. p[nb][i]: token g + 8i, head 4nb + c;
// pb: this warp's p as [token][head]. Accumulators o[nb][m] (units of 2^-9):
//   4-bit, m = u in {0,1}: rows g -> channel 32w + 4g + u, g+8 -> 32w + 4g + 2 + u;
//   2-bit, m = k in 0..3: rows g -> channel 8g + k, g+8 -> 8g + 4 + k of the
//   64-channel column w/2 (channels 64(w/2)..); rows of lanes with g/4 == w%2
//   are this warp's group, the other rows stay zero.
template <int BITS, int NB>
__device__ __forceinline__ void pv_store(const uint8_t* S, int w, int lane, int g, int c, int hh, bool lo_part,
                                         int nvalid, const float (&p)[NB][4], const float* pb,
                                         float (&o)[NB][BITS == 4 ? 2 : 4][4]) {
    constexpr int NH = 4 * NB;
    const float* VS = reinterpret_cast<const float*>(S + kVS);
    const __half* VZ = reinterpret_cast<const __half*>(S + kVZ);
    // sum_t p_t z_tw of head 4nb + c (rows past nvalid have p = 0; their z may be stale)
    float zt[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = g + 8 * i;
        zt[i] = t < nvalid ? __half2float(VZ[t * 4 + w]) : 0.f;
    }
    float pz[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) s = fmaf(p[nb][i], zt[i], s);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        s += __shfl_xor_sync(0xffffffffu, s, 8);
        s += __shfl_xor_sync(0xffffffffu, s, 16);
        pz[nb] = s * (1.0f / 512.f);  // o is kept in units of 2^-9 (codes)
    }
    // B operand: p_t s_tw of head 4nb + hh; K-step ks covers tokens 16ks + {2c, 2c+1 | 2c+8, 2c+9}
    uint32_t bp[NB][2][2];
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const int ta = 16 * ks + 2 * c, tb = ta + 8;
        const float sa0 = ta < nvalid ? VS[ta * 4 + w] : 0.f;
        const float sa1 = ta + 1 < nvalid ? VS[(ta + 1) * 4 + w] : 0.f;
        const float sb0 = tb < nvalid ? VS[tb * 4 + w] : 0.f;
        const float sb1 = tb + 1 < nvalid ? VS[(tb + 1) * 4 + w] : 0.f;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int h = 4 * nb + hh;
            bp[nb][ks][0] = split_pair(pb[ta * NH + h] * sa0, pb[(ta + 1) * NH + h] * sa1, lo_part);
            bp[nb][ks][1] = split_pair(pb[tb * NH + h] * sb0, pb[(tb + 1) * NH + h] * sb1, lo_part);
        }
    }
    if (BITS == 4) {
        uint32_t W[4];  // matrix q: tokens 8q..8q+7 of group w's 16-byte column
        ldsm_x4_t(W, S + kVC + w * 512 + lane * 16);
        uint32_t xl[2][4], xh[2][4];  // [u][q]
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            e4m3x4_to_f16(__byte_perm(W[q] & 0x0f0f0f0fu, 0, 0x3120), xl[0][q], xh[0][q]);
            e4m3x4_to_f16(__byte_perm((W[q] >> 4) & 0x0f0f0f0fu, 0, 0x3120), xl[1][q], xh[1][q]);
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma16816(o[nb][u], xl[u][2 * ks], xh[u][2 * ks], xl[u][2 * ks + 1], xh[u][2 * ks + 1],
                             bp[nb][ks][0], bp[nb][ks][1]);
                o[nb][u][0] += pz[nb];
                o[nb][u][2] += pz[nb];
            }
    } else {
        uint32_t W[4];
        ldsm_x4_t(W, S + kVC + (w >> 1) * 512 + lane * 16);
        const bool mine = (g >> 2) == (w & 1);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t xl[4], xh[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                e4m3x4_to_f16(__byte_perm((W[q] >> (2 * k)) & 0x03030303u, 0, 0x3120), xl[q], xh[q]);
                if (!mine) xl[q] = xh[q] = 0u;
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma16816(o[nb][k], xl[2 * ks], xh[2 * ks], xl[2 * ks + 1], xh[2 * ks + 1], bp[nb][ks][0],
                             bp[nb][ks][1]);
                o[nb][k][0] += pz[nb];
                o[nb][k][2] += pz[nb];
            }
        }
    }
}

// P.V of a residual tile (fp16 V rows) for channels 32w..32w+31:
// orr[nb][mb] rows g -> channel 32w + 16mb + g, g+8 -> 32w + 16mb + 8 + g.
template <int NB>
__device__ __forceinline__ void pv_res(const uint8_t* S, int w, int lane, int c, int hh, bool lo_part,
                                       const float* pb, float (&orr)[NB][2][4]) {
    constexpr int NH = 4 * NB;
    uint32_t bpr[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int h = 4 * nb + hh;
        bpr[nb][0] = split_pair(pb[(2 * c) * NH + h], pb[(2 * c + 1) * NH + h], lo_part);
        bpr[nb][1] = split_pair(pb[(2 * c + 8) * NH + h], pb[(2 * c + 9) * NH + h], lo_part);
    }
    const int q = lane >> 3, r = lane & 7;
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
        const int row = (q >> 1) * 8 + r, chunk = 4 * w + 2 * mb + (q & 1);
        uint32_t A[4];
        ldsm_x4_t(A, S + kRV + row * 256 + ((chunk ^ (row & 7)) << 4));
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) mma16816(orr[nb][mb], A[0], A[1], A[2], A[3], bpr[nb][0], bpr[nb][1]);
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <int BITS, int NB>
__global__ void __launch_bounds__(kThreads, 4) decode_attend_kernel(DecodeArgs a) {
    constexpr int NH = 4 * NB;            // query heads per CTA
    constexpr int NO = BITS == 4 ? 2 : 4; // store-tile accumulators per n8 block
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem<NB>& sm = *reinterpret_cast<Smem<NB>*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int hh = g >> 1;         // head (within an n8 block) of this lane's B column
    const bool lo_part = g & 1;    // hi (0) or lo (1) part of that column
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int bh = b * a.Hkv + hk;
    const int gq = a.Hq / a.Hkv, h0 = hk * gq;
    // this CTA's tiles: the head's n_tiles spread evenly over its n_split CTAs (>= 1 each)
    const int t0 = (int)((long long)split * a.n_tiles / a.n_split);
    const int nt = (int)((long long)(split + 1) * a.n_tiles / a.n_split) - t0;

    pdl_wait();
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
        if (k < nt) fetch_tile<BITS>(a, bh, t0 + k, sm.stage[k], tid);
        cp_async_commit();
    }

    // q of head 4nb + hh, channels 32w + 8c + i, times the softmax scale (exp2 domain)
    float q8[NB][8];
    float qmax = 0.f;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int h = 4 * nb + hh;
        if (h < gq) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(a.q + ((long long)b * a.Hq + h0 + h) * kD +
                                                                 32 * w + 8 * c));
            const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __half22float2(u32_as_h2(uu[k]));
                q8[nb][2 * k] = f.x * a.score_scale;
                q8[nb][2 * k + 1] = f.y * a.score_scale;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) q8[nb][i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) qmax = fmaxf(qmax, fabsf(q8[nb][i]));
    }
    qmax = warp_max(qmax);

    // residual-tile B operand: q 2^Er (hi or lo), K-step s: channels 32w + 16s + {2c, 2c+1 | 2c+8, 2c+9}
    const int Er = safe_exp(qmax);
    const float fBr = pow2i(Er), fCr = pow2i(-Er);
    uint32_t br[NB][2][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int h = 4 * nb + hh;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (h < gq) {
                const __half* qp = a.q + ((long long)b * a.Hq + h0 + h) * kD + 32 * w + 16 * s + 2 * c;
                const float2 x = __half22float2(__ldg(reinterpret_cast<const __half2*>(qp)));
                const float2 y = __half22float2(__ldg(reinterpret_cast<const __half2*>(qp + 8)));
                br[nb][s][0] = split_pair(x.x * a.score_scale * fBr, x.y * a.score_scale * fBr, lo_part);
                br[nb][s][1] = split_pair(y.x * a.score_scale * fBr, y.y * a.score_scale * fBr, lo_part);
            } else {
                br[nb][s][0] = br[nb][s][1] = 0u;
            }
        }
    }

    float m_run[NB], l_run[NB];  // online softmax of head 4nb + c (identical in all warps)
    float o[NB][NO][4], orr[NB][2][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        m_run[nb] = -INFINITY;
        l_run[nb] = 0.f;
#pragma unroll
        for (int m = 0; m < NO; ++m) o[nb][m][0] = o[nb][m][1] = o[nb][m][2] = o[nb][m][3] = 0.f;
#pragma unroll
        for (int m = 0; m < 2; ++m) orr[nb][m][0] = orr[nb][m][1] = orr[nb][m][2] = orr[nb][m][3] = 0.f;
    }

    cp_async_wait<kStages - 2>();
    __syncthreads();  // tile 0 is in shared memory

    for (int it = 0; it < nt; ++it) {
        const int tile = t0 + it;
        const uint8_t* S = sm.stage[it % kStages];
        const bool store = tile < a.n_store_tiles;
        const int nvalid = store ? min(32, a.S_q - tile * 32)
                                 : min(kResTok, a.n_res - (tile - a.n_store_tiles) * kResTok);
        const int ni = store ? 4 : 2;  // token slots g + 8i in this tile
        float sc[NB][4];
        if (store)
            qk_store<BITS, NB>(S, w, g, c, lo_part, q8, qmax, sc);
        else
            qk_res<NB>(S, w, lane, br, fCr, sc);
        float* P = &sm.psc[it & 1][0][0][0];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i < ni) P[((g + 8 * i) * NH + 4 * nb + c) * kWarps + w] = sc[nb][i];

        cp_async_wait<kStages - 3>();  // this thread's copies of tile it+1 have landed
        __syncthreads();               // partial scores and tile it+1 visible; tile it-1 released
        {
            const int nx = it + kStages - 1;
            if (nx < nt) fetch_tile<BITS>(a, bh, t0 + nx, sm.stage[nx % kStages], tid);
            cp_async_commit();
        }

        // full scores, online softmax
        float p[NB][4];
        float* pb = &sm.pbuf[w][0][0];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float s[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = g + 8 * i;
                if (i < ni && t < nvalid) {
                    const float4 v = *reinterpret_cast<const float4*>(&P[(t * NH + 4 * nb + c) * kWarps]);
                    s[i] = ((v.x + v.y) + v.z) + v.w;
                } else {
                    s[i] = -INFINITY;
                }
            }
            float tmax = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
            const float m_new = fmaxf(m_run[nb], tmax);  // finite: every tile has a valid token
            const float corr = exp2f(m_run[nb] - m_new);
            float ps = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                p[nb][i] = exp2f(s[i] - m_new);
                ps += p[nb][i];
            }
            ps += __shfl_xor_sync(0xffffffffu, ps, 4);
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            l_run[nb] = fmaf(l_run[nb], corr, ps);
            m_run[nb] = m_new;
#pragma unroll
            for (int m = 0; m < NO; ++m)
#pragma unroll
                for (int k = 0; k < 4; ++k) o[nb][m][k] *= corr;
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int k = 0; k < 4; ++k) orr[nb][m][k] *= corr;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i < ni) pb[(g + 8 * i) * NH + 4 * nb + c] = p[nb][i];
        }
        __syncwarp();
        if (store)
            pv_store<BITS, NB>(S, w, lane, g, c, hh, lo_part, nvalid, p, pb, o);
        else
            pv_res<NB>(S, w, lane, c, hh, lo_part, pb, orr);
    }
    cp_async_wait<0>();
    pdl_trigger();

    // ---- this warp's 32 output channels per head -> sm.ow[w] ----
    float* ow = &sm.ow[w][0][0];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        float* oh = ow + (4 * nb + c) * kOwStride;
        if (BITS == 4) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                oh[4 * g + u] = (o[nb][u][0] + o[nb][u][1]) * 512.f;
                oh[4 * g + 2 + u] = (o[nb][u][2] + o[nb][u][3]) * 512.f;
            }
        } else if ((g >> 2) == (w & 1)) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                oh[8 * (g & 3) + k] = (o[nb][k][0] + o[nb][k][1]) * 512.f;
                oh[8 * (g & 3) + 4 + k] = (o[nb][k][2] + o[nb][k][3]) * 512.f;
            }
        }
    }
    __syncwarp();
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        float* oh = ow + (4 * nb + c) * kOwStride;
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
            oh[16 * mb + g] += orr[nb][mb][0] + orr[nb][mb][1];
            oh[16 * mb + 8 + g] += orr[nb][mb][2] + orr[nb][mb][3];
        }
    }
    __syncwarp();
#pragma unroll
    for (int h = 0; h < NH; ++h) {
        const float mh = __shfl_sync(0xffffffffu, m_run[h >> 2], h & 3);
        const float lh = __shfl_sync(0xffffffffu, l_run[h >> 2], h & 3);
        if (h >= gq) continue;
        const long long bq = (long long)b * a.Hq + h0 + h;
        const float v = ow[h * kOwStride + lane];
        if (a.n_split == 1) {
            a.out[bq * kD + 32 * w + lane] = v / lh;
        } else {
            a.part_o[(bq * a.n_split + split) * kD + 32 * w + lane] = v;
            if (w == 0 && lane == 0) {
                a.part_ml[(bq * a.n_split + split) * 2 + 0] = mh;
                a.part_ml[(bq * a.n_split + split) * 2 + 1] = lh;
            }
        }
    }
    if (a.n_split == 1) return;
    if (take_last_ticket(a, bh, &sm.last)) merge_splits_by_head<16>(a, (long long)b * a.Hq + h0, min(NH, gq), w, lane);
}

template <int BITS, int NB>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
    static bool configured = false;  // benign race: every caller sets the same value
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_attend_kernel<BITS, NB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem<NB>));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(decode_attend_kernel<BITS, NB>, dim3(a.n_split, a.Hkv, a.B), kThreads, sizeof(Smem<NB>),
                      stream, a);
}

}  // namespace

cudaError_t launch_decode_channel_split(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    cudaError_t e;
    if (gq <= 4)
        e = bits == 4 ? launch_typed<4, 1>(a, stream) : launch_typed<2, 1>(a, stream);
    else if (gq <= 8)
        e = bits == 4 ? launch_typed<4, 2>(a, stream) : launch_typed<2, 2>(a, stream);
    else
        return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kivi

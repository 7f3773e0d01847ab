// decode_pair.cu -- the fused dequantize-and-attend decode for groups of 1, 2
// or 4 query heads per KV head, with two warps per tile: the form for small
// batches, where the time of one tile's dependent chain bounds the launch.
//
// Method: VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly
// 0% Faster", "So why does the kernel ship?" (attention reads the packed
// codes and expands them in registers), and the VeloxQuant-MLX benchmarks
// page, "KV-Cache Kernel Roofline" (one query token per head; the cached
// tokens are split across CTAs and merged by a log-sum-exp combine).
//
// The arithmetic is that of decode_mma.cu: the affine dequant is folded out
// of both contractions, codes enter the tensor cores exactly as the fp16
// subnormals they form when masked in place, and the fp32 products q_d s_d
// and p_t s_tj enter as fp16 hi/lo column pairs, scaled by a power of two per
// tile and warp.
//
// Work split: a CTA has 4 warp pairs (8 warps; two CTAs per SM). A pair owns
// a contiguous run of tiles
// of one (batch, KV head): 32-token store tiles, then 16-token residual
// tiles. The two warps of a pair work on the same tile, split by channels:
// warp hf takes q.k over channels 64hf..64hf+63 and p.v for value groups 2hf
// and 2hf + 1. A 64-thread named barrier per tile exchanges the partial
// scores, and both warps run the same online softmax on the full scores.
// Against one warp per tile, each warp's chain per tile is about half as
// long (the B operands, code conversions and MMAs are split), at the price
// of one duplicated softmax. Each pair stages its tiles through a 3-deep
// cp.async ring; the CTA merges its pairs in shared memory, and the splits of
// a (batch, KV head) merge as in decode_mma.cu (in a thread-block cluster or
// through the workspace ticket).
#include <math.h>

#include "decode_common.cuh"
#include "decode_merge.cuh"
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

namespace {

using namespace dec;

constexpr int kPairs = kPairsPerCta;  // 4: 8 warps, two CTAs per SM
constexpr int kWarps = 2 * kPairs;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 3;
constexpr int kStage = 8192;  // a residual tile (16 K rows + 16 V rows); a 4-bit store tile uses 5696
constexpr int kQRow = kD + 16;  // padded row: channel ch at ch + (ch >> 5) * 4
constexpr int kResTok = kResTileTokensMma;
// store tile inside a stage: KC [32 rows][D*b/8] linear; VC rows with their
// 16-byte chunks swizzled; KS padded like q; KZ; VS [32][4]; VZ [32][4]
constexpr int kKC = 0, kVC = 2048, kKS = 4096, kKZ = 4672, kVS = 4928, kVZ = 5440;
constexpr int kRV = 4096;  // residual tile: K rows at 0, V rows here; chunk c of row r at c ^ (r & 7)
// shared memory (111 KB): rings [pair][stage], partial scores
// [pair][buf][half][32][4], p per warp [32][4], q * score_scale [4][kQRow],
// misc (qmax per warp [8], pair (m, l) [4][4][2] at 16, merge flag at 96,
// cluster (m, l) at 100)
constexpr int kPscOff = kPairs * kStages * kStage;
constexpr int kPbufOff = kPscOff + kPairs * 2048;
constexpr int kQOff = kPbufOff + kWarps * 512;
constexpr int kMiscOff = kQOff + 4 * kQRow * 4;
constexpr int kSmemBytes = kMiscOff + 512;

__device__ __forceinline__ int padc(int ch) { return ch + ((ch >> 5) << 2); }

// ---------------------------------------------------------------------------
// tile staging by the 64 threads of a pair (pt = 0..63)
// ---------------------------------------------------------------------------

template <int BITS>
__device__ __forceinline__ void fetch_tile(const DecodeArgs& a, int bh, int tile, uint8_t* st, int pt) {
    if (tile < a.n_store_tiles) {
        constexpr int ROWB = kD * BITS / 8;  // 64 or 32
        constexpr int CPR = ROWB / 16;       // 16-byte chunks per code row: 4 or 2
        constexpr int NC = 32 * CPR;
        const long long row0 = (long long)bh * a.s_cap + (long long)tile * 32;
        const long long grp = (long long)bh * (a.s_cap / kG) + tile;
#pragma unroll
        for (int i = pt; i < 2 * NC + 96; i += 64) {
            const uint8_t* src;
            int off;
            if (i < NC) {
                src = a.kcodes + row0 * ROWB + i * 16;
                off = kKC + i * 16;
            } else if (i < 2 * NC) {
                const int j = i - NC, row = j / CPR, col = j % CPR;
                const int sw = BITS == 4 ? (col ^ ((row >> 1) & 3)) : (col ^ ((row >> 2) & 1));
                src = a.vcodes + row0 * ROWB + j * 16;
                off = kVC + row * ROWB + sw * 16;
            } else {
                const int j = i - 2 * NC;
                if (j < 32) {
                    src = reinterpret_cast<const uint8_t*>(a.kscale + grp * kD + j * 4);
                    off = kKS + padc(j * 4) * 4;
                } else if (j < 48) {
                    src = reinterpret_cast<const uint8_t*>(a.kzero + grp * kD + (j - 32) * 8);
                    off = kKZ + (j - 32) * 16;
                } else if (j < 80) {
                    src = reinterpret_cast<const uint8_t*>(a.vscale + row0 * (kD / kG) + (j - 48) * 4);
                    off = kVS + (j - 48) * 16;
                } else {
                    src = reinterpret_cast<const uint8_t*>(a.vzero + row0 * (kD / kG) + (j - 80) * 8);
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
        for (int i = pt; i < 2 * kResTok * 16; i += 64) {
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
// the kernel
// ---------------------------------------------------------------------------

template <int BITS, int GQ, bool CL>
__global__ void __launch_bounds__(kThreads, kPairs <= 4 ? 2 : 1) decode_pair_kernel(DecodeArgs a) {
    constexpr int NO = 4;  // P.V accumulators per warp: 4-bit [group jj][u], 2-bit [k]
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pair = warp >> 1, hf = warp & 1, pt = tid & 63;
    const int g = lane >> 2, c = lane & 3;
    const int hh = g >> 1;        // head of this lane's B column n = g
    const bool lo_part = g & 1;   // hi (0) or lo (1) part of that column
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int bh = b * a.Hkv + hk, h0 = hk * GQ;
    uint8_t* ring = smem + pair * kStages * kStage;
    float* psc = reinterpret_cast<float*>(smem + kPscOff + pair * 2048);  // [buf][half][token][head]
    float* pbuf = reinterpret_cast<float*>(smem + kPbufOff + warp * 512);  // [token][head]
    float* q_s = reinterpret_cast<float*>(smem + kQOff);                   // [head][channel]
    float* misc = reinterpret_cast<float*>(smem + kMiscOff);
    const int bar = 1 + pair;  // named barrier of this pair

    // this pair's tiles: the head's n_tiles spread evenly over its n_split * kPairs pairs
    const long long np_head = (long long)a.n_split * kPairs, gp = (long long)split * kPairs + pair;
    const int t0 = (int)(gp * a.n_tiles / np_head);
    const int nt = (int)((gp + 1) * a.n_tiles / np_head) - t0;

    // with store_ready (the store is not written by the preceding kernel on
    // the stream) a pair whose first stages are all store tiles requests them
    // before waiting for that kernel; q and the residual window are read only
    // after the wait
    const bool early = a.store_ready && t0 + (kStages - 1) <= a.n_store_tiles;
    if (!early) pdl_wait();
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
        if (k < nt) fetch_tile<BITS>(a, bh, t0 + k, ring + k * kStage, pt);
        cp_async_commit();
    }
    if (early) pdl_wait();

    // q * score_scale for the GQ heads of this KV head (heads >= GQ are zero)
    float qm = 0.f;
#pragma unroll
    for (int i = tid; i < 4 * kD; i += kThreads) {
        const int h = i / kD, d = i % kD;
        const float v = h < GQ ? __half2float(a.q[((long long)b * a.Hq + h0 + h) * kD + d]) * a.score_scale : 0.f;
        q_s[h * kQRow + padc(d)] = v;
        qm = fmaxf(qm, fabsf(v));
    }
    qm = warp_max(qm);
    if (lane == 0) misc[warp] = qm;
    __syncthreads();
    float qmax = misc[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) qmax = fmaxf(qmax, misc[w]);
    const float* qrow = q_s + hh * kQRow;
    const int Er = safe_exp(qmax);  // residual tiles: B operand q 2^Er
    const float fBr = pow2i(Er), fCr = pow2i(-Er);

    // online softmax of head c: m_run is shared by the lanes of equal c (and by both warps);
    // l_run and pzl (sum_t p_t z_tj for this warp's value groups 2hf + jj) are this lane's
    // shares, summed over the lanes of equal c once, after the last tile
    float m_run = -INFINITY, l_run = 0.f;
    float pzl[2] = {0.f, 0.f};
    float o[NO][4];
#pragma unroll
    for (int i = 0; i < NO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    cp_async_wait<kStages - 2>();
    named_sync(bar, 64);  // tile 0 is in shared memory

    for (int it = 0; it < nt; ++it) {
        const int tile = t0 + it;
        const uint8_t* S = ring + (it % kStages) * kStage;
        const bool store = tile < a.n_store_tiles;
        const int nvalid = store ? min(32, a.S_q - tile * 32)
                                 : min(kResTok, a.n_res - (tile - a.n_store_tiles) * kResTok);
        float sc[4];  // partial scores over this warp's 64 channels: tokens g + 8i, head c
        if (store) {
            // ---- B operand: q s 2^E (this lane's head, hi or lo), channels 64hf + 16c + 0..15 ----
            const int cb = 64 * hf + 16 * c;
            const float* KS = reinterpret_cast<const float*>(S + kKS) + padc(cb);
            const float* qb = qrow + padc(cb);
            float s16[16], q16[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 s4 = *reinterpret_cast<const float4*>(KS + 4 * k);
                const float4 q4 = *reinterpret_cast<const float4*>(qb + 4 * k);
                s16[4 * k] = s4.x, s16[4 * k + 1] = s4.y, s16[4 * k + 2] = s4.z, s16[4 * k + 3] = s4.w;
                q16[4 * k] = q4.x, q16[4 * k + 1] = q4.y, q16[4 * k + 2] = q4.z, q16[4 * k + 3] = q4.w;
            }
            float smax = 0.f;  // scales are >= 0
#pragma unroll
            for (int i = 0; i < 16; ++i) smax = fmaxf(smax, s16[i]);
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 1));
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 2));
            const int E = safe_exp(qmax * smax);
            const float fB = pow2i(E);
            // codes enter as fp16 subnormals: channel i's nibble (4-bit) or crumb (2-bit) is worth
            // 16^(i % 2) or 4^(i % 4) times c 2^-24, so its B carries the inverse factor
            const float fC = pow2i(24 - E);
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                v[i] = q16[i] * s16[i] * (BITS == 4 ? ((i & 1) ? fB * 0.0625f : fB) : fB * kOUnit2[0] / kOUnit2[i & 3]);
            uint32_t bq[4][2];  // K-step ks
            if (BITS == 4) {
                // word m: channels cb + 8m + 0..7 (nibble j: channel 8m + j); K-step 2m pairs
                // channels (0,4),(2,6), K-step 2m+1 pairs (1,5),(3,7)
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    bq[2 * m][0] = split_pair(v[8 * m + 0], v[8 * m + 4], lo_part);
                    bq[2 * m][1] = split_pair(v[8 * m + 2], v[8 * m + 6], lo_part);
                    bq[2 * m + 1][0] = split_pair(v[8 * m + 1], v[8 * m + 5], lo_part);
                    bq[2 * m + 1][1] = split_pair(v[8 * m + 3], v[8 * m + 7], lo_part);
                }
            } else {
                // one word: channels cb + 0..15 (crumb j of byte b: channel 4b + j); K-step k
                // pairs channels (k, k+8), (k+4, k+12)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    bq[k][0] = split_pair(v[k], v[k + 8], lo_part);
                    bq[k][1] = split_pair(v[k + 4], v[k + 12], lo_part);
                }
            }
            // ---- sum_d q_d z_d of head c over this warp's 64 channels ----
            float qz_c;
            {
                const int zb = 64 * hf + 8 * (4 * (g & 1) + c);
                const uint4 zw = *reinterpret_cast<const uint4*>(S + kKZ + zb * 2);
                const uint32_t z4[4] = {zw.x, zw.y, zw.z, zw.w};
                const float* qz = qrow + padc(zb);  // 8 contiguous floats
                const float4 qa = *reinterpret_cast<const float4*>(qz);
                const float4 qc = *reinterpret_cast<const float4*>(qz + 4);
                const float q8[8] = {qa.x, qa.y, qa.z, qa.w, qc.x, qc.y, qc.z, qc.w};
                float t = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 zf = __half22float2(u32_as_h2(z4[k]));
                    t = fmaf(q8[2 * k], zf.x, t);
                    t = fmaf(q8[2 * k + 1], zf.y, t);
                }
                t += __shfl_xor_sync(0xffffffffu, t, 1);
                t += __shfl_xor_sync(0xffffffffu, t, 2);
                t += __shfl_xor_sync(0xffffffffu, t, 4);
                qz_c = __shfl_sync(0xffffffffu, t, 8 * c);  // lane 8c has g = 2c: head c
            }
            // ---- partial scores: 2 M-tiles of 16 tokens ----
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int r0 = 16 * mt + g, r1 = r0 + 8;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                if (BITS == 4) {
                    const uint2 x0 = *reinterpret_cast<const uint2*>(S + kKC + r0 * 64 + 32 * hf + 8 * c);
                    const uint2 x1 = *reinterpret_cast<const uint2*>(S + kKC + r1 * 64 + 32 * hf + 8 * c);
                    const uint32_t w0v[2] = {x0.x, x0.y}, w1v[2] = {x1.x, x1.y};
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const uint32_t u0 = w0v[m], u1 = w1v[m], u0s = u0 >> 8, u1s = u1 >> 8;
                        mma16816(acc, u0 & 0x000f000fu, u1 & 0x000f000fu, u0s & 0x000f000fu, u1s & 0x000f000fu,
                                 bq[2 * m][0], bq[2 * m][1]);
                        mma16816(acc, u0 & 0x00f000f0u, u1 & 0x00f000f0u, u0s & 0x00f000f0u, u1s & 0x00f000f0u,
                                 bq[2 * m + 1][0], bq[2 * m + 1][1]);
                    }
                } else {
                    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(S + kKC + r0 * 32 + 16 * hf + 4 * c);
                    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(S + kKC + r1 * 32 + 16 * hf + 4 * c);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t mk = 0x00030003u << (2 * k);
                        mma16816(acc, w0 & mk, w1 & mk, (w0 >> 8) & mk, (w1 >> 8) & mk, bq[k][0], bq[k][1]);
                    }
                }
                sc[2 * mt] = fmaf(acc[0] + acc[1], fC, qz_c);
                sc[2 * mt + 1] = fmaf(acc[2] + acc[3], fC, qz_c);
            }
        } else {
            // residual tile: fp16 K rows, K-steps 4hf .. 4hf + 3 (16 channels each)
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const int q = lane >> 3, r = lane & 7;
            const int row = (q & 1) * 8 + r;
#pragma unroll
            for (int ss = 0; ss < 4; ++ss) {
                const int s = 4 * hf + ss;
                const float2 qa = *reinterpret_cast<const float2*>(qrow + padc(16 * s + 2 * c));
                const float2 qc = *reinterpret_cast<const float2*>(qrow + padc(16 * s + 8 + 2 * c));
                const uint32_t b0 = split_pair(qa.x * fBr, qa.y * fBr, lo_part);
                const uint32_t b1 = split_pair(qc.x * fBr, qc.y * fBr, lo_part);
                const int chunk = 2 * s + (q >> 1);
                uint32_t A[4];
                ldsm_x4(A, S + row * 256 + ((chunk ^ (row & 7)) << 4));
                mma16816(acc, A[0], A[1], A[2], A[3], b0, b1);
            }
            sc[0] = (acc[0] + acc[1]) * fCr;
            sc[1] = (acc[2] + acc[3]) * fCr;
            sc[2] = sc[3] = 0.f;
        }
        float* mine = psc + ((it & 1) * 2 + hf) * 128;
        const float* other = psc + ((it & 1) * 2 + (hf ^ 1)) * 128;
        const int ni = store ? 4 : 2;  // token slots g + 8i of this tile
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (i < ni) mine[(g + 8 * i) * 4 + c] = sc[i];

        cp_async_wait<0>();   // this thread's copies of tile it+1 have landed
        named_sync(bar, 64);  // partner's partial scores and tile it+1 visible; tile it-1 released
        if (it + kStages - 1 < nt)
            fetch_tile<BITS>(a, bh, tile + kStages - 1, ring + ((it + kStages - 1) % kStages) * kStage, pt);
        cp_async_commit();

        // ---- full scores (mine + partner's: the same sum in both warps), online softmax ----
        float s4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = g + 8 * i;
            s4[i] = (i < ni && t < nvalid) ? sc[i] + other[t * 4 + c] : -INFINITY;
        }
        float tmax = fmaxf(fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3]));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        const float m_new = fmaxf(m_run, tmax);  // finite: every tile has a valid token
        const float corr = exp2f(m_run - m_new);
        float p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = exp2f(s4[i] - m_new);
        l_run = fmaf(l_run, corr, (p[0] + p[1]) + (p[2] + p[3]));
        m_run = m_new;
        if (__any_sync(0xffffffffu, corr != 1.f)) {  // the running max moved (x * 1 == x: skip)
#pragma unroll
            for (int i = 0; i < NO; ++i)
#pragma unroll
                for (int k = 0; k < 4; ++k) o[i][k] *= corr;
            pzl[0] *= corr;
            pzl[1] *= corr;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (i < ni) pbuf[(g + 8 * i) * 4 + c] = p[i];
        __syncwarp();

        if (store) {
            const float* VS = reinterpret_cast<const float*>(S + kVS);
            const __half* VZ = reinterpret_cast<const __half*>(S + kVZ);
            // this lane's share of sum_t p_t z_tj (head c, groups j = 2hf + jj; stale rows past
            // nvalid masked)
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * hf + jj;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tk = g + 8 * i;
                    const float z = tk < nvalid ? __half2float(VZ[tk * 4 + j]) : 0.f;
                    pzl[jj] = fmaf(p[i], z, pzl[jj]);
                }
            }
            // B operand: p_t s_tj of head hh; K-step ks: tokens 16ks + {2c, 2c+1 | 2c+8, 2c+9}
            uint32_t bp[2][2][2];  // [jj][ks][b0/b1]
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int ta = 16 * ks + 2 * c, tb = ta + 8;
                const float pa0 = pbuf[ta * 4 + hh], pa1 = pbuf[(ta + 1) * 4 + hh];
                const float pb0 = pbuf[tb * 4 + hh], pb1 = pbuf[(tb + 1) * 4 + hh];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = 2 * hf + jj;
                    const float sa0 = ta < nvalid ? VS[ta * 4 + j] : 0.f;
                    const float sa1 = ta + 1 < nvalid ? VS[(ta + 1) * 4 + j] : 0.f;
                    const float sb0 = tb < nvalid ? VS[tb * 4 + j] : 0.f;
                    const float sb1 = tb + 1 < nvalid ? VS[(tb + 1) * 4 + j] : 0.f;
                    bp[jj][ks][0] = split_pair(pa0 * sa0, pa1 * sa1, lo_part);
                    bp[jj][ks][1] = split_pair(pb0 * sb0, pb1 * sb1, lo_part);
                }
            }
            const uint8_t* VC = S + kVC;
            if (BITS == 4) {
                // o[2jj + u]: rows g -> channel 32j + 4g + u, g+8 -> 32j + 4g + 2 + u (j = 2hf + jj)
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = 2 * hf + jj;
                    const int row = lane;  // matrix lane>>3: tokens 8(lane>>3) .. +7
                    uint32_t W[4];
                    ldsm_x4_t(W, VC + row * 64 + 16 * (j ^ ((row >> 1) & 3)));
                    uint32_t xl[2][4], xh[2][4];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        // bytes of W: token 2c (channels 4g, 4g+1 | 4g+2, 4g+3), token 2c+1 (same)
                        const uint32_t Ws = W[qq] >> 8;
                        xl[0][qq] = W[qq] & 0x000f000fu;
                        xh[0][qq] = Ws & 0x000f000fu;
                        xl[1][qq] = W[qq] & 0x00f000f0u;
                        xh[1][qq] = Ws & 0x00f000f0u;
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks)
                            mma16816(o[2 * jj + u], xl[u][2 * ks], xh[u][2 * ks], xl[u][2 * ks + 1],
                                     xh[u][2 * ks + 1], bp[jj][ks][0], bp[jj][ks][1]);
                    }
                }
            } else {
                // groups 2hf and 2hf + 1 share this warp's 16-byte chunk; as in the
                // one-warp-per-tile kernel, a shuffle hands every lane half (g & 3)
                // of each group and MMA m takes crumb 2m + (g >> 2):
                // o[2grp + m]: row g -> channel 64hf + 32grp + 8(g & 3) + 2m + (g >> 2), row g + 8 -> + 4,
                // in units of 4^(2m + (g >> 2)) 2^-24
                const int row = lane;
                uint32_t W[4];
                ldsm_x4_t(W, VC + row * 32 + 16 * (hf ^ ((row >> 2) & 1)));
                uint32_t X[2][4], Xs[2][4];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    X[0][qq] = __shfl_sync(0xffffffffu, W[qq], lane & 15);
                    X[1][qq] = __shfl_sync(0xffffffffu, W[qq], lane | 16);
                    Xs[0][qq] = X[0][qq] >> 8;
                    Xs[1][qq] = X[1][qq] >> 8;
                }
                const int gh = g >> 2;
#pragma unroll
                for (int grp = 0; grp < 2; ++grp)
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const uint32_t mk = 0x00030003u << (2 * (2 * m + gh));
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks)
                            mma16816(o[2 * grp + m], X[grp][2 * ks] & mk, Xs[grp][2 * ks] & mk,
                                     X[grp][2 * ks + 1] & mk, Xs[grp][2 * ks + 1] & mk, bp[grp][ks][0], bp[grp][ks][1]);
                    }
            }
        } else {
            // residual tile: B = p of head hh (hi or lo), tokens {2c, 2c+1 | 2c+8, 2c+9}; the P.V of
            // each 16-channel block accumulates in fp32 and lands in o (in o's units)
            const uint8_t* VR = S + kRV;
            const uint32_t bp0 = split_pair(pbuf[(2 * c) * 4 + hh], pbuf[(2 * c + 1) * 4 + hh], lo_part);
            const uint32_t bp1 = split_pair(pbuf[(2 * c + 8) * 4 + hh], pbuf[(2 * c + 9) * 4 + hh], lo_part);
            if (BITS == 4) {
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = 2 * hf + jj;
                    uint2 rv[4];  // tokens 2c, 2c+1, 2c+8, 2c+9: channels 32j + 4g .. 32j + 4g + 3
#pragma unroll
                    for (int ti = 0; ti < 4; ++ti) {
                        const int t = 2 * c + (ti & 1) + 8 * (ti >> 1);
                        rv[ti] = *reinterpret_cast<const uint2*>(VR + t * 256 + (((4 * j + (g >> 1)) ^ (t & 7)) << 4) +
                                                                 (g & 1) * 8);
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t sel = u ? 0x7632u : 0x5410u;  // half u of each word
                        float tmp[4] = {0.f, 0.f, 0.f, 0.f};
                        mma16816(tmp, __byte_perm(rv[0].x, rv[1].x, sel), __byte_perm(rv[0].y, rv[1].y, sel),
                                 __byte_perm(rv[2].x, rv[3].x, sel), __byte_perm(rv[2].y, rv[3].y, sel), bp0, bp1);
#pragma unroll
                        for (int k = 0; k < 4; ++k) o[2 * jj + u][k] = fmaf(tmp[k], kOUnit4[u], o[2 * jj + u][k]);
                    }
                }
            } else {
                // the store tiles' layout: o[2grp + m]: row g -> channel 64hf + 32grp + 8(g & 3) + p, row
                // g + 8 -> + 4, with p = 2m + (g >> 2), in units of 4^p 2^-24
                const int gh = g >> 2;
                const uint32_t sel = gh ? 0x7632u : 0x5410u;  // half p & 1 = g >> 2 of each word
#pragma unroll
                for (int grp = 0; grp < 2; ++grp) {
                    uint32_t rv[4][4];  // tokens 2c, 2c+1, 2c+8, 2c+9: channels 64hf + 32grp + 8(g & 3) .. + 7
                    const int chunk = 8 * hf + 4 * grp + (g & 3);
#pragma unroll
                    for (int ti = 0; ti < 4; ++ti) {
                        const int t = 2 * c + (ti & 1) + 8 * (ti >> 1);
                        const uint4 v4 = *reinterpret_cast<const uint4*>(VR + t * 256 + ((chunk ^ (t & 7)) << 4));
                        rv[ti][0] = v4.x;
                        rv[ti][1] = v4.y;
                        rv[ti][2] = v4.z;
                        rv[ti][3] = v4.w;
                    }
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const int wa = m, wb = 2 + m;  // words of halves p and p + 4
                        float tmp[4] = {0.f, 0.f, 0.f, 0.f};
                        mma16816(tmp, __byte_perm(rv[0][wa], rv[1][wa], sel), __byte_perm(rv[0][wb], rv[1][wb], sel),
                                 __byte_perm(rv[2][wa], rv[3][wa], sel), __byte_perm(rv[2][wb], rv[3][wb], sel), bp0,
                                 bp1);
                        const float unit = pow2i(2 * (2 * m + gh) - 24);
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[2 * grp + m][e] = fmaf(tmp[e], unit, o[2 * grp + m][e]);
                    }
                }
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();

    // ---------------------------- merge the pairs ----------------------------
    // Each warp rescales its accumulators by 2^(m_pair - M) (M: the CTA's
    // largest running max of the head) before they meet in shared memory, so
    // the cross-pair combine is a plain sum.
    __syncthreads();  // every pair is done with its ring
    float* Ow = reinterpret_cast<float*>(ring);  // [4 heads][128] of this pair (each warp its 64 channels)
    float* ml = misc + 16;                        // [pair][head][2]: m, then l * 2^(m - M)
    float* Mh = misc + 8;                         // [head]: M
    // l and sum_t p_t z_tj of head c: the lanes of equal c hold disjoint tokens
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
        l_run += __shfl_xor_sync(0xffffffffu, l_run, x);
        pzl[0] += __shfl_xor_sync(0xffffffffu, pzl[0], x);
        pzl[1] += __shfl_xor_sync(0xffffffffu, pzl[1], x);
    }
    if (hf == 0 && g == 0) ml[(pair * 4 + c) * 2] = m_run;
    __syncthreads();
    {
        float Mc = -INFINITY;
#pragma unroll
        for (int pp = 0; pp < kPairs; ++pp) Mc = fmaxf(Mc, ml[(pp * 4 + c) * 2]);
        const float f = m_run == -INFINITY ? 0.f : exp2f(m_run - Mc);  // a pair without tiles adds nothing
        // o holds sum p s c in units of kOUnit4 / kOUnit2; the z term adds per value group
        if (BITS == 4) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int j = 2 * hf + jj;
                    const float sc = f / kOUnit4[u], zf = pzl[jj] * f;
                    Ow[c * kD + 32 * j + 4 * g + u] = fmaf(o[2 * jj + u][0] + o[2 * jj + u][1], sc, zf);
                    Ow[c * kD + 32 * j + 4 * g + 2 + u] = fmaf(o[2 * jj + u][2] + o[2 * jj + u][3], sc, zf);
                }
        } else {
            const int gh = g >> 2;
#pragma unroll
            for (int grp = 0; grp < 2; ++grp) {
                const float zf = pzl[grp] * f;
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int pc = 2 * m + gh;  // crumb position: units 4^pc 2^-24
                    const float sc = f * pow2i(24 - 2 * pc);
                    const int ch = 64 * hf + 32 * grp + 8 * (g & 3) + pc;
                    Ow[c * kD + ch] = fmaf(o[2 * grp + m][0] + o[2 * grp + m][1], sc, zf);
                    Ow[c * kD + ch + 4] = fmaf(o[2 * grp + m][2] + o[2 * grp + m][3], sc, zf);
                }
            }
        }
        if (hf == 0 && g == 0) {
            ml[(pair * 4 + c) * 2 + 1] = l_run * f;
            if (pair == 0) Mh[c] = Mc;
        }
    }
    pdl_trigger();
    __syncthreads();
    for (int i4 = tid; i4 < GQ * (kD / 4); i4 += kThreads) {
        const int h = i4 / (kD / 4), d = 4 * (i4 % (kD / 4));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
#pragma unroll
        for (int pp = 0; pp < kPairs; ++pp) {
            const float4 v =
                *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(smem + pp * kStages * kStage) + h * kD + d);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
            L += ml[(pp * 4 + h) * 2 + 1];
        }
        const float M = Mh[h];
        const long long bq = (long long)b * a.Hq + h0 + h;
        if (a.n_split == 1) {
            const float r = 1.0f / L;
            *reinterpret_cast<float4*>(a.out + bq * kD + d) = make_float4(acc.x * r, acc.y * r, acc.z * r, acc.w * r);
        } else if (CL) {  // the partial stays in this CTA's shared memory (the q area is free now)
            *reinterpret_cast<float4*>(q_s + h * kD + d) = acc;
            if (d == 0) {
                misc[100 + 2 * h] = M;
                misc[101 + 2 * h] = L;
            }
        } else {
            __stcg(reinterpret_cast<float4*>(a.part_o + (bq * a.n_split + split) * kD + d), acc);
            if (d == 0)
                __stcg(reinterpret_cast<float2*>(a.part_ml + (bq * a.n_split + split) * 2), make_float2(M, L));
        }
    }
    if (a.n_split == 1) return;
    if (CL) {
        cluster_sync();
        const uint32_t rank = cluster_ctarank();
        const int n = a.n_split;
        for (int idx = (int)rank * kThreads + tid; idx < GQ * kD; idx += n * kThreads) {
            const int h = idx / kD, dd = idx % kD;
            float mk[kMaxClusterSplits];
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < kMaxClusterSplits; ++k) {
                mk[k] = k < n ? ld_cluster(misc + 100 + 2 * h, k) : -INFINITY;
                M = fmaxf(M, mk[k]);
            }
            float L = 0.f, acc = 0.f;
#pragma unroll
            for (int k = 0; k < kMaxClusterSplits; ++k) {
                if (k < n && mk[k] != -INFINITY) {
                    const float wk = exp2f(mk[k] - M);
                    L = fmaf(ld_cluster(misc + 101 + 2 * h, k), wk, L);
                    acc = fmaf(ld_cluster(q_s + h * kD + dd, k), wk, acc);
                }
            }
            a.out[((long long)b * a.Hq + h0 + h) * kD + dd] = acc / L;
        }
        cluster_sync();
        return;
    }
    if (take_last_ticket(a, bh, reinterpret_cast<int*>(misc + 96)))
        merge_splits<kWarps, kD>(a, (long long)b * a.Hq + h0, GQ, warp, lane);
}

template <int BITS, int GQ, bool CL>
cudaError_t configure_pair() {
    static cudaError_t status = cudaErrorNotReady;  // benign race: every caller sets the same values
    if (status == cudaErrorNotReady) {
        cudaError_t e = cudaFuncSetAttribute(decode_pair_kernel<BITS, GQ, CL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e == cudaSuccess && CL)
            e = cudaFuncSetAttribute(decode_pair_kernel<BITS, GQ, CL>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                     1);
        status = e;
    }
    return status;
}

// Resident CTAs in clusters of n (0 if such clusters cannot be resident):
// occupancy calculator, once per device and n.
template <int BITS, int GQ>
int pair_cluster_ctas(int n, cudaStream_t stream) {
    constexpr int kDevs = 16;
    static int cache[kDevs][kMaxClusterSplits + 1];  // 0 unknown, -1 none, else CTAs + 1
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs || n < 2 || n > kMaxClusterSplits) {
        cudaGetLastError();
        return 0;
    }
    if (cache[dev][n] == 0) {
        int ctas = 0;
        if (configure_pair<BITS, GQ, true>() == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(n, 1, 1);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = kSmemBytes;
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = n;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, decode_pair_kernel<BITS, GQ, true>, &cfg) == cudaSuccess)
                ctas = clusters * n;
        }
        cudaGetLastError();
        cache[dev][n] = ctas > 0 ? ctas + 1 : -1;
    }
    return cache[dev][n] > 0 ? cache[dev][n] - 1 : 0;
}

// The splits of a head merge inside a cluster when the whole grid fits in one
// wave of resident clusters (the kernel serves small batches) and has at
// least as many CTAs as SMs; a smaller grid spreads one CTA per SM and merges
// through the workspace (13 splits at B=1: 6.1 us against 6.9 in clusters).
template <int BITS, int GQ>
cudaError_t launch_pair_typed(const DecodeArgs& a, cudaStream_t stream) {
    const dim3 grid(a.n_split, a.Hkv, a.B);
    const int n = a.n_split;
    const long long ctas = (long long)n * a.Hkv * a.B;
    if (n >= 2 && n <= kMaxClusterSplits && ctas >= sm_count() && ctas <= pair_cluster_ctas<BITS, GQ>(n, stream)) {
        cudaError_t e = configure_pair<BITS, GQ, true>();
        if (e != cudaSuccess) return e;
        return launch_pdl_cluster(decode_pair_kernel<BITS, GQ, true>, grid, kThreads, kSmemBytes, stream, n, a);
    }
    cudaError_t e = configure_pair<BITS, GQ, false>();
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_pair_kernel<BITS, GQ, false>, grid, kThreads, kSmemBytes, stream, a);
}

}  // namespace

cudaError_t launch_decode_pair(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    cudaError_t e = cudaErrorInvalidValue;
    if (bits == 4) {
        if (gq == 1) e = launch_pair_typed<4, 1>(a, stream);
        if (gq == 2) e = launch_pair_typed<4, 2>(a, stream);
        if (gq == 4) e = launch_pair_typed<4, 4>(a, stream);
    } else {
        if (gq == 1) e = launch_pair_typed<2, 1>(a, stream);
        if (gq == 2) e = launch_pair_typed<2, 2>(a, stream);
        if (gq == 4) e = launch_pair_typed<2, 4>(a, stream);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kivi

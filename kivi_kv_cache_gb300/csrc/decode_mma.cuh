// decode_mma.cuh -- fused dequantize-and-attend single-token decode on the
// tensor cores (mma.sync m16n8k16, fp16 operands, fp32 accumulation), one warp
// per tile, for groups of up to 4 query heads per KV head; larger groups run
// in sub-groups of up to 4 heads (one CTA group each, reading the same tiles).
// Templated on the head dim D (64, 128, 256) and on the scale storage (fp32
// or fp16); decode_mma.cu, decode_mma_f16s.cu, decode_mma_d64.cu,
// decode_mma_d256.cu and decode_mma_d256_f16s.cu split the instantiations so
// that they compile in parallel.
//
// Method: VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly
// 0% Faster", "So why does the kernel ship?" (attention reads the packed
// codes and expands them in registers), and the VeloxQuant-MLX benchmarks
// page, "KV-Cache Kernel Roofline" (one query token per head; too few
// threadgroups per (batch, head) leave the GPU idle, so the cached tokens
// are split across CTAs and merged by a log-sum-exp combine).
//
// Why tensor cores: with 4 query heads per KV head every packed byte feeds
// ~6 multiply-adds (1024 per token of K and V at 4-bit, 176 bytes), more
// than the fp32 pipes sustain at HBM rate. The dequant is folded out of the
// contraction (a key group shares s_d, z_d per channel; a value row shares
// s_j, z_j per 32-channel group):
//     q . khat_t  = sum_d (q_d s_d) c_td + sum_d q_d z_d
//     sum_t p_t vhat_td = sum_t (p_t s_tj) c_td + sum_t p_t z_tj
// so the codes c are one MMA operand, exactly representable in fp16, and the
// fp32 products q_d s_d / p_t s_tj the other. Exactness of the operands:
//   * a code masked in place within a 16-bit half is an fp16 subnormal: a
//     nibble at bit 4j is c 16^j 2^-24, a crumb at bit 2j is c 4^j 2^-24, so
//     one AND turns two codes into an exact fp16 pair; the factor 16^j or 4^j
//     goes into the q_d s_d operand (scores) or into the units of the P.V
//     accumulator (one per nibble or crumb position), and the tensor cores
//     take subnormal fp16 operands exactly;
//   * each fp32 operand is split into fp16 hi + lo (hi = fp16(x), lo =
//     fp16(x - hi)), carried as two MMA columns per query head: n = 2h + part.
//     The sum keeps ~22 significant bits, far below the 2e-3 output budget;
//   * a per-tile power-of-two factor keeps every hi below 2^14 (no fp16
//     overflow for any finite input); it is divided out exactly afterwards.
//
// Work split: grid (n_split, Hkv * q_sub, B), 2, 4 or 8 warps per CTA; each warp owns a
// contiguous run of tiles of its split (32-token store tiles, then 16-token
// residual tiles) and keeps its own online softmax; the warps merge in shared
// memory and the CTA writes one partial (or the output when n_split == 1; the
// last CTA of a (batch, KV head) merges the partials, see decode_merge.cuh).
// Tiles are staged per warp with cp.async, double buffered: packed K/V codes,
// key scale/zero of the group, value scale/zero of the 32 rows (5.6 KB at
// 4-bit and D = 128); residual tiles stage 16 fp16 K and V rows (zero-filled
// past n_res). At D = 128: 128 registers and 50 KB (4 warps) or 97 KB (8
// warps) of shared memory per CTA, 16 warps per SM either way; D = 64 halves
// the stages, D = 256 doubles them and runs 8 warps per SM. 8-warp CTAs halve
// the partials a merge reads; the plan takes them when 4-warp CTAs would leave
// more than 16 splits. 2-warp CTAs (27 KB, D = 128 only) split a head group
// finer when short warp runs would otherwise leave a ragged wave.
// MMA layouts (m16n8k16, row.col): lane = 4 g + c; A regs hold (row g,
// k 2c..2c+1), (row g+8, same k), (row g, k 2c+8..9), (row g+8, k 2c+8..9);
// B regs (k 2c..2c+1, n g), (k 2c+8..9, n g); C regs (row g, n 2c..2c+1),
// (row g+8, n 2c..2c+1).
#pragma once

#include <math.h>

#include <type_traits>

#include "decode_common.cuh"
#include "decode_merge.cuh"
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

namespace {

using namespace dec;

// Shared-memory geometry of head dim D (64, 128 or 256). A store tile holds
// 32 token rows: K codes [32][D/2] linear, V codes [32][D/2] with the 16-byte
// chunks of a row swizzled, the key scales padded like q (channel ch at
// ch + (ch >> 5) * 4), key zeros, value scales and zeros [32][D/32] (one
// entry per 32 channels); 2-bit tiles use the first half of each code area.
// A residual tile holds kResTok fp16 K rows in one stage and V rows in the
// other (16-byte chunk c of row r at c ^ (r & 7)).
template <int D>
struct Geo {
    static constexpr int kKC = 0;
    static constexpr int kVC = 16 * D;
    static constexpr int kKS = 32 * D;
    static constexpr int kKZ = kKS + (D + D / 8) * 4;
    static constexpr int kVS = kKZ + 2 * D;
    static constexpr int kVZ = kVS + 4 * D;
    static constexpr int kTileBytes = kVZ + 2 * D;                // 2848, 5696, 11392
    static constexpr int kStage = (kTileBytes + 127) / 128 * 128;  // bytes per stage
    static constexpr int kWarpSmem = 2 * kStage;                   // two stages per warp
    static constexpr int kQRow = D + D / 8;                        // padded q row
    static constexpr int kNE = D / 32;                             // value groups of 32 channels per row
    static_assert(kResTileTokensMma * 2 * D <= kStage, "a residual tile fits a stage");
};

// Shared memory of a CTA of NW warps: each warp's two stages, per-warp p
// buffers [32][4] f32, q * score_scale [4][kQRow] f32, then misc: qmax per
// warp [8], the warps' (m, l) [NW][4][2] at 16, the merge flag at 96, the
// cluster (m, l) at 100.
template <int NW, int D>
struct Layout {
    static constexpr int kPbufOff = NW * Geo<D>::kWarpSmem;
    static constexpr int kQOff = kPbufOff + NW * 512;
    static constexpr int kMiscOff = kQOff + 4 * Geo<D>::kQRow * 4;
    static constexpr int kSmemBytes = kMiscOff + 512;
};
constexpr int kResTok = kResTileTokensMma;  // residual tile: 16 K rows in stage 0, 16 V rows in stage 1

// Resident warps per SM: 16 at 128 registers, 8 at D = 256 (its stages and
// accumulators are twice as large).
template <int D>
__host__ __device__ constexpr int warps_per_sm() { return D == 256 ? 8 : 16; }

__device__ __forceinline__ int padc(int ch) { return ch + ((ch >> 5) << 2); }

// N consecutive 32-bit words from shared memory (N = 1, 2, 4 or 8) in the
// widest aligned loads: one 4-, 8- or 16-byte load, or two 16-byte loads
template <int N>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&w)[N]) {
    if constexpr (N == 1) {
        w[0] = *reinterpret_cast<const uint32_t*>(p);
    } else if constexpr (N == 2) {
        const uint2 x = *reinterpret_cast<const uint2*>(p);
        w[0] = x.x;
        w[1] = x.y;
    } else {
        static_assert(N % 4 == 0, "1, 2 or a multiple of 4 words");
#pragma unroll
        for (int k = 0; k < N / 4; ++k) {
            const uint4 x = *reinterpret_cast<const uint4*>(p + 16 * k);
            w[4 * k] = x.x;
            w[4 * k + 1] = x.y;
            w[4 * k + 2] = x.z;
            w[4 * k + 3] = x.w;
        }
    }
}

// physical 16-byte chunk of logical chunk col in row `row` of a code area with
// CPR chunks per row: rows are XOR-swizzled so that the 8 rows one ldmatrix
// matrix reads fall in distinct bank groups
template <int CPR>
__device__ __forceinline__ int swz(int row, int col) {
    return CPR == 1 ? col : col ^ ((row / (8 / CPR)) & (CPR - 1));
}


// ---------------------------------------------------------------------------
// tile staging
// ---------------------------------------------------------------------------

template <int BITS, int D, bool HS>
__device__ __forceinline__ void fetch_store_tile(const DecodeArgs& a, int bh, int tile, uint8_t* st, int lane) {
    using GE = Geo<D>;
    constexpr int ROWB = D * BITS / 8;       // bytes per code row
    constexpr int CPR = ROWB / 16;           // 16-byte chunks per code row: 1 .. 8
    const int tok0 = tile * 32;
    const uint8_t* kc = a.kcodes + ((long long)bh * a.s_cap + tok0) * ROWB;
    const uint8_t* vc = a.vcodes + ((long long)bh * a.s_cap + tok0) * ROWB;
#pragma unroll
    for (int i = lane; i < 32 * CPR; i += 32) {
        const int row = i / CPR, col = i % CPR;
        cp_async16(st + GE::kKC + i * 16, kc + i * 16, true);
        cp_async16(st + GE::kVC + row * ROWB + swz<CPR>(row, col) * 16, vc + i * 16, true);
    }
    // the key group (32 << g_shift tokens) holding this tile, and the value
    // metadata of its 32 tokens: (D / 32) >> g_shift entries per token, packed
    // at the front of VS and VZ (widen_value_meta spreads them for G > 32).
    // fp16 scales (HS) land in plain channel order at the front of KS and VS
    // and are read as fp16 by the tile code.
    const int sh = a.g_shift;
    const long long krow = (long long)bh * (a.s_cap >> (5 + sh)) + (tile >> sh);
    const long long vrow = ((long long)bh * a.s_cap + tok0) * ((D / 32) >> sh);
    const int nvz = (D / 8) >> sh;  // 16-byte chunks of the 32 tokens' zeros (and fp16 scales)
    if (HS) {
        const __half* ks = reinterpret_cast<const __half*>(a.kscale) + krow * D;
        const __half* vs = reinterpret_cast<const __half*>(a.vscale) + vrow;
        if (lane < D / 8) cp_async16(st + GE::kKS + lane * 16, ks + lane * 8, true);
        if (lane < nvz) cp_async16(st + GE::kVS + lane * 16, vs + lane * 8, true);
    }
    const float* ks = a.kscale + krow * D;
    const __half* kz = a.kzero + krow * D;
    if (!HS) {
#pragma unroll
        for (int i = lane; i < D / 4; i += 32) cp_async16(st + GE::kKS + padc(i * 4) * 4, ks + i * 4, true);
    }
    if (lane < D / 8) cp_async16(st + GE::kKZ + lane * 16, kz + lane * 8, true);
    const float* vs = a.vscale + vrow;
    const __half* vz = a.vzero + vrow;
    const int nvs = (D / 4) >> sh;  // 16-byte chunks of the 32 tokens' fp32 scales
    if (!HS) {
#pragma unroll
        for (int i = lane; i < D / 4; i += 32)
            if (i < nvs) cp_async16(st + GE::kVS + i * 16, vs + i * 4, true);
    }
    if (lane < nvz) cp_async16(st + GE::kVZ + lane * 16, vz + lane * 8, true);
}

// A store of group size 64 (g_shift 1) or 128 (g_shift 2) has 2 or 4 times
// fewer value scales and zeros per token than the tile code reads (VS and VZ
// [32 tokens][D / 32], one entry per 32 channels). Each lane takes its
// token's entries, then, once the warp has read them all, writes them back
// with each repeated 2 or 4 times. Value scales are fp32, or fp16 (HS); key
// scales need no change (fp32 in padded channel order, or fp16 in plain
// channel order, which the tile code reads as such).
template <int D, bool HS>
__device__ __forceinline__ void widen_value_meta(uint8_t* st, int sh, int lane) {
    using GE = Geo<D>;
    constexpr int NE = GE::kNE;
    using ST = typename std::conditional<HS, unsigned short, float>::type;  // one stored scale
    ST* vs = reinterpret_cast<ST*>(st + GE::kVS);
    unsigned short* vz = reinterpret_cast<unsigned short*>(st + GE::kVZ);
    const int nr = NE >> sh;  // entries per token in the store
    ST s[NE];
    unsigned short z[NE];
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        const int idx = lane * nr + (e >> sh);
        s[e] = vs[idx];
        z[e] = vz[idx];
    }
    __syncwarp();
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        vs[lane * NE + e] = s[e];
        vz[lane * NE + e] = z[e];
    }
    __syncwarp();
}

// fp16 scales of the staged tile (HS) as fp32: key scales of channels cb ..
// cb + 7 (cb a multiple of 8) or cb .. cb + 3 (a multiple of 4), in plain
// channel order at ks; the NE value scales of token t at vs ([32][NE]).
__device__ __forceinline__ void key_scales8_h(const uint8_t* ks, int cb, float4& a, float4& b) {
    const uint4 h = *reinterpret_cast<const uint4*>(ks + 2 * cb);
    const float2 f0 = __half22float2(u32_as_h2(h.x)), f1 = __half22float2(u32_as_h2(h.y));
    const float2 f2 = __half22float2(u32_as_h2(h.z)), f3 = __half22float2(u32_as_h2(h.w));
    a = make_float4(f0.x, f0.y, f1.x, f1.y);
    b = make_float4(f2.x, f2.y, f3.x, f3.y);
}
__device__ __forceinline__ float4 key_scales4_h(const uint8_t* ks, int cb) {
    const uint2 h = *reinterpret_cast<const uint2*>(ks + 2 * cb);
    const float2 f0 = __half22float2(u32_as_h2(h.x)), f1 = __half22float2(u32_as_h2(h.y));
    return make_float4(f0.x, f0.y, f1.x, f1.y);
}
template <int NE>
__device__ __forceinline__ void value_scales_h(const uint8_t* vs, int t, float (&x)[NE]) {
    uint32_t w[NE / 2];
    load_words<NE / 2>(vs + 2 * NE * t, w);
#pragma unroll
    for (int e = 0; e < NE / 2; ++e) {
        const float2 f = __half22float2(u32_as_h2(w[e]));
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}

// kResTok fp16 rows of K into st0 and of V into st1, 16-byte chunk c of row r
// at position c ^ (r & 7); rows past nvalid are zero-filled (nothing is read).
template <int D>
__device__ __forceinline__ void fetch_res_tile(const DecodeArgs& a, int bh, int rtile, int nvalid, uint8_t* st0,
                                               uint8_t* st1, int lane) {
    constexpr int CPR = D / 8;  // 16-byte chunks per fp16 row
    const int tok0 = rtile * kResTok;
    const __half* kr = a.k_res + ((long long)bh * a.res_cap + tok0) * D;
    const __half* vr = a.v_res + ((long long)bh * a.res_cap + tok0) * D;
#pragma unroll 4
    for (int i = lane; i < kResTok * CPR; i += 32) {
        const int row = i / CPR, col = i % CPR;
        const bool ok = row < nvalid;
        const int off = row * (2 * D) + ((col ^ (row & 7)) << 4);
        cp_async16(st0 + off, ok ? (const void*)(kr + row * D + col * 8) : (const void*)kr, ok);
        cp_async16(st1 + off, ok ? (const void*)(vr + row * D + col * 8) : (const void*)vr, ok);
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

// GQ = 1, 2 or 4: the group size, blockIdx.y = KV head. GQ = kSubGroupGQ: any
// other group size, in sub-groups of 4 heads (blockIdx.y = KV head times q_sub
// + sub-group; the last sub-group possibly partial).
constexpr int kSubGroupGQ = 8;
template <int GQ>
__device__ __forceinline__ int cta_kv_head(const DecodeArgs& a) {
    return GQ == kSubGroupGQ ? (int)blockIdx.y / a.q_sub : (int)blockIdx.y;
}
// Query heads h0 .. h0 + nh - 1 (of the batch row) of this CTA.
template <int GQ>
__device__ __forceinline__ void cta_heads(const DecodeArgs& a, int& h0, int& nh) {
    if (GQ == kSubGroupGQ) {
        const int gq = a.Hq / a.Hkv;
        const int hk = (int)blockIdx.y / a.q_sub, sg = (int)blockIdx.y - hk * a.q_sub;
        h0 = hk * gq + 4 * sg;
        nh = min(4, gq - 4 * sg);
    } else {
        h0 = (int)blockIdx.y * GQ;
        nh = GQ;
    }
}

// NW warps per CTA (2, 4 or 8): 16 warps per SM at 128 registers
// (D <= 128), or 8 at up to 255 registers (D = 256).
// CL: the n_split CTAs of a (batch, KV head) form one thread-block cluster
// (n_split <= kMaxClusterSplits) and merge through distributed shared memory.
// D: head dim. A lane's share of a code row is D / 4 contiguous channels; the
// score operands are built and applied in chunks of at most 128 channels so
// that D = 256 holds no more of them at a time than D = 128.
template <int BITS, int GQ, int NW, bool CL, int D, bool HS>
__global__ void __launch_bounds__(32 * NW, warps_per_sm<D>() / NW) decode_mma_kernel(DecodeArgs a) {
    constexpr int kWarps = NW;
    constexpr int kThreads = 32 * NW;
    using LY = Layout<NW, D>;
    using GE = Geo<D>;
    constexpr int kStage = GE::kStage;
    constexpr int kQRow = GE::kQRow;
    constexpr int NE = GE::kNE;  // 32-channel value groups per row
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int split = blockIdx.x, b = blockIdx.z;
    const int bh = b * a.Hkv + cta_kv_head<GQ>(a);
    uint8_t* const st0 = smem + warp * GE::kWarpSmem;  // two stages: st0, st0 + kStage
    float* pbuf = reinterpret_cast<float*>(smem + LY::kPbufOff + warp * 512);  // [token][head]
    float* q_s = reinterpret_cast<float*>(smem + LY::kQOff);                   // [head][channel]
    float* misc = reinterpret_cast<float*>(smem + LY::kMiscOff);

    // this warp's tiles: the head's n_tiles spread evenly over its n_split * NW warps
    const long long nw_head = (long long)a.n_split * kWarps, gw = (long long)split * kWarps + warp;
    const int w0 = (int)(gw * a.n_tiles / nw_head);
    const int w1 = (int)((gw + 1) * a.n_tiles / nw_head);
    const int s_end = min(w1, a.n_store_tiles);           // store tiles [w0, s_end)
    const int r_begin = max(w0, a.n_store_tiles);         // residual tiles [r_begin, w1)
    const int ns = s_end - w0;

    // start the first store tile's copy, then stage q while it flies; with
    // store_ready (the store is not written by the preceding kernel on the
    // stream) the copy starts before waiting for that kernel, and q and the
    // residual window are read only after the wait. Each warp requests one
    // tile ahead (the next one when the current one has landed): every SM
    // still has more bytes in flight than the HBM latency-bandwidth product
    // needs, and a launch's first tiles arrive about twice as early as with
    // two tiles requested up front.
    if (!a.store_ready) pdl_wait();
    if (ns > 0) fetch_store_tile<BITS, D, HS>(a, bh, w0, st0, lane);
    cp_async_commit();
    if (a.store_ready) pdl_wait();

    // q * score_scale for the nh heads of this CTA (heads >= nh are zero)
    float qm = 0.f;
    {
        int h0, nh;
        cta_heads<GQ>(a, h0, nh);
#pragma unroll
        for (int i = tid; i < 4 * D; i += kThreads) {
            const int h = i / D, d = i % D;
            const float v = h < nh ? __half2float(a.q[((long long)b * a.Hq + h0 + h) * D + d]) * a.score_scale : 0.f;
            q_s[h * kQRow + padc(d)] = v;
            qm = fmaxf(qm, fabsf(v));
        }
    }
    qm = warp_max(qm);
    if (lane == 0) misc[warp] = qm;
    __syncthreads();
    float qmax = misc[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) qmax = fmaxf(qmax, misc[w]);

    const int hh = g >> 1;          // head of this lane's B column n = g
    const bool lo_part = g & 1;     // hi (0) or lo (1) part of that column
    const float* qrow = q_s + hh * kQRow;

    // residual tiles take q 2^Er (hi or lo) in natural channel order as their B operand
    const int Er = safe_exp(qmax);
    const float fBr = pow2i(Er), fCr = pow2i(-Er);

    // online softmax of head c: m_run is shared by the lanes of equal c; l_run
    // and pzl (sum_t p_t z_tj per value group j) are this lane's shares, summed
    // over the lanes of equal c once, after the last tile
    float m_run = -INFINITY, l_run = 0.f;
    float pzl[NE];
#pragma unroll
    for (int j = 0; j < NE; ++j) pzl[j] = 0.f;
    float o[D / 16][4];                    // P.V of head c, store-tile channel layout
#pragma unroll
    for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    // ---------------------------- store tiles ----------------------------
    for (int it = 0; it < ns; ++it) {
        const int tile = w0 + it;
        uint8_t* S = st0 + (it & 1) * kStage;
        cp_async_wait<0>();  // this tile
        __syncwarp();
        if (it + 1 < ns) fetch_store_tile<BITS, D, HS>(a, bh, tile + 1, st0 + ((it + 1) & 1) * kStage, lane);
        cp_async_commit();
        if (a.g_shift != 0) widen_value_meta<D, HS>(S, a.g_shift, lane);
        const int nvalid = min(32, a.S_q - tile * 32);
        if (nvalid < 32) {  // zero the value metadata of rows past S_q
            using ST = typename std::conditional<HS, unsigned short, float>::type;
            ST* vsz = reinterpret_cast<ST*>(S + GE::kVS);
            unsigned short* vzz = reinterpret_cast<unsigned short*>(S + GE::kVZ);
            if (lane >= nvalid) {
#pragma unroll
                for (int j = 0; j < NE; ++j) {
                    vsz[lane * NE + j] = 0;
                    vzz[lane * NE + j] = 0;
                }
            }
            __syncwarp();
        }
        const float* KS = reinterpret_cast<const float*>(S + GE::kKS);
        const __half* KZ = reinterpret_cast<const __half*>(S + GE::kKZ);
        const float* VS = reinterpret_cast<const float*>(S + GE::kVS);
        const __half* VZ = reinterpret_cast<const __half*>(S + GE::kVZ);

        // ---- QK operand B: q s 2^E for this lane's channels, hi or lo ----
        float smax = 0.f;
#pragma unroll
        for (int i = lane; i < D / 4; i += 32) {
            float4 s4;  // scales are >= 0
            if constexpr (HS) s4 = key_scales4_h(S + GE::kKS, 4 * i);
            else s4 = *reinterpret_cast<const float4*>(KS + padc(4 * i));
            smax = fmaxf(smax, fmaxf(fmaxf(s4.x, s4.y), fmaxf(s4.z, s4.w)));
        }
        smax = warp_max(smax);
        const int E = safe_exp(qmax * smax);
        const float fB = pow2i(E);  // B = q s 2^E
        // codes enter the MMA as fp16 subnormals (a nibble at bit 4j of a half
        // is c 16^j 2^-24, a crumb at bit 2j is c 4^j 2^-24); B of that
        // channel carries 16^-j or 4^-j
        const float fC = pow2i(24 - E);  // score = C 2^(24-E)
        const f32x2 fB2 = BITS == 4 ? pk(fB, fB * 0.0625f) : pk(fB, fB * 0.25f);
        const f32x2 fB2h = pk(fB * 0.0625f, fB * 0.015625f);  // 2-bit crumbs 2, 3 of a byte

        // ---- sum_d q_d z_d of head c: this lane sums D / 8 channels of head hh ----
        float qz_c;
        {
            const int cb = (D / 8) * (4 * (g & 1) + c);
            const float* qz = qrow + padc(cb);  // D / 8 contiguous floats
            float t = 0.f;
#pragma unroll
            for (int v8 = 0; v8 < D / 64; ++v8) {
                const uint4 zv = *reinterpret_cast<const uint4*>(KZ + cb + 8 * v8);
                const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w};
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float4 q4 = *reinterpret_cast<const float4*>(qz + 8 * v8 + 4 * k);
                    const float2 z01 = __half22float2(u32_as_h2(zw[2 * k]));
                    const float2 z23 = __half22float2(u32_as_h2(zw[2 * k + 1]));
                    t = fmaf(q4.x, z01.x, t);
                    t = fmaf(q4.y, z01.y, t);
                    t = fmaf(q4.z, z23.x, t);
                    t = fmaf(q4.w, z23.y, t);
                }
            }
            t += __shfl_xor_sync(0xffffffffu, t, 1);
            t += __shfl_xor_sync(0xffffffffu, t, 2);
            t += __shfl_xor_sync(0xffffffffu, t, 4);
            qz_c = __shfl_sync(0xffffffffu, t, 8 * c);  // lane 8c has g = 2c: head c
        }

        // ---- scores: 2 M-tiles of 16 tokens, channel chunks of at most 128 ----
        const uint8_t* KC = S + GE::kKC;
        constexpr int ROWB = D * BITS / 8;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (BITS == 4) {
            // word m of this lane's D / 8 bytes: channels (D / 4) c + 8m + {0..7}
            // (channel 8m + j in nibble j); K-step 2m pairs channels (0,4),(2,6),
            // K-step 2m+1 pairs (1,5),(3,7)
            constexpr int NWD = D / 32;                 // words per lane
            constexpr int WPC = NWD < 4 ? NWD : 4;      // words per chunk
#pragma unroll
            for (int ch = 0; ch < NWD / WPC; ++ch) {
                uint32_t bq[2 * WPC][2];
#pragma unroll
                for (int mm = 0; mm < WPC; ++mm) {
                    const int cb = (D / 4) * c + 8 * (WPC * ch + mm);
                    float4 sa, sb;
                    if constexpr (HS) {
                        key_scales8_h(S + GE::kKS, cb, sa, sb);
                    } else {
                        sa = *reinterpret_cast<const float4*>(KS + padc(cb));
                        sb = *reinterpret_cast<const float4*>(KS + padc(cb + 4));
                    }
                    const float4 qa = *reinterpret_cast<const float4*>(qrow + padc(cb));
                    const float4 qb = *reinterpret_cast<const float4*>(qrow + padc(cb + 4));
                    const float2 v01 = upk(mul2(mul2(pk(qa.x, qa.y), pk(sa.x, sa.y)), fB2));
                    const float2 v23 = upk(mul2(mul2(pk(qa.z, qa.w), pk(sa.z, sa.w)), fB2));
                    const float2 v45 = upk(mul2(mul2(pk(qb.x, qb.y), pk(sb.x, sb.y)), fB2));
                    const float2 v67 = upk(mul2(mul2(pk(qb.z, qb.w), pk(sb.z, sb.w)), fB2));
                    bq[2 * mm][0] = split_pair(v01.x, v45.x, lo_part);
                    bq[2 * mm][1] = split_pair(v23.x, v67.x, lo_part);
                    bq[2 * mm + 1][0] = split_pair(v01.y, v45.y, lo_part);
                    bq[2 * mm + 1][1] = split_pair(v23.y, v67.y, lo_part);
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int r0 = mt * 16 + g, r1 = r0 + 8;
                    uint32_t w0v[WPC], w1v[WPC];
                    const uint8_t* p0 = KC + r0 * ROWB + (D / 8) * c + 16 * ch;
                    const uint8_t* p1 = KC + r1 * ROWB + (D / 8) * c + 16 * ch;
                    load_words<WPC>(p0, w0v);
                    load_words<WPC>(p1, w1v);
#pragma unroll
                    for (int mm = 0; mm < WPC; ++mm) {
                        const uint32_t u0 = w0v[mm], u1 = w1v[mm], u0s = u0 >> 8, u1s = u1 >> 8;
                        mma16816(acc[mt], u0 & 0x000f000fu, u1 & 0x000f000fu, u0s & 0x000f000fu,
                                 u1s & 0x000f000fu, bq[2 * mm][0], bq[2 * mm][1]);
                        mma16816(acc[mt], u0 & 0x00f000f0u, u1 & 0x00f000f0u, u0s & 0x00f000f0u,
                                 u1s & 0x00f000f0u, bq[2 * mm + 1][0], bq[2 * mm + 1][1]);
                    }
                }
            }
        } else {
            // word m (4 bytes) of this lane's D / 16 bytes: channels (D / 4) c +
            // 16m + {0..15} (channel 16m + 4b + j in crumb j of byte b); K-step
            // 4m + k pairs channels (k, k+8), (k+4, k+12)
            constexpr int NWD = D / 64;                 // words per lane
            constexpr int WPC = NWD < 2 ? NWD : 2;      // words per chunk
#pragma unroll
            for (int ch = 0; ch < NWD / WPC; ++ch) {
                uint32_t bq[4 * WPC][2];
#pragma unroll
                for (int mm = 0; mm < WPC; ++mm) {
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int cb = (D / 4) * c + 16 * (WPC * ch + mm) + 4 * i;
                        float4 s4;
                        if constexpr (HS) s4 = key_scales4_h(S + GE::kKS, cb);
                        else s4 = *reinterpret_cast<const float4*>(KS + padc(cb));
                        const float4 q4 = *reinterpret_cast<const float4*>(qrow + padc(cb));
                        const float2 lo2 = upk(mul2(mul2(pk(q4.x, q4.y), pk(s4.x, s4.y)), fB2));
                        const float2 hi2 = upk(mul2(mul2(pk(q4.z, q4.w), pk(s4.z, s4.w)), fB2h));
                        v[4 * i] = lo2.x;
                        v[4 * i + 1] = lo2.y;
                        v[4 * i + 2] = hi2.x;
                        v[4 * i + 3] = hi2.y;
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        bq[4 * mm + k][0] = split_pair(v[k], v[k + 8], lo_part);
                        bq[4 * mm + k][1] = split_pair(v[k + 4], v[k + 12], lo_part);
                    }
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int r0 = mt * 16 + g, r1 = r0 + 8;
                    uint32_t w0v[WPC], w1v[WPC];
                    const uint8_t* p0 = KC + r0 * ROWB + (D / 16) * c + 8 * ch;
                    const uint8_t* p1 = KC + r1 * ROWB + (D / 16) * c + 8 * ch;
                    load_words<WPC>(p0, w0v);
                    load_words<WPC>(p1, w1v);
#pragma unroll
                    for (int mm = 0; mm < WPC; ++mm) {
                        const uint32_t u0 = w0v[mm], u1 = w1v[mm], u0s = u0 >> 8, u1s = u1 >> 8;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t mk = 0x00030003u << (2 * k);
                            mma16816(acc[mt], u0 & mk, u1 & mk, u0s & mk, u1s & mk, bq[4 * mm + k][0],
                                     bq[4 * mm + k][1]);
                        }
                    }
                }
            }
        }
        float sc[4];  // tokens g, g+8, g+16, g+24 for head c
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const int t0 = mt * 16 + g;
            const float s0 = fmaf(acc[mt][0] + acc[mt][1], fC, qz_c);
            const float s1 = fmaf(acc[mt][2] + acc[mt][3], fC, qz_c);
            sc[2 * mt] = t0 < nvalid ? s0 : -INFINITY;
            sc[2 * mt + 1] = t0 + 8 < nvalid ? s1 : -INFINITY;
        }

        // ---- online softmax (head c; lanes with equal c share it) ----
        float tmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        const float m_new = fmaxf(m_run, tmax);
        const float corr = exp2f(m_run - m_new);
        float p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = exp2f(sc[i] - m_new);
        l_run = fmaf(l_run, corr, (p[0] + p[1]) + (p[2] + p[3]));
        m_run = m_new;
        if (__any_sync(0xffffffffu, corr != 1.f)) {  // the running max moved (x * 1 == x: skip)
            const f32x2 c2 = pk(corr, corr);
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                const float2 lo = upk(mul2(pk(o[i][0], o[i][1]), c2)), hi = upk(mul2(pk(o[i][2], o[i][3]), c2));
                o[i][0] = lo.x;
                o[i][1] = lo.y;
                o[i][2] = hi.x;
                o[i][3] = hi.y;
            }
#pragma unroll
            for (int j = 0; j < NE; ++j) pzl[j] *= corr;
        }
        // p of tokens g, g+8, g+16, g+24 (head c) -> pbuf; p.vzero partials
        pbuf[(g) * 4 + c] = p[0];
        pbuf[(g + 8) * 4 + c] = p[1];
        pbuf[(g + 16) * 4 + c] = p[2];
        pbuf[(g + 24) * 4 + c] = p[3];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = g + 8 * i;
            uint32_t zw[NE / 2];  // the NE zeros of token t, two per word
            load_words<NE / 2>(reinterpret_cast<const uint8_t*>(VZ + t * NE), zw);
#pragma unroll
            for (int j2 = 0; j2 < NE / 2; ++j2) {
                const float2 zz = __half22float2(u32_as_h2(zw[j2]));
                pzl[2 * j2] = fmaf(p[i], zz.x, pzl[2 * j2]);
                pzl[2 * j2 + 1] = fmaf(p[i], zz.y, pzl[2 * j2 + 1]);
            }
        }
        __syncwarp();

        // ---- PV operand B: p_t s_tj of head hh, tokens of this lane's k slots ----
        // value group j's operand for K-step ks: bp(j, ks) = {split(p_ta s_ta,j,
        // p_ta+1 s_ta+1,j), split(p_tb s_tb,j, p_tb+1 s_tb+1,j)}
        float pp[2][4];  // [ks] p of tokens ta, ta+1, tb, tb+1 (head hh)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int ta = 16 * ks + 2 * c, tb = ta + 8;
            pp[ks][0] = pbuf[ta * 4 + hh];
            pp[ks][1] = pbuf[(ta + 1) * 4 + hh];
            pp[ks][2] = pbuf[tb * 4 + hh];
            pp[ks][3] = pbuf[(tb + 1) * 4 + hh];
        }
        // D <= 128: all NE groups' operands up front (the scales of a token are
        // one 8- or 16-byte load); D = 256: each group's operand right before
        // its MMAs
        constexpr int NBP = D <= 128 ? NE : 1;
        uint32_t bp[NBP][2][2];  // [group j][K-step][b0/b1]
        auto build_bp = [&](int j, uint32_t (&dst)[2][2]) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int ta = 16 * ks + 2 * c, tb = ta + 8;
                if constexpr (HS) {
                    const __half* VH = reinterpret_cast<const __half*>(VS);
                    dst[ks][0] = split_pair(pp[ks][0] * __half2float(VH[ta * NE + j]),
                                            pp[ks][1] * __half2float(VH[(ta + 1) * NE + j]), lo_part);
                    dst[ks][1] = split_pair(pp[ks][2] * __half2float(VH[tb * NE + j]),
                                            pp[ks][3] * __half2float(VH[(tb + 1) * NE + j]), lo_part);
                } else {
                    dst[ks][0] = split_pair(pp[ks][0] * VS[ta * NE + j], pp[ks][1] * VS[(ta + 1) * NE + j], lo_part);
                    dst[ks][1] = split_pair(pp[ks][2] * VS[tb * NE + j], pp[ks][3] * VS[(tb + 1) * NE + j], lo_part);
                }
            }
        };
        if (D <= 128) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int ta = 16 * ks + 2 * c, tb = ta + 8;
                float xa0[NE], xa1[NE], xb0[NE], xb1[NE];
                // p of one token times its NE group scales: pairs (s_t0, s_t1), ... of one load
                auto prodN = [](float pt, const float* v, float (&x)[NE]) {
                    const f32x2 p2 = pk(pt, pt);
                    uint32_t vw[NE];
                    load_words<NE>(reinterpret_cast<const uint8_t*>(v), vw);
#pragma unroll
                    for (int e = 0; e < NE; e += 2) {
                        const float2 r = upk(mul2(p2, pk(__uint_as_float(vw[e]), __uint_as_float(vw[e + 1]))));
                        x[e] = r.x;
                        x[e + 1] = r.y;
                    }
                };
                if constexpr (HS) {
                    auto prodH = [&](float pt, int t, float (&x)[NE]) {
                        const f32x2 p2 = pk(pt, pt);
                        float v[NE];
                        value_scales_h<NE>(S + GE::kVS, t, v);
#pragma unroll
                        for (int e = 0; e < NE; e += 2) {
                            const float2 r = upk(mul2(p2, pk(v[e], v[e + 1])));
                            x[e] = r.x;
                            x[e + 1] = r.y;
                        }
                    };
                    prodH(pp[ks][0], ta, xa0);
                    prodH(pp[ks][1], ta + 1, xa1);
                    prodH(pp[ks][2], tb, xb0);
                    prodH(pp[ks][3], tb + 1, xb1);
                } else {
                    prodN(pp[ks][0], VS + ta * NE, xa0);
                    prodN(pp[ks][1], VS + (ta + 1) * NE, xa1);
                    prodN(pp[ks][2], VS + tb * NE, xb0);
                    prodN(pp[ks][3], VS + (tb + 1) * NE, xb1);
                }
#pragma unroll
                for (int j = 0; j < NBP; ++j) {
                    bp[j][ks][0] = split_pair(xa0[j], xa1[j], lo_part);
                    bp[j][ks][1] = split_pair(xb0[j], xb1[j], lo_part);
                }
            }
        }

        // ---- P.V on the tensor cores ----
        const uint8_t* VC = S + GE::kVC;
        if (BITS == 4) {
            // o[2j + u]: rows g -> channel 32j + 4g + u, g+8 -> 32j + 4g + 2 + u
            constexpr int CPR = D / 32;  // 16-byte chunks (32 channels) per 4-bit row
#pragma unroll
            for (int j = 0; j < NE; ++j) {
                if (D > 128) build_bp(j, bp[0]);
                const uint32_t(&bj)[2][2] = bp[D <= 128 ? j : 0];
                const int row = 8 * (lane >> 3) + (lane & 7);  // token block lane>>3, row lane&7
                uint32_t W[4];
                ldsm_x4_t(W, VC + row * (D / 2) + 16 * swz<CPR>(row, j));
                uint32_t xl[2][4], xh[2][4];  // [u][token block] -> (row g, row g+8) halves
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // bytes of W: token 2c (channels 4g, 4g+1 | 4g+2, 4g+3), token 2c+1 (same)
                    const uint32_t Ws = W[q] >> 8;
                    xl[0][q] = W[q] & 0x000f000fu;  // channel 4g, units 2^-24
                    xh[0][q] = Ws & 0x000f000fu;    // channel 4g+2
                    xl[1][q] = W[q] & 0x00f000f0u;  // channel 4g+1, units 2^-20
                    xh[1][q] = Ws & 0x00f000f0u;    // channel 4g+3
                }
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma16816(o[2 * j + u], xl[u][2 * ks], xh[u][2 * ks], xl[u][2 * ks + 1], xh[u][2 * ks + 1],
                                 bj[ks][0], bj[ks][1]);
            }
        } else {
            // A 16-byte chunk of a 2-bit row holds value groups 2hc and 2hc + 1
            // (4 halves of 8 crumbs each). The transposed ldmatrix gives lane g
            // half g of the chunk, so lanes g < 4 hold group 2hc and lanes g >= 4
            // group 2hc + 1; one shuffle hands every lane half (g & 3) of each
            // group. MMA m of group grp then takes crumb 2m + (g >> 2) of the
            // low byte (row g) and of the high byte (row g + 8), so all 16 rows
            // share the group's B operand:
            // o[4hc + 2grp + m]: row g -> channel 64hc + 32grp + 8(g & 3) + 2m + (g >> 2),
            // row g + 8 -> that channel + 4, in units of 4^(2m + (g >> 2)) 2^-24
            constexpr int CPR = D / 64;  // 16-byte chunks (64 channels) per 2-bit row
            const int gh = g >> 2;
#pragma unroll
            for (int hc = 0; hc < CPR; ++hc) {
                uint32_t bA[2][2], bB[2][2];
                if (D > 128) {
                    build_bp(2 * hc, bA);
                    build_bp(2 * hc + 1, bB);
                }
                const uint32_t(&b0)[2][2] = D <= 128 ? bp[(2 * hc) % NBP] : bA;
                const uint32_t(&b1)[2][2] = D <= 128 ? bp[(2 * hc + 1) % NBP] : bB;
                const int row = 8 * (lane >> 3) + (lane & 7);
                uint32_t W[4];
                ldsm_x4_t(W, VC + row * (D / 4) + 16 * swz<CPR>(row, hc));
                uint32_t X[2][4], Xs[2][4];  // [group][token block]: half (g & 3), its high byte shifted down
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    X[0][q] = __shfl_sync(0xffffffffu, W[q], lane & 15);  // lanes g < 4 hold group 2hc
                    X[1][q] = __shfl_sync(0xffffffffu, W[q], lane | 16);  // lanes g >= 4 hold group 2hc + 1
                    Xs[0][q] = X[0][q] >> 8;
                    Xs[1][q] = X[1][q] >> 8;
                }
#pragma unroll
                for (int grp = 0; grp < 2; ++grp)
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const uint32_t mk = 0x00030003u << (2 * (2 * m + gh));
                        const uint32_t(&bg)[2][2] = grp ? b1 : b0;
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks)
                            mma16816(o[4 * hc + 2 * grp + m], X[grp][2 * ks] & mk, Xs[grp][2 * ks] & mk,
                                     X[grp][2 * ks + 1] & mk, Xs[grp][2 * ks + 1] & mk, bg[ks][0], bg[ks][1]);
                    }
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
    __syncwarp();

    // ---------------------------- residual tiles ----------------------------
    // kResTok fp16 K and V rows per tile. Their P.V is accumulated in fp32 per
    // 16-channel block and added into o (store-tile channel layout, o's units).
    for (int rt = r_begin; rt < w1; ++rt) {
        const int rtile = rt - a.n_store_tiles;
        const int nvalid = min(kResTok, a.n_res - rtile * kResTok);
        fetch_res_tile<D>(a, bh, rtile, nvalid, st0, st0 + kStage, lane);
        cp_async_commit();
        cp_async_wait<0>();
        __syncwarp();
        const uint8_t* KR = st0;
        const uint8_t* VR = st0 + kStage;
        float sc[4];
        {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const int q = lane >> 3, r = lane & 7;
            const int row = (q & 1) * 8 + r;
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                // B: q 2^Er of this lane's head (hi or lo), channels 16s + {2c, 2c+1 | 2c+8, 2c+9}
                const float2 qa = *reinterpret_cast<const float2*>(qrow + padc(16 * s + 2 * c));
                const float2 qb = *reinterpret_cast<const float2*>(qrow + padc(16 * s + 8 + 2 * c));
                const uint32_t b0 = split_pair(qa.x * fBr, qa.y * fBr, lo_part);
                const uint32_t b1 = split_pair(qb.x * fBr, qb.y * fBr, lo_part);
                const int chunk = 2 * s + (q >> 1);
                uint32_t A[4];
                ldsm_x4(A, KR + row * (2 * D) + ((chunk ^ (row & 7)) << 4));
                mma16816(acc, A[0], A[1], A[2], A[3], b0, b1);
            }
            sc[0] = g < nvalid ? (acc[0] + acc[1]) * fCr : -INFINITY;
            sc[1] = g + 8 < nvalid ? (acc[2] + acc[3]) * fCr : -INFINITY;
            sc[2] = sc[3] = -INFINITY;
        }
        float tmax = fmaxf(sc[0], sc[1]);
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        const float m_new = fmaxf(m_run, tmax);
        const float corr = exp2f(m_run - m_new);
        const float p0 = exp2f(sc[0] - m_new), p1 = exp2f(sc[1] - m_new);
        l_run = fmaf(l_run, corr, p0 + p1);
        m_run = m_new;
        if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
            for (int i = 0; i < D / 16; ++i)
#pragma unroll
                for (int k = 0; k < 4; ++k) o[i][k] *= corr;
#pragma unroll
            for (int j = 0; j < NE; ++j) pzl[j] *= corr;
        }
        pbuf[g * 4 + c] = p0;
        pbuf[(g + 8) * 4 + c] = p1;
        __syncwarp();
        // B: p of head hh (hi or lo), tokens {2c, 2c+1 | 2c+8, 2c+9}
        const uint32_t bp0 = split_pair(pbuf[(2 * c) * 4 + hh], pbuf[(2 * c + 1) * 4 + hh], lo_part);
        const uint32_t bp1 = split_pair(pbuf[(2 * c + 8) * 4 + hh], pbuf[(2 * c + 9) * 4 + hh], lo_part);
        if (BITS == 4) {
            // o[2j + u]: rows g -> channel 32j + 4g + u, g+8 -> 32j + 4g + 2 + u
#pragma unroll
            for (int j = 0; j < NE; ++j) {
                uint2 rv[4];  // tokens 2c, 2c+1, 2c+8, 2c+9: channels 32j + 4g .. 32j + 4g + 3
#pragma unroll
                for (int ti = 0; ti < 4; ++ti) {
                    const int t = 2 * c + (ti & 1) + 8 * (ti >> 1);
                    rv[ti] = *reinterpret_cast<const uint2*>(VR + t * (2 * D) + (((4 * j + (g >> 1)) ^ (t & 7)) << 4) +
                                                             (g & 1) * 8);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t sel = u ? 0x7632u : 0x5410u;  // half u of each word
                    float tmp[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(tmp, __byte_perm(rv[0].x, rv[1].x, sel), __byte_perm(rv[0].y, rv[1].y, sel),
                             __byte_perm(rv[2].x, rv[3].x, sel), __byte_perm(rv[2].y, rv[3].y, sel), bp0, bp1);
#pragma unroll
                    for (int k = 0; k < 4; ++k) o[2 * j + u][k] = fmaf(tmp[k], kOUnit4[u], o[2 * j + u][k]);
                }
            }
        } else {
            // the store tiles' layout: o[4hc + 2grp + m]: row g -> channel 64hc + 32grp + 8(g & 3) + p,
            // row g + 8 -> + 4, with p = 2m + (g >> 2), in units of 4^p 2^-24
            const int gh = g >> 2;
            const uint32_t sel = gh ? 0x7632u : 0x5410u;  // half p & 1 = g >> 2 of each word
#pragma unroll
            for (int hc = 0; hc < D / 64; ++hc)
#pragma unroll
                for (int grp = 0; grp < 2; ++grp) {
                    uint32_t rv[4][4];  // tokens 2c, 2c+1, 2c+8, 2c+9: channels 64hc + 32grp + 8(g & 3) .. + 7
                    const int chunk = 8 * hc + 4 * grp + (g & 3);
#pragma unroll
                    for (int ti = 0; ti < 4; ++ti) {
                        const int t = 2 * c + (ti & 1) + 8 * (ti >> 1);
                        const uint4 v4 = *reinterpret_cast<const uint4*>(VR + t * (2 * D) + ((chunk ^ (t & 7)) << 4));
                        rv[ti][0] = v4.x;
                        rv[ti][1] = v4.y;
                        rv[ti][2] = v4.z;
                        rv[ti][3] = v4.w;
                    }
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const int wa = m, wb = 2 + m;  // words of halves p and p + 4 (p = 2m + (g >> 2))
                        float tmp[4] = {0.f, 0.f, 0.f, 0.f};
                        mma16816(tmp, __byte_perm(rv[0][wa], rv[1][wa], sel), __byte_perm(rv[0][wb], rv[1][wb], sel),
                                 __byte_perm(rv[2][wa], rv[3][wa], sel), __byte_perm(rv[2][wb], rv[3][wb], sel), bp0,
                                 bp1);
                        const float unit = pow2i(2 * (2 * m + gh) - 24);
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[4 * hc + 2 * grp + m][e] = fmaf(tmp[e], unit, o[4 * hc + 2 * grp + m][e]);
                    }
                }
        }
        __syncwarp();
    }

    // ---------------------------- merge the warps ----------------------------
    // Each warp rescales its own accumulators by 2^(m_w - M) (M: the CTA's
    // largest running max of the head) before they meet in shared memory, so
    // the cross-warp combine is a plain sum.
    __syncthreads();  // every warp is done with its stages (they now take its share of the output)
    float* Ow = reinterpret_cast<float*>(st0);  // [4 heads][D] of this warp
    float* ml = misc + 16;                       // [warp][head][2]: m, then l * 2^(m - M)
    float* Mh = misc + 8;                        // [head]: M
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {  // l and sum_t p_t z_tj of head c: the lanes of equal c hold disjoint tokens
        l_run += __shfl_xor_sync(0xffffffffu, l_run, x);
#pragma unroll
        for (int j = 0; j < NE; ++j) pzl[j] += __shfl_xor_sync(0xffffffffu, pzl[j], x);
    }
    if (g == 0) ml[(warp * 4 + c) * 2] = m_run;
    __syncthreads();
    {
        float Mc = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) Mc = fmaxf(Mc, ml[(w * 4 + c) * 2]);
        const float f = m_run == -INFINITY ? 0.f : exp2f(m_run - Mc);  // a warp without tiles adds nothing
        // o holds sum p s c in units of kOUnit4 / kOUnit2; the z term adds per value group
        if (BITS == 4) {
#pragma unroll
            for (int j = 0; j < NE; ++j)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float sc = f / kOUnit4[u], zf = pzl[j] * f;
                    Ow[c * D + 32 * j + 4 * g + u] = fmaf(o[2 * j + u][0] + o[2 * j + u][1], sc, zf);
                    Ow[c * D + 32 * j + 4 * g + 2 + u] = fmaf(o[2 * j + u][2] + o[2 * j + u][3], sc, zf);
                }
        } else {
            const int gh = g >> 2;
#pragma unroll
            for (int hc = 0; hc < D / 64; ++hc)
#pragma unroll
                for (int grp = 0; grp < 2; ++grp) {
                    const float zf = pzl[2 * hc + grp] * f;
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const int p = 2 * m + gh;  // crumb position: units 4^p 2^-24
                        const float sc = f * pow2i(24 - 2 * p);
                        const int ch = 64 * hc + 32 * grp + 8 * (g & 3) + p;
                        const float(&oo)[4] = o[4 * hc + 2 * grp + m];
                        Ow[c * D + ch] = fmaf(oo[0] + oo[1], sc, zf);
                        Ow[c * D + ch + 4] = fmaf(oo[2] + oo[3], sc, zf);
                    }
                }
        }
        if (g == 0) {
            ml[(warp * 4 + c) * 2 + 1] = l_run * f;
            if (warp == 0) Mh[c] = Mc;
        }
    }
    pdl_trigger();
    __syncthreads();
    int h0, nh;  // recomputed here rather than held through the tile loop
    cta_heads<GQ>(a, h0, nh);
    for (int i4 = tid; i4 < nh * (D / 4); i4 += kThreads) {
        const int h = i4 / (D / 4), d = 4 * (i4 % (D / 4));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float4 v = *reinterpret_cast<const float4*>(
                reinterpret_cast<const float*>(smem + w * GE::kWarpSmem) + h * D + d);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
            L += ml[(w * 4 + h) * 2 + 1];
        }
        const float M = Mh[h];
        const long long bq = (long long)b * a.Hq + h0 + h;
        if (a.n_split == 1) {
            const float r = 1.0f / L;
            *reinterpret_cast<float4*>(a.out + bq * D + d) = make_float4(acc.x * r, acc.y * r, acc.z * r, acc.w * r);
        } else if (CL) {  // the partial stays in this CTA's shared memory (the q area is free now)
            *reinterpret_cast<float4*>(q_s + h * D + d) = acc;
            if (d == 0) {
                misc[100 + 2 * h] = M;
                misc[101 + 2 * h] = L;
            }
        } else {
            __stcg(reinterpret_cast<float4*>(a.part_o + (bq * a.n_split + split) * D + d), acc);
            if (d == 0) __stcg(reinterpret_cast<float2*>(a.part_ml + (bq * a.n_split + split) * 2), make_float2(M, L));
        }
    }
    if (a.n_split == 1) return;
    if (CL) {
        // Every CTA of the cluster holds one partial; CTA r merges outputs
        // r * kThreads + tid, ... of the head group, reading all partials
        // through distributed shared memory.
        cluster_sync();
        const uint32_t rank = cluster_ctarank();
        const int n = a.n_split;
        for (int idx = (int)rank * kThreads + tid; idx < nh * D; idx += n * kThreads) {
            const int h = idx / D, dd = idx % D;
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
                if (k < n && mk[k] != -INFINITY) {  // -inf: a CTA without tiles
                    const float wk = exp2f(mk[k] - M);
                    L = fmaf(ld_cluster(misc + 101 + 2 * h, k), wk, L);
                    acc = fmaf(ld_cluster(q_s + h * D + dd, k), wk, acc);
                }
            }
            a.out[((long long)b * a.Hq + h0 + h) * D + dd] = acc / L;
        }
        cluster_sync();  // no CTA leaves while another still reads its shared memory
        return;
    }
    // one ticket counter per (batch, KV head, sub-group)
    if (take_last_ticket(a, b * (int)gridDim.y + (int)blockIdx.y, reinterpret_cast<int*>(misc + 96)))
        merge_splits<kWarps, D>(a, (long long)b * a.Hq + h0, nh, warp, lane);
}

template <int BITS, int GQ, int NW, bool CL, int D, bool HS>
cudaError_t configure_mma() {
    static cudaError_t status = cudaErrorNotReady;  // benign race: every caller sets the same values
    if (status == cudaErrorNotReady) {
        cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<BITS, GQ, NW, CL, D, HS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<NW, D>::kSmemBytes);
        if (e == cudaSuccess && CL)
            e = cudaFuncSetAttribute(decode_mma_kernel<BITS, GQ, NW, CL, D, HS>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        status = e;
    }
    return status;
}

// Resident CTAs of this kernel on the device: without clusters (n = 1) or in
// clusters of n CTAs (0 if such clusters cannot be resident). Computed once
// per device and n with the occupancy calculator.
template <int BITS, int GQ, int NW, int D, bool HS>
int resident_ctas(int n, cudaStream_t stream) {
    constexpr int kDevs = 16;
    static int cache[kDevs][kMaxClusterSplits + 1];  // 0 unknown, -1 none, else CTAs + 1
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs || n < 1 || n > kMaxClusterSplits) {
        cudaGetLastError();
        return 0;
    }
    if (cache[dev][n] == 0) {
        int ctas = 0;
        if (n == 1) {
            int per_sm = 0, sms = 0;
            if (configure_mma<BITS, GQ, NW, false, D, HS>() == cudaSuccess &&
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_mma_kernel<BITS, GQ, NW, false, D, HS>,
                                                              32 * NW, Layout<NW, D>::kSmemBytes) == cudaSuccess &&
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
                ctas = per_sm * sms;
        } else if (configure_mma<BITS, GQ, NW, true, D, HS>() == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(n, 1, 1);
            cfg.blockDim = dim3(32 * NW);
            cfg.dynamicSmemBytes = Layout<NW, D>::kSmemBytes;
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = n;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, decode_mma_kernel<BITS, GQ, NW, true, D, HS>, &cfg) ==
                cudaSuccess)
                ctas = clusters * n;
        }
        cudaGetLastError();
        cache[dev][n] = ctas > 0 ? ctas + 1 : -1;
    }
    return cache[dev][n] > 0 ? cache[dev][n] - 1 : 0;
}

// Merge the splits inside clusters when they can be resident and either the
// whole grid fits in one wave of clusters (the latency case) or clusters keep
// at least 95 % of the resident CTAs (otherwise a cluster size that packs the
// GPU's processor clusters badly costs more than the merge saves). A grid of
// fewer CTAs than SMs merges through the workspace: spread one CTA per SM it
// has every SM's share of HBM bandwidth, while its clusters would pack two
// CTAs on an SM (13-split B=1 decodes took 8.2 us in clusters against 7.1).
template <int BITS, int GQ, int NW, int D, bool HS>
bool use_cluster(const DecodeArgs& a, cudaStream_t stream) {
    const int n = a.n_split;
    if (n < 2 || n > kMaxClusterSplits) return false;
    const long long ctas = (long long)n * a.Hkv * a.q_sub * a.B;
    if (ctas < sm_count()) return false;
    const long long with = resident_ctas<BITS, GQ, NW, D, HS>(n, stream);
    if (with <= 0) return false;
    return ctas <= with || 20 * with >= 19LL * resident_ctas<BITS, GQ, NW, D, HS>(1, stream);
}

template <int BITS, int GQ, int NW, int D, bool HS>
cudaError_t launch_mma_typed(const DecodeArgs& a, cudaStream_t stream) {
    const dim3 grid(a.n_split, a.Hkv * a.q_sub, a.B);
    constexpr int kSmem = Layout<NW, D>::kSmemBytes;
    if (use_cluster<BITS, GQ, NW, D, HS>(a, stream)) {
        cudaError_t e = configure_mma<BITS, GQ, NW, true, D, HS>();
        if (e != cudaSuccess) return e;
        return launch_pdl_cluster(decode_mma_kernel<BITS, GQ, NW, true, D, HS>, grid, 32 * NW, kSmem, stream,
                                  a.n_split, a);
    }
    cudaError_t e = configure_mma<BITS, GQ, NW, false, D, HS>();
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_mma_kernel<BITS, GQ, NW, false, D, HS>, grid, 32 * NW, kSmem, stream, a);
}

template <int BITS, int GQ, int D, bool HS>
cudaError_t launch_mma_warps(const DecodeArgs& a, cudaStream_t stream) {
    if constexpr (D == 128) {
        if (a.warps_per_cta == 2) return launch_mma_typed<BITS, GQ, 2, D, HS>(a, stream);
    }
    return a.warps_per_cta == 8 ? launch_mma_typed<BITS, GQ, 8, D, HS>(a, stream)
                                : launch_mma_typed<BITS, GQ, 4, D, HS>(a, stream);
}

// The one-warp-per-tile decode of head dim D, with fp32 (HS false) or fp16
// (HS true) scales: groups of 1, 2 or 4 heads run their own width; other
// groups run in sub-groups of 4 heads (a.q_sub of them per KV head, the last
// possibly partial).
template <int D, bool HS>
cudaError_t launch_decode_mma_impl(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    cudaError_t e = cudaErrorInvalidValue;
    if (gq < 1 || (gq > 2 && (gq + 3) / 4 != a.q_sub) || (gq <= 2 && a.q_sub != 1)) return e;
    if (bits == 4) {
        if (gq == 1) e = launch_mma_warps<4, 1, D, HS>(a, stream);
        else if (gq == 2) e = launch_mma_warps<4, 2, D, HS>(a, stream);
        else if (gq == 4) e = launch_mma_warps<4, 4, D, HS>(a, stream);
        else e = launch_mma_warps<4, kSubGroupGQ, D, HS>(a, stream);
    } else {
        if (gq == 1) e = launch_mma_warps<2, 1, D, HS>(a, stream);
        else if (gq == 2) e = launch_mma_warps<2, 2, D, HS>(a, stream);
        else if (gq == 4) e = launch_mma_warps<2, 4, D, HS>(a, stream);
        else e = launch_mma_warps<2, kSubGroupGQ, D, HS>(a, stream);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

}  // namespace kivi

// flush.cu -- KIVI flush: quantize + bit-pack keys (per-channel groups along
// the token axis) and values (per-token groups along head_dim).
//
// Method: VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly
// 0% Faster" -- "What we're actually optimizing" (zero = min, scale =
// (max - min)/(2^bits - 1), q = round((x - zero)/scale), clipped),
// "The layout problem that shapes everything" (keys group along the strided
// token axis, values along the contiguous head_dim), "Three ways to be off by
// one bit" (half-to-even rounding; a ragged group's edge padding leaves min
// and max unchanged).
//
// GB300 design (not the pages' one-thread-per-group Metal kernels):
//  * keys: lanes are laid across D with 16-byte loads (8 channels each), so a
//    warp load covers whole 128-byte lines of consecutive token rows and the
//    strided per-channel group reads as contiguous rows, with no transpose.
//    Four threads share one (group, 8-channel) column, 8 tokens each, and
//    combine min/max with two shuffles; every thread then quantizes its own
//    8 tokens from registers (x is read from HBM exactly once).
//  * values: 4 lanes (4 x 8 channels) form one 32-channel group; min/max is a
//    2-step __shfl_xor butterfly on packed half2 min/max.
//  * min/max run on packed fp16 (exact), the quantizer in fp32 with explicit
//    _rn intrinsics; the quotient is an IEEE division inside a guard band.
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

namespace {

constexpr int kThreads = 128;

// ---------------------------------------------------------------------------
// keys
// ---------------------------------------------------------------------------

// One warp covers (head, group, 64 channels): lane = part * 8 + octet, part
// in [0, 4) owns tokens [8*part, 8*part + 8) of the group, octet owns 8
// channels. Two warps cover the 128 channels of a group.
template <int BITS>
__device__ __forceinline__ void flush_keys_warp(const FlushArgs& a, long long warp_id) {
    constexpr int TPT = 8;  // tokens per thread
    const int lane = threadIdx.x & 31;
    const int octet = (int)(warp_id & 1) * 8 + (lane & 7);
    const int part = lane >> 3;
    const long long grp = warp_id >> 1;
    const int ng = (a.n_flush + kG - 1) / kG;
    if (grp >= (long long)a.BH * ng) return;  // warp-uniform
    const int bh = (int)(grp / ng);
    const int g = (int)(grp - (long long)bh * ng);
    const int t0 = g * kG + part * TPT;

    const uint4* xrow = reinterpret_cast<const uint4*>(a.x) +
                        ((long long)bh * a.x_bh_stride + t0) * (kD / 8) + octet;
    uint4 v[TPT];
    const __half2 pinf = __half2half2(__ushort_as_half(0x7c00));
    const __half2 ninf = __half2half2(__ushort_as_half(0xfc00));
    __half2 mn[4] = {pinf, pinf, pinf, pinf};
    __half2 mx[4] = {ninf, ninf, ninf, ninf};
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
        if (t0 + i < a.n_flush) v[i] = __ldg(xrow + (long long)i * (kD / 8));
        else v[i] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
        if (t0 + i < a.n_flush) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mn[k] = __hmin2(mn[k], u32_as_h2(w[k]));
                mx[k] = __hmax2(mx[k], u32_as_h2(w[k]));
            }
        }
    }
    // combine the 4 parts of this column (lanes octet, octet+8, +16, +24)
#pragma unroll
    for (int o = 8; o < 32; o <<= 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            mn[k] = __hmin2(mn[k], u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mn[k]), o)));
            mx[k] = __hmax2(mx[k], u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mx[k]), o)));
        }
    }
    float zf[8], sf[8], rf[8];
    const float L = (float)Levels<BITS>::value;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 lo = __half22float2(mn[k]);
        const float2 hi = __half22float2(mx[k]);
        zf[2 * k] = __fadd_rn(lo.x, 0.0f);      // -0 -> +0 for min and max
        zf[2 * k + 1] = __fadd_rn(lo.y, 0.0f);
        sf[2 * k] = __fdiv_rn(__fsub_rn(__fadd_rn(hi.x, 0.0f), zf[2 * k]), L);
        sf[2 * k + 1] = __fdiv_rn(__fsub_rn(__fadd_rn(hi.y, 0.0f), zf[2 * k + 1]), L);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) rf[k] = sf[k] == 0.0f ? 0.0f : __frcp_rn(sf[k]);

    if (part == 0) {
        const long long m = ((long long)bh * (a.s_cap / kG) + a.s_off / kG + g) * kD + octet * 8;
        float4* sp = reinterpret_cast<float4*>(a.scale + m);
        sp[0] = make_float4(sf[0], sf[1], sf[2], sf[3]);
        sp[1] = make_float4(sf[4], sf[5], sf[6], sf[7]);
        uint4 zp;
        zp.x = h2_as_u32(__floats2half2_rn(zf[0], zf[1]));
        zp.y = h2_as_u32(__floats2half2_rn(zf[2], zf[3]));
        zp.z = h2_as_u32(__floats2half2_rn(zf[4], zf[5]));
        zp.w = h2_as_u32(__floats2half2_rn(zf[6], zf[7]));
        *reinterpret_cast<uint4*>(a.zero + m) = zp;
    }

    constexpr int ROWB = kD * BITS / 8;
    uint8_t* crow = a.codes + ((long long)bh * a.s_cap + a.s_off + t0) * ROWB + octet * BITS;
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
        if (t0 + i < a.n_flush) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t packed = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 xf = __half22float2(u32_as_h2(w[k]));
                const uint32_t c0 = quant_code<BITS>(__fsub_rn(xf.x, zf[2 * k]), sf[2 * k], rf[2 * k]);
                const uint32_t c1 = quant_code<BITS>(__fsub_rn(xf.y, zf[2 * k + 1]), sf[2 * k + 1], rf[2 * k + 1]);
                packed |= c0 << (2 * k * BITS);
                packed |= c1 << ((2 * k + 1) * BITS);
            }
            if (BITS == 4) *reinterpret_cast<uint32_t*>(crow + (long long)i * ROWB) = packed;
            else *reinterpret_cast<uint16_t*>(crow + (long long)i * ROWB) = (uint16_t)packed;
        }
    }
}

// ---------------------------------------------------------------------------
// values
// ---------------------------------------------------------------------------

// One warp covers 8 consecutive (head, token) rows: lane = sub * 16 + octet;
// iteration i handles row 2*i + sub, so each warp load reads 512 contiguous
// bytes. Lanes 4j..4j+3 of a half-warp form value group j.
template <int BITS>
__device__ __forceinline__ void flush_values_warp(const FlushArgs& a, long long warp_id) {
    constexpr int RPT = 4;  // rows per thread
    const int lane = threadIdx.x & 31;
    const int octet = lane & 15;
    const int sub = lane >> 4;
    const long long rows = (long long)a.BH * a.n_flush;
    const long long r0 = warp_id * (2 * RPT);
    if (r0 >= rows) return;  // warp-uniform
    constexpr int ROWB = kD * BITS / 8;
    const float L = (float)Levels<BITS>::value;

    uint4 v[RPT];
    int bh[RPT], t[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const long long r = r0 + 2 * i + sub;
        bh[i] = (int)(r / a.n_flush);
        t[i] = (int)(r - (long long)bh[i] * a.n_flush);
        if (r < rows)
            v[i] = __ldg(reinterpret_cast<const uint4*>(a.x) +
                         ((long long)bh[i] * a.x_bh_stride + t[i]) * (kD / 8) + octet);
        else
            v[i] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const bool ok = r0 + 2 * i + sub < rows;
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        // packed (min, max) of this lane's 8 channels
        __half2 m2 = __hmin2(__hmin2(u32_as_h2(w[0]), u32_as_h2(w[1])), __hmin2(u32_as_h2(w[2]), u32_as_h2(w[3])));
        __half2 x2 = __hmax2(__hmax2(u32_as_h2(w[0]), u32_as_h2(w[1])), __hmax2(u32_as_h2(w[2]), u32_as_h2(w[3])));
        __half2 mm = __halves2half2(__hmin(__low2half(m2), __high2half(m2)),
                                    __hmax(__low2half(x2), __high2half(x2)));
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            const __half2 other = u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mm), o));
            mm = __halves2half2(__hmin(__low2half(mm), __low2half(other)),
                                __hmax(__high2half(mm), __high2half(other)));
        }
        const float z = __fadd_rn(__low2float(mm), 0.0f);  // -0 -> +0 for min and max
        const float s = __fdiv_rn(__fsub_rn(__fadd_rn(__high2float(mm), 0.0f), z), L);
        const float rc = s == 0.0f ? 0.0f : __frcp_rn(s);
        if (!ok) continue;
        const long long row = (long long)bh[i] * a.s_cap + a.s_off + t[i];
        uint32_t packed = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 xf = __half22float2(u32_as_h2(w[k]));
            packed |= quant_code<BITS>(__fsub_rn(xf.x, z), s, rc) << (2 * k * BITS);
            packed |= quant_code<BITS>(__fsub_rn(xf.y, z), s, rc) << ((2 * k + 1) * BITS);
        }
        uint8_t* c = a.codes + row * ROWB + octet * BITS;
        if (BITS == 4) *reinterpret_cast<uint32_t*>(c) = packed;
        else *reinterpret_cast<uint16_t*>(c) = (uint16_t)packed;
        if ((octet & 3) == 0) {
            const long long m = row * (kD / kG) + (octet >> 2);
            a.scale[m] = s;
            a.zero[m] = __float2half_rn(z);
        }
    }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) flush_keys_kernel(FlushArgs a) {
    flush_keys_warp<BITS>(a, ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) flush_values_kernel(FlushArgs a) {
    flush_values_warp<BITS>(a, ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5);
}

// Keys and values of the same tokens in one launch: the first key_blocks
// blocks run the key flush, the rest the value flush.
template <int BITS>
__global__ void __launch_bounds__(kThreads) flush_kv_kernel(FlushArgs k, FlushArgs v, int key_blocks) {
    if ((int)blockIdx.x < key_blocks)
        flush_keys_warp<BITS>(k, ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5);
    else
        flush_values_warp<BITS>(v, ((long long)(blockIdx.x - key_blocks) * kThreads + threadIdx.x) >> 5);
}

long long key_blocks(const FlushArgs& a) {
    const long long warps = (long long)a.BH * ((a.n_flush + kG - 1) / kG) * 2;
    return (warps * 32 + kThreads - 1) / kThreads;
}

long long value_blocks(const FlushArgs& a) {
    const long long warps = ((long long)a.BH * a.n_flush + 7) / 8;
    return (warps * 32 + kThreads - 1) / kThreads;
}

}  // namespace

cudaError_t launch_flush(int axis, const FlushArgs& a, int bits, cudaStream_t stream) {
    const long long blocks = axis == 0 ? key_blocks(a) : value_blocks(a);
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (axis == 0) {
        if (bits == 4) flush_keys_kernel<4><<<(unsigned)blocks, kThreads, 0, stream>>>(a);
        else flush_keys_kernel<2><<<(unsigned)blocks, kThreads, 0, stream>>>(a);
    } else {
        if (bits == 4) flush_values_kernel<4><<<(unsigned)blocks, kThreads, 0, stream>>>(a);
        else flush_values_kernel<2><<<(unsigned)blocks, kThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_flush_kv(const FlushArgs& k, const FlushArgs& v, int bits, cudaStream_t stream) {
    const long long kb = key_blocks(k), vb = value_blocks(v);
    if (kb + vb <= 0) return cudaSuccess;
    if (kb + vb > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (bits == 4) flush_kv_kernel<4><<<(unsigned)(kb + vb), kThreads, 0, stream>>>(k, v, (int)kb);
    else flush_kv_kernel<2><<<(unsigned)(kb + vb), kThreads, 0, stream>>>(k, v, (int)kb);
    return cudaGetLastError();
}

}  // namespace kivi

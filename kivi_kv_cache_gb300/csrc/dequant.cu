// dequant.cu -- KIVI dequantize: packed codes + per-group scale/zero -> fp16.
//
// recon = fp16_rn(RN(RN(q * scale) + zero)): VeloxQuant-MLX blog, "A 5.65x
// Metal Kernel That Made My LLM Exactly 0% Faster", "What we're actually
// optimizing" (recon = q*scale + zero) and "Three ways to be off by one bit"
// #1 (multiply, then a separate add: two roundings, never an FMA).
//
// Memory pattern: each thread owns 8 channels (one 16-byte fp16 store per
// token row); code words are 4 bytes (4-bit) or 2 bytes (2-bit) per thread
// per row, so a warp's loads and stores cover whole contiguous row segments.
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

namespace {

constexpr int kThreads = 128;

template <int BITS>
__device__ __forceinline__ uint4 recon8(uint32_t w, const float* s, const float* z) {
    constexpr uint32_t M = Levels<BITS>::value;
    float r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) r[k] = recon((w >> (k * BITS)) & M, s[k], z[k]);
    uint4 o;
    o.x = h2_as_u32(__floats2half2_rn(r[0], r[1]));
    o.y = h2_as_u32(__floats2half2_rn(r[2], r[3]));
    o.z = h2_as_u32(__floats2half2_rn(r[4], r[5]));
    o.w = h2_as_u32(__floats2half2_rn(r[6], r[7]));
    return o;
}

template <int BITS>
__device__ __forceinline__ uint32_t load_word(const uint8_t* p) {
    if (BITS == 4) return __ldg(reinterpret_cast<const uint32_t*>(p));
    return __ldg(reinterpret_cast<const uint16_t*>(p));
}

// keys: one warp per (head, key group, 64-channel half); lane = part*8 + octet,
// part owns 8 tokens of the group. Scale and zero are per (group, channel).
template <int BITS>
__global__ void __launch_bounds__(kThreads) dequant_keys_kernel(DequantArgs a) {
    constexpr int ROWB = kD * BITS / 8;
    const long long warp_id = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int octet = (int)(warp_id & 1) * 8 + (lane & 7);
    const int part = lane >> 3;
    const long long grp = warp_id >> 1;
    const int ng = (a.S + kG - 1) / kG;
    if (grp >= (long long)a.BH * ng) return;
    const int bh = (int)(grp / ng);
    const int g = (int)(grp - (long long)bh * ng);
    const int t0 = g * kG + part * 8;

    const long long m = ((long long)bh * (a.s_cap / kG) + g) * kD + octet * 8;
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(a.scale + m));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(a.scale + m) + 1);
    const uint4 zw = __ldg(reinterpret_cast<const uint4*>(a.zero + m));
    const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    float z[8];
    {
        const uint32_t zz[4] = {zw.x, zw.y, zw.z, zw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(u32_as_h2(zz[k]));
            z[2 * k] = f.x;
            z[2 * k + 1] = f.y;
        }
    }
    const uint8_t* crow = a.codes + ((long long)bh * a.s_cap + t0) * ROWB + octet * BITS;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (t0 + i < a.S) ? load_word<BITS>(crow + (long long)i * ROWB) : 0u;
    uint4* orow = reinterpret_cast<uint4*>(a.out) + ((long long)bh * a.S + t0) * (kD / 8) + octet;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (t0 + i < a.S) orow[(long long)i * (kD / 8)] = recon8<BITS>(w[i], s, z);
}

// values: one warp per 8 consecutive (head, token) rows; lane = sub*16 + octet,
// iteration i handles row 2*i + sub. Scale and zero are per (token, group).
template <int BITS>
__global__ void __launch_bounds__(kThreads) dequant_values_kernel(DequantArgs a) {
    constexpr int ROWB = kD * BITS / 8;
    constexpr int RPT = 4;
    const long long warp_id = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int octet = lane & 15;
    const int sub = lane >> 4;
    const long long rows = (long long)a.BH * a.S;
    const long long r0 = warp_id * (2 * RPT);
    if (r0 >= rows) return;
    uint32_t w[RPT];
    float s[RPT], z[RPT];
    long long orow[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const long long r = r0 + 2 * i + sub;
        const int bh = (int)(r / a.S);
        const int t = (int)(r - (long long)bh * a.S);
        const long long row = (long long)bh * a.s_cap + t;
        orow[i] = r;
        if (r < rows) {
            w[i] = load_word<BITS>(a.codes + row * ROWB + octet * BITS);
            s[i] = __ldg(a.scale + row * (kD / kG) + (octet >> 2));
            z[i] = __half2float(a.zero[row * (kD / kG) + (octet >> 2)]);
        } else {
            w[i] = 0u;
            s[i] = 0.f;
            z[i] = 0.f;
        }
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        if (orow[i] < rows) {
            const float sv[8] = {s[i], s[i], s[i], s[i], s[i], s[i], s[i], s[i]};
            const float zv[8] = {z[i], z[i], z[i], z[i], z[i], z[i], z[i], z[i]};
            reinterpret_cast<uint4*>(a.out)[orow[i] * (kD / 8) + octet] = recon8<BITS>(w[i], sv, zv);
        }
    }
}

}  // namespace

cudaError_t launch_dequant(int axis, const DequantArgs& a, int bits, cudaStream_t stream) {
    long long warps;
    if (axis == 0) warps = (long long)a.BH * ((a.S + kG - 1) / kG) * 2;
    else warps = ((long long)a.BH * a.S + 7) / 8;
    const long long blocks = (warps * 32 + kThreads - 1) / kThreads;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (axis == 0) {
        if (bits == 4) dequant_keys_kernel<4><<<(unsigned)blocks, kThreads, 0, stream>>>(a);
        else dequant_keys_kernel<2><<<(unsigned)blocks, kThreads, 0, stream>>>(a);
    } else {
        if (bits == 4) dequant_values_kernel<4><<<(unsigned)blocks, kThreads, 0, stream>>>(a);
        else dequant_values_kernel<2><<<(unsigned)blocks, kThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kivi

// dequant.cu -- KIVI dequantize: packed codes + per-group scale/zero -> fp16.
//
// recon = fp16_rn(RN(RN(q * scale) + zero)): VeloxQuant-MLX blog, "A 5.65x
// Metal Kernel That Made My LLM Exactly 0% Faster", "What we're actually
// optimizing" (recon = q*scale + zero) and "Three ways to be off by one bit"
// #1 (multiply, then a separate add: two roundings, never one fused op for
// the reconstruction).
//
// Arithmetic: a byte permute turns each code q into the fp32 pattern of
// 2^23 + q. Then fma(2^23 + q, s, -2^23 * s) is the exact value q * s rounded
// once, i.e. RN(q * s) (-2^23 * s is exact: a power-of-two scaling). The add
// of zero is a separate round-to-nearest add, as the method requires. Both
// run as packed fp32x2 operations.
//
// Memory pattern: each thread owns 8 channels (one 16-byte fp16 store per
// token row); a warp's loads and stores cover whole contiguous row segments.
// Keys and values can run in one launch (blocks [0, kbx) of each grid row
// dequantize keys, the rest values); blockIdx.y is the head.
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

namespace {

constexpr int kThreads = 128;

// fp32 patterns 2^23 + q of the 8 codes of one row segment (element i at bit
// offset i*BITS): qm[k] for element k.
template <int BITS>
__device__ __forceinline__ void codes_to_magic(uint32_t w, uint32_t (&qm)[8]) {
    const uint32_t C = 0x4B000000u;  // byte 3 = 0x4B, bytes 0..2 = 0
    if (BITS == 4) {
        const uint32_t e = w & 0x0f0f0f0fu;         // elements 0,2,4,6
        const uint32_t o = (w >> 4) & 0x0f0f0f0fu;  // elements 1,3,5,7
        qm[0] = __byte_perm(e, C, 0x7440);
        qm[2] = __byte_perm(e, C, 0x7441);
        qm[4] = __byte_perm(e, C, 0x7442);
        qm[6] = __byte_perm(e, C, 0x7443);
        qm[1] = __byte_perm(o, C, 0x7440);
        qm[3] = __byte_perm(o, C, 0x7441);
        qm[5] = __byte_perm(o, C, 0x7442);
        qm[7] = __byte_perm(o, C, 0x7443);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t p = (w >> (2 * k)) & 0x0303u;  // elements k, k+4
            qm[k] = __byte_perm(p, C, 0x7440);
            qm[k + 4] = __byte_perm(p, C, 0x7441);
        }
    }
}

// 8 reconstructions -> 8 fp16 (one 16-byte vector). s2/ns2/z2: per element
// scale, -2^23*scale and zero, as fp32x2 pairs.
template <int BITS>
__device__ __forceinline__ uint4 recon8(uint32_t w, const f32x2 (&s2)[4], const f32x2 (&ns2)[4],
                                        const f32x2 (&z2)[4]) {
    uint32_t qm[8];
    codes_to_magic<BITS>(w, qm);
    uint32_t h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const f32x2 q2 = pk(__uint_as_float(qm[2 * k]), __uint_as_float(qm[2 * k + 1]));
        const float2 r = upk(add2(fma2(q2, s2[k], ns2[k]), z2[k]));
        h[k] = h2_as_u32(__floats2half2_rn(r.x, r.y));
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

template <int BITS>
__device__ __forceinline__ uint32_t load_word(const uint8_t* p) {
    if (BITS == 4) return __ldg(reinterpret_cast<const uint32_t*>(p));
    return __ldg(reinterpret_cast<const uint16_t*>(p));
}

// keys: one warp per (head, 32-token block, 64-channel slice); lane =
// part*8 + oc, part owns 8 tokens of the block. Scale and zero are per (key
// group of G tokens, channel): the block's group is block * 32 / G.
template <int BITS, int G, int D, bool HS>
__device__ __forceinline__ void dequant_keys_warp(const DequantArgs& a, int warp_id, int bh) {
    constexpr int ROWB = D * BITS / 8;
    constexpr int NSL = D / 64;  // 64-channel slices per row
    const int lane = threadIdx.x & 31;
    const unsigned wu = warp_id;
    const int octet = (wu % NSL) * 8 + (lane & 7);
    const int part = lane >> 3;
    const int tb = wu / NSL;
    if (tb >= (a.S + 31) / 32) return;
    const int g = tb * 32 / G;
    const int t0 = tb * 32 + part * 8;

    const uint8_t* crow = a.codes + ((long long)bh * a.s_cap + t0) * ROWB + octet * BITS;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (t0 + i < a.S) ? load_word<BITS>(crow + i * ROWB) : 0u;
    const long long m = ((long long)bh * (a.s_cap / G) + g) * D + octet * 8;
    float s[8];
    if (HS) {  // 8 fp16 scales
        const uint4 hw = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(a.scale) + m));
        const uint32_t hv[4] = {hw.x, hw.y, hw.z, hw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(u32_as_h2(hv[k]));
            s[2 * k] = f.x;
            s[2 * k + 1] = f.y;
        }
    } else {
        const float4 sa = __ldg(reinterpret_cast<const float4*>(a.scale + m));
        const float4 sb = __ldg(reinterpret_cast<const float4*>(a.scale + m) + 1);
        s[0] = sa.x, s[1] = sa.y, s[2] = sa.z, s[3] = sa.w, s[4] = sb.x, s[5] = sb.y, s[6] = sb.z, s[7] = sb.w;
    }
    const uint4 zw = __ldg(reinterpret_cast<const uint4*>(a.zero + m));
    pdl_trigger();
    const uint32_t zz[4] = {zw.x, zw.y, zw.z, zw.w};
    f32x2 s2[4], ns2[4], z2[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        s2[k] = pk(s[2 * k], s[2 * k + 1]);
        ns2[k] = pk(-kMagic * s[2 * k], -kMagic * s[2 * k + 1]);
        const float2 f = __half22float2(u32_as_h2(zz[k]));
        z2[k] = pk(f.x, f.y);
    }
    uint4* orow = reinterpret_cast<uint4*>(a.out) + ((long long)bh * a.S + t0) * (D / 8) + octet;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (t0 + i < a.S) orow[i * (D / 8)] = recon8<BITS>(w[i], s2, ns2, z2);
}

// values: one warp per NR * RPT consecutive tokens of one head (NR = 32 / (D /
// 8) rows per pass); lane = sub * (D / 8) + octet, iteration i handles token
// NR * i + sub. Scale and zero are per (token, G-channel group).
template <int BITS, int G, int D, bool HS>
__device__ __forceinline__ void dequant_values_warp(const DequantArgs& a, int warp_id, int bh) {
    constexpr int ROWB = D * BITS / 8;
    constexpr int RPT = 4;
    constexpr int OPR = D / 8;    // octets per row: 8, 16 or 32
    constexpr int NR = 32 / OPR;  // rows per pass: 4, 2 or 1
    const int lane = threadIdx.x & 31;
    const int octet = lane % OPR;
    const int sub = lane / OPR;
    const int tw = warp_id * (NR * RPT);
    if (tw >= a.S) return;
    const long long row0 = (long long)bh * a.s_cap + tw + sub;
    uint32_t w[RPT];
    float s[RPT], z[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const long long row = row0 + NR * i;
        if (tw + NR * i + sub < a.S) {
            w[i] = load_word<BITS>(a.codes + row * ROWB + octet * BITS);
            const long long mi = row * (D / G) + octet / (G / 8);
            s[i] = HS ? __half2float(reinterpret_cast<const __half*>(a.scale)[mi]) : __ldg(a.scale + mi);
            z[i] = __half2float(a.zero[row * (D / G) + octet / (G / 8)]);
        } else {
            w[i] = 0u;
            s[i] = 0.f;
            z[i] = 0.f;
        }
    }
    pdl_trigger();
    uint4* orow = reinterpret_cast<uint4*>(a.out) + ((long long)bh * a.S + tw + sub) * (D / 8) + octet;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        if (tw + NR * i + sub < a.S) {
            const f32x2 s1 = pk(s[i], s[i]), n1 = pk(-kMagic * s[i], -kMagic * s[i]), z1 = pk(z[i], z[i]);
            const f32x2 s2[4] = {s1, s1, s1, s1}, ns2[4] = {n1, n1, n1, n1}, z2[4] = {z1, z1, z1, z1};
            orow[NR * i * (D / 8)] = recon8<BITS>(w[i], s2, ns2, z2);
        }
    }
}

// blocks of 4 warps: keys take one warp per (32-token block, 64-channel
// slice); values one warp per 4 passes of 32 / (D / 8) rows
int key_blocks_x(int S, int D) { return ((S + 31) / 32 * (D / 64) + 3) / 4; }
int value_blocks_x(int S, int D) {
    const int tokens_per_block = 4 * 4 * (256 / D);
    return (S + tokens_per_block - 1) / tokens_per_block;
}

template <int BITS, int G, int D, bool HS>
__global__ void __launch_bounds__(kThreads) dequant_keys_kernel(DequantArgs a) {
    pdl_wait();
    dequant_keys_warp<BITS, G, D, HS>(a, blockIdx.x * 4 + (threadIdx.x >> 5), blockIdx.y);
}

template <int BITS, int G, int D, bool HS>
__global__ void __launch_bounds__(kThreads) dequant_values_kernel(DequantArgs a) {
    pdl_wait();
    dequant_values_warp<BITS, G, D, HS>(a, blockIdx.x * 4 + (threadIdx.x >> 5), blockIdx.y);
}

template <int BITS, int G, int D, bool HS>
__global__ void __launch_bounds__(kThreads) dequant_kv_kernel(DequantArgs k, DequantArgs v, int kbx) {
    pdl_wait();
    if ((int)blockIdx.x < kbx)
        dequant_keys_warp<BITS, G, D, HS>(k, blockIdx.x * 4 + (threadIdx.x >> 5), blockIdx.y);
    else
        dequant_values_warp<BITS, G, D, HS>(v, (blockIdx.x - kbx) * 4 + (threadIdx.x >> 5), blockIdx.y);
}


DequantArgs head_slice(const DequantArgs& a, int h0, int nh, int bits, int axis) {
    DequantArgs s = a;
    s.BH = nh;
    s.codes += (long long)h0 * a.s_cap * (a.D * bits / 8);
    const long long meta = axis == 0 ? (long long)(a.s_cap / a.G) * a.D : (long long)a.s_cap * (a.D / a.G);
    s.scale = a.scale_f16 ? reinterpret_cast<const float*>(reinterpret_cast<const __half*>(a.scale) + h0 * meta)
                          : a.scale + h0 * meta;
    s.zero += h0 * meta;
    s.out += (long long)h0 * a.S * a.D;
    return s;
}

template <int BITS, int G, int D, bool HS>
cudaError_t launch_dequant_typed(int axis, const DequantArgs& a, cudaStream_t stream) {
    const int bx = axis == 0 ? key_blocks_x(a.S, D) : value_blocks_x(a.S, D);
    for (int h0 = 0; h0 < a.BH; h0 += 65535) {
        const int nh = a.BH - h0 < 65535 ? a.BH - h0 : 65535;
        const DequantArgs s = head_slice(a, h0, nh, BITS, axis);
        const dim3 grid(bx, nh);
        const cudaError_t e = axis == 0 ? launch_pdl(dequant_keys_kernel<BITS, G, D, HS>, grid, kThreads, 0, stream, s)
                                        : launch_pdl(dequant_values_kernel<BITS, G, D, HS>, grid, kThreads, 0, stream, s);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

template <int BITS, int G, int D, bool HS>
cudaError_t launch_dequant_kv_typed(const DequantArgs& k, const DequantArgs& v, cudaStream_t stream) {
    const int kbx = key_blocks_x(k.S, D), vbx = value_blocks_x(v.S, D);
    for (int h0 = 0; h0 < k.BH; h0 += 65535) {
        const int nh = k.BH - h0 < 65535 ? k.BH - h0 : 65535;
        const DequantArgs ks = head_slice(k, h0, nh, BITS, 0), vs = head_slice(v, h0, nh, BITS, 1);
        const dim3 grid(kbx + vbx, nh);
        const cudaError_t e = launch_pdl(dequant_kv_kernel<BITS, G, D, HS>, grid, kThreads, 0, stream, ks, vs, kbx);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

// (G, D) pairs: G in {32, 64, 128}, D in {64, 128, 256}, G <= D. One
// launch function per (BITS, G, D); F<BITS, G, D>::run forwards to it.
template <template <int, int, int> class F, typename... A>
cudaError_t by_shape(int bits, int G, int D, A&&... args) {
    switch (bits * 1000000 + G * 1000 + D) {
        case 4032064: return F<4, 32, 64>::run(args...);
        case 4032128: return F<4, 32, 128>::run(args...);
        case 4032256: return F<4, 32, 256>::run(args...);
        case 4064064: return F<4, 64, 64>::run(args...);
        case 4064128: return F<4, 64, 128>::run(args...);
        case 4064256: return F<4, 64, 256>::run(args...);
        case 4128128: return F<4, 128, 128>::run(args...);
        case 4128256: return F<4, 128, 256>::run(args...);
        case 2032064: return F<2, 32, 64>::run(args...);
        case 2032128: return F<2, 32, 128>::run(args...);
        case 2032256: return F<2, 32, 256>::run(args...);
        case 2064064: return F<2, 64, 64>::run(args...);
        case 2064128: return F<2, 64, 128>::run(args...);
        case 2064256: return F<2, 64, 256>::run(args...);
        case 2128128: return F<2, 128, 128>::run(args...);
        case 2128256: return F<2, 128, 256>::run(args...);
        default: return cudaErrorInvalidValue;
    }
}

template <int BITS, int G, int D>
struct DequantOne {
    static cudaError_t run(int axis, const DequantArgs& a, cudaStream_t stream) {
        return a.scale_f16 ? launch_dequant_typed<BITS, G, D, true>(axis, a, stream)
                           : launch_dequant_typed<BITS, G, D, false>(axis, a, stream);
    }
};

template <int BITS, int G, int D>
struct DequantKV {
    static cudaError_t run(const DequantArgs& k, const DequantArgs& v, cudaStream_t stream) {
        return k.scale_f16 ? launch_dequant_kv_typed<BITS, G, D, true>(k, v, stream)
                           : launch_dequant_kv_typed<BITS, G, D, false>(k, v, stream);
    }
};

}  // namespace

cudaError_t launch_dequant(int axis, const DequantArgs& a, int bits, cudaStream_t stream) {
    if (a.S <= 0 || a.BH <= 0) return cudaSuccess;
    return by_shape<DequantOne>(bits, a.G, a.D, axis, a, stream);
}

cudaError_t launch_dequant_kv(const DequantArgs& k, const DequantArgs& v, int bits, cudaStream_t stream) {
    if (k.S <= 0 || k.BH <= 0) return cudaSuccess;
    return by_shape<DequantKV>(bits, k.G, k.D, k, v, stream);
}

}  // namespace kivi

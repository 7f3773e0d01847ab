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
//    combine min/max with two shuffles; each of the four computes the scale
//    of two channels and shares it; every thread then quantizes its own 8
//    tokens from registers (x is read from HBM exactly once).
//  * values: 4 lanes (4 x 8 channels) form one 32-channel group; min/max is a
//    2-step __shfl_xor butterfly on packed (min, max) halves; each of the 4
//    lanes computes the scale of one of its 4 rows and shares it.
//  * min/max run on packed fp16 (exact). The quantizer runs on packed fp32x2
//    IEEE operations. The quotient: y = RN(a * RN(1/s)) lies within 2^-18 of
//    RN(a/s) for quotients below 16, so rint(y) == rint(RN(a/s)) whenever y is
//    farther than 2^-14 from every half-integer; one check per 8 elements
//    sends the rare near-tie element to an exact IEEE division (out of line).
//    RN(y + 2^23) rounds half to even and leaves the code in the low byte;
//    byte permutes pack 8 codes per 32-bit word.
//  * 2-D grids (y = head) keep all index arithmetic in 32 bits.
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

namespace {

constexpr int kThreads = 128;
constexpr float kTieBand = 0.5f - 1.0f / 16384.0f;

// rint(RN(a / s)) by IEEE division, as an fp32 bit pattern 0x4B0000qq. Only
// called for quotients within the guard band of a half-integer.
__device__ __noinline__ uint32_t exact_code_bits(float a, float s) {
    return __float_as_uint(__fadd_rn(__fdiv_rn(a, s), kMagic));
}

// Pack the codes held in byte 0 of tb[0..7] (element i of the row at bit
// offset i*BITS, low bits first). For finite inputs every code is at most
// 2^BITS - 1 (y <= L * (1 + 3 * 2^-24)), so bytes add without carries; for
// NaN/Inf inputs the codes are unspecified but the store stays in bounds.
template <int BITS>
__device__ __forceinline__ uint32_t pack8(const uint32_t (&tb)[8]) {
    if (BITS == 4) {
        const uint32_t e = __byte_perm(__byte_perm(tb[0], tb[2], 0x0040), __byte_perm(tb[4], tb[6], 0x0040), 0x5410);
        const uint32_t o = __byte_perm(__byte_perm(tb[1], tb[3], 0x0040), __byte_perm(tb[5], tb[7], 0x0040), 0x5410);
        return e + (o << 4);
    } else {
        const uint32_t p0 = __byte_perm(tb[0], tb[4], 0x0040);
        const uint32_t p1 = __byte_perm(tb[1], tb[5], 0x0040);
        const uint32_t p2 = __byte_perm(tb[2], tb[6], 0x0040);
        const uint32_t p3 = __byte_perm(tb[3], tb[7], 0x0040);
        return (p0 + (p1 << 2) + (p2 << 4) + (p3 << 6)) & 0xffffu;
    }
}

// Codes of 8 fp16 elements (one 16-byte vector) packed into BITS*8 bits.
// z2/r2: per-element zero and RN(1/scale) as fp32x2 pairs; s: scales.
template <int BITS>
__device__ __forceinline__ uint32_t quant8(const uint4 xv, const f32x2 (&z2)[4], const f32x2 (&r2)[4],
                                           const float (&s)[8]) {
    const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
    const f32x2 M2 = pk(kMagic, kMagic);
    f32x2 a[4], y[4], t[4];
    float fm = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 xf = __half22float2(u32_as_h2(w[k]));
        a[k] = sub2(pk(xf.x, xf.y), z2[k]);
        y[k] = mul2(a[k], r2[k]);
        t[k] = add2(y[k], M2);
        const float2 f = upk(sub2(y[k], sub2(t[k], M2)));
        fm = fmaxf(fm, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    uint32_t tb[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 tt = upk(t[k]);
        tb[2 * k] = __float_as_uint(tt.x);
        tb[2 * k + 1] = __float_as_uint(tt.y);
    }
    if (fm > kTieBand) {  // rare: a quotient within 2^-14 of a half-integer
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 aa = upk(a[k]), yy = upk(y[k]), tt = upk(t[k]);
            if (fabsf(__fsub_rn(yy.x, __fsub_rn(tt.x, kMagic))) > kTieBand)
                tb[2 * k] = exact_code_bits(aa.x, s[2 * k]);
            if (fabsf(__fsub_rn(yy.y, __fsub_rn(tt.y, kMagic))) > kTieBand)
                tb[2 * k + 1] = exact_code_bits(aa.y, s[2 * k + 1]);
        }
    }
    return pack8<BITS>(tb);
}

// -0 -> +0 (applied to min and max, so zero and scale carry no negative sign)
__device__ __forceinline__ float canon(float v) { return __fadd_rn(v, 0.0f); }

// ---------------------------------------------------------------------------
// keys
// ---------------------------------------------------------------------------

// One warp covers (head, group, 64 channels): lane = part * 8 + oc, part in
// [0, 4) owns tokens [8*part, 8*part + 8) of the group, oc owns 8 channels.
// Two warps cover the 128 channels of a group.
template <int BITS>
__device__ __forceinline__ void flush_keys_warp(const FlushArgs& a, int warp_id, int bh) {
    constexpr int TPT = 8;
    const int lane = threadIdx.x & 31;
    const int oc = lane & 7;
    const int part = lane >> 3;
    const int octet = (warp_id & 1) * 8 + oc;
    const int g = warp_id >> 1;
    const int ng = (a.n_flush + kG - 1) / kG;
    if (g >= ng) return;  // warp-uniform
    const int t0 = g * kG + part * TPT;

    const uint4* xrow = reinterpret_cast<const uint4*>(a.x) +
                        ((long long)bh * a.x_bh_stride + t0) * (kD / 8) + octet;
    uint4 v[TPT];
#pragma unroll
    for (int i = 0; i < TPT; ++i)
        v[i] = (t0 + i < a.n_flush) ? __ldg(xrow + i * (kD / 8)) : make_uint4(0, 0, 0, 0);
    pdl_trigger();

    const __half2 pinf = __half2half2(__ushort_as_half(0x7c00));
    const __half2 ninf = __half2half2(__ushort_as_half(0xfc00));
    __half2 mn[4] = {pinf, pinf, pinf, pinf};
    __half2 mx[4] = {ninf, ninf, ninf, ninf};
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
#pragma unroll
    for (int o = 8; o < 32; o <<= 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            mn[k] = __hmin2(mn[k], u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mn[k]), o)));
            mx[k] = __hmax2(mx[k], u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mx[k]), o)));
        }
    }
    // zero of all 8 channels; this part's 2 channels' scale and reciprocal
    float z[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 lo = __half22float2(mn[k]);
        z[2 * k] = canon(lo.x);
        z[2 * k + 1] = canon(lo.y);
    }
    const float L = (float)Levels<BITS>::value;
    float my_s[2], my_r[2];
    {
        __half2 hx = mx[0], hn = mn[0];  // channels 2*part, 2*part + 1 of this octet
#pragma unroll
        for (int k = 1; k < 4; ++k)
            if (part == k) {
                hx = mx[k];
                hn = mn[k];
            }
        const float2 hi = __half22float2(hx), lo = __half22float2(hn);
        my_s[0] = __fdiv_rn(__fsub_rn(canon(hi.x), canon(lo.x)), L);
        my_s[1] = __fdiv_rn(__fsub_rn(canon(hi.y), canon(lo.y)), L);
        my_r[0] = my_s[0] == 0.0f ? 0.0f : __frcp_rn(my_s[0]);
        my_r[1] = my_s[1] == 0.0f ? 0.0f : __frcp_rn(my_s[1]);
    }
    float s[8], r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int src = (k >> 1) * 8 + oc;
        s[k] = __shfl_sync(0xffffffffu, my_s[k & 1], src);
        r[k] = __shfl_sync(0xffffffffu, my_r[k & 1], src);
    }
    f32x2 z2[4], r2[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        z2[k] = pk(z[2 * k], z[2 * k + 1]);
        r2[k] = pk(r[2 * k], r[2 * k + 1]);
    }

    if (part == 0) {
        const long long m = ((long long)bh * (a.s_cap / kG) + a.s_off / kG + g) * kD + octet * 8;
        float4* sp = reinterpret_cast<float4*>(a.scale + m);
        sp[0] = make_float4(s[0], s[1], s[2], s[3]);
        sp[1] = make_float4(s[4], s[5], s[6], s[7]);
        uint4 zp;
        zp.x = h2_as_u32(__floats2half2_rn(z[0], z[1]));
        zp.y = h2_as_u32(__floats2half2_rn(z[2], z[3]));
        zp.z = h2_as_u32(__floats2half2_rn(z[4], z[5]));
        zp.w = h2_as_u32(__floats2half2_rn(z[6], z[7]));
        *reinterpret_cast<uint4*>(a.zero + m) = zp;
    }

    constexpr int ROWB = kD * BITS / 8;
    uint8_t* crow = a.codes + ((long long)bh * a.s_cap + a.s_off + t0) * ROWB + octet * BITS;
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
        if (t0 + i < a.n_flush) {
            const uint32_t packed = quant8<BITS>(v[i], z2, r2, s);
            if (BITS == 4) *reinterpret_cast<uint32_t*>(crow + i * ROWB) = packed;
            else *reinterpret_cast<uint16_t*>(crow + i * ROWB) = (uint16_t)packed;
        }
    }
}

// ---------------------------------------------------------------------------
// values
// ---------------------------------------------------------------------------

// One warp covers 8 consecutive tokens of one head: lane = sub * 16 + octet;
// iteration i handles token 2*i + sub, so each warp load reads 512 contiguous
// bytes. Lanes 4j..4j+3 of a half-warp form value group j.
template <int BITS>
__device__ __forceinline__ void flush_values_warp(const FlushArgs& a, int warp_id, int bh) {
    constexpr int RPT = 4;
    const int lane = threadIdx.x & 31;
    const int octet = lane & 15;
    const int sub = lane >> 4;
    const int tw = warp_id * (2 * RPT);  // first token of this warp
    if (tw >= a.n_flush) return;         // warp-uniform
    constexpr int ROWB = kD * BITS / 8;
    const float L = (float)Levels<BITS>::value;

    const uint4* xrow = reinterpret_cast<const uint4*>(a.x) + ((long long)bh * a.x_bh_stride + tw + sub) * (kD / 8) + octet;
    uint4 v[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i)
        v[i] = (tw + 2 * i + sub < a.n_flush) ? __ldg(xrow + 2 * i * (kD / 8)) : make_uint4(0, 0, 0, 0);
    pdl_trigger();

    float z[RPT], range[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        const __half2 m2 = __hmin2(__hmin2(u32_as_h2(w[0]), u32_as_h2(w[1])), __hmin2(u32_as_h2(w[2]), u32_as_h2(w[3])));
        const __half2 x2 = __hmax2(__hmax2(u32_as_h2(w[0]), u32_as_h2(w[1])), __hmax2(u32_as_h2(w[2]), u32_as_h2(w[3])));
        __half2 mm = __halves2half2(__hmin(__low2half(m2), __high2half(m2)), __hmax(__low2half(x2), __high2half(x2)));
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            const __half2 other = u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mm), o));
            mm = __halves2half2(__hmin(__low2half(mm), __low2half(other)), __hmax(__high2half(mm), __high2half(other)));
        }
        z[i] = canon(__low2float(mm));
        range[i] = __fsub_rn(canon(__high2float(mm)), z[i]);
    }
    // lane (octet & 3) == i computes row i's scale, then all 4 lanes share it
    const int mine = octet & 3;
    float rg = range[0];
#pragma unroll
    for (int i = 1; i < RPT; ++i)
        if (mine == i) rg = range[i];
    const float my_s = __fdiv_rn(rg, L);
    const float my_r = my_s == 0.0f ? 0.0f : __frcp_rn(my_s);

    uint8_t* cbase = a.codes + ((long long)bh * a.s_cap + a.s_off + tw + sub) * ROWB + octet * BITS;
    const long long mbase = ((long long)bh * a.s_cap + a.s_off + tw + sub) * (kD / kG) + (octet >> 2);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const float s = __shfl_sync(0xffffffffu, my_s, (lane & ~3) | i);
        const float rc = __shfl_sync(0xffffffffu, my_r, (lane & ~3) | i);
        if (tw + 2 * i + sub >= a.n_flush) continue;
        const f32x2 z2[4] = {pk(z[i], z[i]), pk(z[i], z[i]), pk(z[i], z[i]), pk(z[i], z[i])};
        const f32x2 r2[4] = {pk(rc, rc), pk(rc, rc), pk(rc, rc), pk(rc, rc)};
        const float sv[8] = {s, s, s, s, s, s, s, s};
        const uint32_t packed = quant8<BITS>(v[i], z2, r2, sv);
        uint8_t* c = cbase + 2 * i * ROWB;
        if (BITS == 4) *reinterpret_cast<uint32_t*>(c) = packed;
        else *reinterpret_cast<uint16_t*>(c) = (uint16_t)packed;
        if ((octet & 3) == 0) {
            a.scale[mbase + 2 * i * (kD / kG)] = s;
            a.zero[mbase + 2 * i * (kD / kG)] = __float2half_rn(z[i]);
        }
    }
}

int key_blocks_x(int n_flush) { return ((n_flush + kG - 1) / kG * 2 + 3) / 4; }   // 4 warps per block
int value_blocks_x(int n_flush) { return (n_flush + 31) / 32; }                    // 32 tokens per block

template <int BITS>
__global__ void __launch_bounds__(kThreads, 6) flush_keys_kernel(FlushArgs a) {
    pdl_wait();
    flush_keys_warp<BITS>(a, blockIdx.x * 4 + (threadIdx.x >> 5), blockIdx.y);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) flush_values_kernel(FlushArgs a) {
    pdl_wait();
    flush_values_warp<BITS>(a, blockIdx.x * 4 + (threadIdx.x >> 5), blockIdx.y);
}

// Keys and values of the same tokens in one launch: blocks [0, kbx) of each
// grid row (blockIdx.y = head) run the key flush, the rest the value flush.
template <int BITS>
__global__ void __launch_bounds__(kThreads, 6) flush_kv_kernel(FlushArgs k, FlushArgs v, int kbx) {
    pdl_wait();
    if ((int)blockIdx.x < kbx)
        flush_keys_warp<BITS>(k, blockIdx.x * 4 + (threadIdx.x >> 5), blockIdx.y);
    else
        flush_values_warp<BITS>(v, (blockIdx.x - kbx) * 4 + (threadIdx.x >> 5), blockIdx.y);
}

// Heads are split into launches of at most 65535 (the grid's y limit).
FlushArgs head_slice(const FlushArgs& a, int h0, int nh, int bits, int axis) {
    FlushArgs s = a;
    s.BH = nh;
    s.x += (long long)h0 * a.x_bh_stride * kD;
    s.codes += (long long)h0 * a.s_cap * (kD * bits / 8);
    const long long meta = axis == 0 ? (long long)(a.s_cap / kG) * kD : (long long)a.s_cap * (kD / kG);
    s.scale += h0 * meta;
    s.zero += h0 * meta;
    return s;
}

}  // namespace

cudaError_t launch_flush(int axis, const FlushArgs& a, int bits, cudaStream_t stream) {
    if (a.n_flush <= 0 || a.BH <= 0) return cudaSuccess;
    const int bx = axis == 0 ? key_blocks_x(a.n_flush) : value_blocks_x(a.n_flush);
    for (int h0 = 0; h0 < a.BH; h0 += 65535) {
        const int nh = a.BH - h0 < 65535 ? a.BH - h0 : 65535;
        const FlushArgs s = head_slice(a, h0, nh, bits, axis);
        const dim3 grid(bx, nh);
        cudaError_t e;
        if (axis == 0)
            e = bits == 4 ? launch_pdl(flush_keys_kernel<4>, grid, kThreads, 0, stream, s)
                          : launch_pdl(flush_keys_kernel<2>, grid, kThreads, 0, stream, s);
        else
            e = bits == 4 ? launch_pdl(flush_values_kernel<4>, grid, kThreads, 0, stream, s)
                          : launch_pdl(flush_values_kernel<2>, grid, kThreads, 0, stream, s);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_flush_kv(const FlushArgs& k, const FlushArgs& v, int bits, cudaStream_t stream) {
    if (k.n_flush <= 0 || k.BH <= 0) return cudaSuccess;
    const int kbx = key_blocks_x(k.n_flush), vbx = value_blocks_x(v.n_flush);
    for (int h0 = 0; h0 < k.BH; h0 += 65535) {
        const int nh = k.BH - h0 < 65535 ? k.BH - h0 : 65535;
        const FlushArgs ks = head_slice(k, h0, nh, bits, 0), vs = head_slice(v, h0, nh, bits, 1);
        const dim3 grid(kbx + vbx, nh);
        cudaError_t e = bits == 4 ? launch_pdl(flush_kv_kernel<4>, grid, kThreads, 0, stream, ks, vs, kbx)
                                  : launch_pdl(flush_kv_kernel<2>, grid, kThreads, 0, stream, ks, vs, kbx);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace kivi

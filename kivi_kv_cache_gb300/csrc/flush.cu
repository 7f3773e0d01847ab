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
//  * values: one lane owns whole 32-channel groups of a row (min/max, scale
//    and the 16-byte code word of a group in one lane, no shuffles); shared
//    memory chunks are swizzled by row so a warp's reads are conflict-free.
//  * min/max run on packed fp16 (exact). x - zero is one mixed-precision
//    subtraction (fp16 operand, fp32 result: no separate conversion). The
//    scale RN((max - min) / L) is one multiply and two fmas (division by the
//    constant L = 3 or 15 with one remainder correction; checked equal to
//    the IEEE quotient for every non-negative finite fp32). The quotient:
//    with r = 1/s to within 1 ulp (rcp.approx.f32), the exact product a * r
//    lies within 2^-18 of RN(a/s) for quotients below 16, so one fp32x2 fma
//    RN(a r + 2^23) rounds it half to even and leaves the code in the low
//    byte, and a second fma measures its distance from that integer; when
//    the distance is within 0.5 - 2^-14 the code equals rint(RN(a/s)). One
//    check per 8 elements sends the rare near-tie element to an exact IEEE
//    division (out of line). Byte permutes pack 8 codes per 32-bit word.
//  * work is cut into 4 KB items (a key group's G tokens x 2048 / G channels,
//    or 2048 / D value rows; at G = 128 a key item of 128 tokens x 32
//    channels, 64-byte row pieces, is split over a warp pair, 64 tokens per
//    warp); each warp walks the items with a grid stride, staging two at a
//    time in shared memory, so the copy of the next item overlaps the
//    quantization of the current one; the key loop takes two token rows per
//    trip. Long flushes at G = 32 stage an item from one lane with bulk
//    tensor copies (TMA: one 32 x 64 key box, or D / 64 value boxes of 64
//    channels in the 128-byte swizzle) that complete on the stage's
//    shared-memory barrier, at 6 CTAs per SM; everything else stages with
//    per-lane 16-byte cp.async at 4 (launch_items says which and why).
#include <cuda.h>  // CUtensorMap (the encoder is taken from the driver at run time)

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

// RN(x - z) for the two fp16 elements of w (x exact in fp32): one mixed-
// precision subtraction each, no separate fp16 -> fp32 conversion.
__device__ __forceinline__ f32x2 sub_h2(uint32_t w, f32x2 z) {
    const float2 zz = upk(z);
    float a, b;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "sub.rn.f32.f16 %0, l, %3;\n\tsub.rn.f32.f16 %1, h, %4;\n\t}"
        : "=f"(a), "=f"(b)
        : "r"(w), "f"(zz.x), "f"(zz.y));
    return pk(a, b);
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// With an fp16 scale a subnormal stored scale can leave a quotient past
// 2^BITS - 1 (up to about 1.5 (2^BITS - 1)): clip the codes, whose fp32
// patterns 2^23 + q order like q.
template <int BITS>
__device__ __forceinline__ void clip8(uint32_t (&tb)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) tb[i] = min(tb[i], 0x4B000000u + (uint32_t)Levels<BITS>::value);
}

// Codes of 8 fp16 elements (one 16-byte vector), each as the fp32 bit
// pattern of 2^23 + q in tb[i]. z2/r2: per-element zero and r = 1/scale to
// within 1 ulp, as fp32x2 pairs; s: scales. With a = RN(x - z), the exact
// product a * r lies within (a/s) 2^-23 + 2^-21 < 2^-18 of RN(a / s)
// (quotients below 16; below 2^-17 for the quotients below 32 that an fp16
// scale allows), so t = RN(a r + 2^23)
// (one fma) holds q = rint(RN(a / s)) whenever f = RN(a r - (t - 2^23)) is
// within 0.5 - 2^-14 of zero; the rare element outside that band takes an
// IEEE division (out of line). With fp16 scales (HS), clip (warp-uniform,
// set only where a subnormal scale can push a code past 2^BITS - 1) sends
// the 8 codes down the same rare branch to be clipped.
template <int BITS, bool HS>
__device__ __forceinline__ void quant8_codes(const uint4 xv, const f32x2 (&z2)[4], const f32x2 (&r2)[4],
                                             const float (&s)[8], uint32_t (&tb)[8], bool clip) {
    const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
    const f32x2 M2 = pk(kMagic, kMagic);
    f32x2 a[4];
    float d[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        a[k] = sub_h2(w[k], z2[k]);
        const f32x2 t = fma2(a[k], r2[k], M2);
        const float2 f = upk(fma2(a[k], r2[k], sub2(M2, t)));
        d[2 * k] = fabsf(f.x);
        d[2 * k + 1] = fabsf(f.y);
        const float2 tt = upk(t);
        tb[2 * k] = __float_as_uint(tt.x);
        tb[2 * k + 1] = __float_as_uint(tt.y);
    }
    const float fm = max3f(max3f(d[0], d[1], d[2]), max3f(d[3], d[4], d[5]), fmaxf(d[6], d[7]));
    if (fm > kTieBand || (HS && clip)) {  // rare: a quotient within about 2^-14 of a half-integer
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 aa = upk(a[k]);
            if (d[2 * k] > kTieBand) tb[2 * k] = exact_code_bits(aa.x, s[2 * k]);
            if (d[2 * k + 1] > kTieBand) tb[2 * k + 1] = exact_code_bits(aa.y, s[2 * k + 1]);
        }
        if (HS && clip) clip8<BITS>(tb);
    }
}

// Only a scale below the smallest normal fp16 (2^-14) can push a code past
// 2^BITS - 1 once rounded to fp16: a normal fp16 scale lies within a relative
// 2^-11 of the fp32 one, and every a is at most max - min, so a / s stays
// below L (1 + 2^-10) < L + 1/2. The decision is taken per warp (a vote over
// its active lanes); warps without such a scale never take the clip, and the
// others take it in the rare branch of quant8_codes (one copy of the loop).
__device__ __forceinline__ bool warp_has_subnormal_scale(bool lane_has) {
    return __any_sync(__activemask(), lane_has);
}
constexpr float kMinNormalF16 = 6.103515625e-05f;  // 2^-14

// The codes of quant8_codes packed into BITS*8 bits.
template <int BITS, bool HS>
__device__ __forceinline__ uint32_t quant8(const uint4 xv, const f32x2 (&z2)[4], const f32x2 (&r2)[4],
                                           const float (&s)[8], bool clip) {
    uint32_t tb[8];
    quant8_codes<BITS, HS>(xv, z2, r2, s, tb, clip);
    return pack8<BITS>(tb);
}

// Fake quantization of the same 8 elements: fp16(RN(RN(q * s) + z)), the
// dequantized value of each code (VeloxQuant-MLX blog, "A 5.65x Metal Kernel
// That Made My LLM Exactly 0% Faster", "What we're actually optimizing";
// multiply, then a separate add: "Three ways to be off by one bit" #1).
// With tb = bits of 2^23 + q, fma(2^23 + q, s, -2^23 s) is q * s rounded once.
template <int BITS, bool HS>
__device__ __forceinline__ uint4 fake8(const uint4 xv, const f32x2 (&z2)[4], const f32x2 (&r2)[4],
                                       const float (&s)[8], bool clip) {
    uint32_t tb[8];
    quant8_codes<BITS, HS>(xv, z2, r2, s, tb, clip);
    uint32_t h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const f32x2 q2 = pk(__uint_as_float(tb[2 * k]), __uint_as_float(tb[2 * k + 1]));
        const f32x2 s2 = pk(s[2 * k], s[2 * k + 1]);
        const f32x2 n2 = pk(-kMagic * s[2 * k], -kMagic * s[2 * k + 1]);
        const float2 r = upk(add2(fma2(q2, s2, n2), z2[k]));
        h[k] = h2_as_u32(__floats2half2_rn(r.x, r.y));
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

// The scale RN(x / L) for x = max - min >= 0 and L = 2^BITS - 1 (3 or 15):
// q = RN(x c) with c = RN(1 / L), the remainder x - q L (exact in one fma),
// then one fma correction q + RN(remainder) c (the division-by-a-constant
// step with an fma-computed remainder, as in Markstein's division
// algorithms). That this equals the IEEE quotient for L = 3 and 15 is not a
// general theorem: tests/test_guard_band.py checks it against IEEE division
// for every non-negative finite fp32 x.
template <int BITS>
__device__ __forceinline__ float div_levels(float x) {
    constexpr float L = (float)Levels<BITS>::value;
    constexpr float c = 1.0f / L;
    const float q = __fmul_rn(x, c);
    const float r = __fmaf_rn(-q, L, x);
    return __fmaf_rn(r, c, q);
}

// 1 / s within 1 ulp (rcp.approx.f32, s a positive normal fp32): the fast
// quotient only needs a r within a relative 2^-23 of a / s.
__device__ __forceinline__ float rcp_1ulp(float s) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
    return r;
}

// -0 -> +0 (applied to min and max, so zero and scale carry no negative sign)
__device__ __forceinline__ float canon(float v) { return __fadd_rn(v, 0.0f); }

// Scale stores: fp32, or fp16 (HS; the scale is already an fp16 value, so the
// conversion is exact) at element index m of the scale array.
template <bool HS>
__device__ __forceinline__ void store_scale(float* scale, long long m, float s) {
    if (HS) reinterpret_cast<__half*>(scale)[m] = __float2half_rn(s);
    else scale[m] = s;
}
template <bool HS>
__device__ __forceinline__ void store_scales8(float* scale, long long m, const float (&s)[8]) {
    if (HS) {
        uint4 h;
        h.x = h2_as_u32(__floats2half2_rn(s[0], s[1]));
        h.y = h2_as_u32(__floats2half2_rn(s[2], s[3]));
        h.z = h2_as_u32(__floats2half2_rn(s[4], s[5]));
        h.w = h2_as_u32(__floats2half2_rn(s[6], s[7]));
        *reinterpret_cast<uint4*>(reinterpret_cast<__half*>(scale) + m) = h;
    } else {
        float4* sp = reinterpret_cast<float4*>(scale + m);
        sp[0] = make_float4(s[0], s[1], s[2], s[3]);
        sp[1] = make_float4(s[4], s[5], s[6], s[7]);
    }
}

// ---------------------------------------------------------------------------
// work items, staged per warp through shared memory
// ---------------------------------------------------------------------------
//
// A key item is (head, key group, 64-channel half): 32 tokens x 128 bytes. A
// value item is (head, 16 consecutive tokens): 16 rows x 256 bytes. Both are
// 4 KB. Each warp walks the item list with a grid stride and keeps two items
// in flight (cp.async, double buffered), so copies of the next item overlap
// the quantization of the current one. Rows past n_flush are zero-filled and
// never read from global memory.

// Key items are a key group's G tokens x 2048 / G channels (4 KB) at G = 32
// and 64. At G = 128 a key item is the group's 128 tokens x 32 channels
// (64-byte row pieces) split over a warp pair: each warp stages and
// quantizes 64 of the tokens (4 KB) and the pair exchanges its column minima
// and maxima once through shared memory. (A whole 8 KB item per warp fits
// only 12 warps per SM; 128 tokens x 16 channels read 32-byte pieces.)
__host__ __device__ constexpr int key_item_channels(int G) { return G == 128 ? 32 : 4096 / (2 * G); }
__host__ __device__ constexpr int key_warp_tokens(int G) { return G == 128 ? 64 : G; }  // per warp

// A stage holds one warp's share of an item (4 KB). Each warp has two stages.
template <int G>
struct Stage {
    static constexpr int kBytes = 4096;
};
#ifndef KIVI_FLUSH_BLOCKS_PER_SM
#define KIVI_FLUSH_BLOCKS_PER_SM 4
#endif
#ifndef KIVI_FLUSH_TMA_BLOCKS_PER_SM
#define KIVI_FLUSH_TMA_BLOCKS_PER_SM 6
#endif
// resident CTAs per SM the grid is sized for (and the register bound): the
// bulk-copy kernel needs no per-lane copy addressing and fits 6 CTAs in 80
// registers without spills (measured: 6 faster than 5 and 4 on long
// flushes); the cp.async kernel runs 4
template <bool TMA>
constexpr int blocks_per_sm() {
    return TMA ? KIVI_FLUSH_TMA_BLOCKS_PER_SM : KIVI_FLUSH_BLOCKS_PER_SM;
}
// G = 128: per CTA, the warps' minima and maxima for the pair exchange, two
// slots (alternate items) of 32 words per warp
constexpr int kXchgBytes = 2 * (kThreads / 32) * 32 * 4;
#ifndef KIVI_FLUSH_KEY_UNROLL
#define KIVI_FLUSH_KEY_UNROLL 2
#endif
constexpr int kKeyUnroll = KIVI_FLUSH_KEY_UNROLL;  // key rows per loop trip (instruction footprint vs overlap)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool fill) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(fill ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
// barrier over `threads` threads (a multiple of 32) with named barrier ID (1..15)
template <int ID>
__device__ __forceinline__ void named_barrier(int threads) {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "r"(threads) : "memory");
}

// --- bulk tensor copies (TMA) with shared-memory barrier completion, for the
// G = 32, D = 128 items: one elected lane starts a 4 KB copy, the warp waits
// on the stage's barrier. Every wait is bounded (one second of the global
// timer): a wait that runs out counts itself in g_wait_timeouts and the warp
// stops (the count is read through kivi_wait_timeouts; it is zero unless a
// copy never completes).
__device__ unsigned int g_wait_timeouts = 0;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// box of the 3-d tensor map at element coordinates (x, y, z) into shared dst
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// fetch a tensor map into the descriptor cache ahead of its first copy
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// true once the barrier's phase of the given parity has completed (all lanes
// agree); false if it has not within kWaitLimitNs
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    bool done = mbar_try(bar, parity);
    if (!done) {
        const unsigned long long t0 = global_ns();
        while (!(done = mbar_try(bar, parity)) && global_ns() - t0 < kWaitLimitNs) {
        }
    }
    return __all_sync(0xffffffffu, done);
}

struct Items {
    int key_items;   // BH * ng * (D / key item channels)
    int val_items;   // BH * ceil(n_flush / value item rows)
    int ng;          // key groups per head
    int nv;          // value items per head
};

// Key items of group size G and head dim D: G tokens x kCh channels (a warp
// takes key_warp_tokens(G) of them, staged as plain rows of kCh channels); a
// lane owns kTPP tokens x 8 channels, lane = part * kNOc + oc, and part p
// the rows p, p + kNPart, p + 2 kNPart, ... of the warp's share. With
// 64-byte rows (kNOc = 4) the two parts of a quarter warp then read rows of
// both parities, eight different 16-byte bank groups, with no padding rows.
template <int G, int D>
struct KeyShape {
    static constexpr int kCh = key_item_channels(G);  // channels of an item: 64, 32, 32
    static constexpr int kNOc = kCh / 8;              // 8-channel octets: 8, 4 or 4
    static constexpr int kNPart = 32 / kNOc;          // token parts: 4, 8 or 8
    static constexpr int kTPP = key_warp_tokens(G) / kNPart;  // tokens per part: 8
    static constexpr int kQ = D / kCh;                // items per key group: 1 to 16
    static_assert(kQ >= 1, "a key item spans at most the head dim");
};

// Value items of head dim D: kRows token rows of D channels (4 KB); a lane
// owns 64 channels of one row, lane = jp * kRows + row.
template <int D>
struct ValueShape {
    static constexpr int kRows = 2048 / D;  // rows of an item: 32, 16 or 8
    static constexpr int kCpr = D / 8;      // 16-byte chunks per row: 8, 16 or 32
};

// Stage this warp's share of item `item`: key item tokens half * 64 ..
// (G = 128) or the whole key group, or value item vi (a value index, or
// -1 for none).
template <int G, int D>
__device__ __forceinline__ void fetch_item(const FlushArgs& k, const FlushArgs& v, const Items& it, int item,
                                           int half, int vi_in, uint8_t* st, int lane) {
    using KS = KeyShape<G, D>;
    using VS = ValueShape<D>;
    constexpr int RB = 2 * D;  // bytes per fp16 token row
    constexpr int KT = key_warp_tokens(G);
    if (item < it.key_items) {
        const unsigned u = item;  // item >= 0: unsigned division by the power of two kQ is a shift
        const int qs = u % KS::kQ, g = (u / KS::kQ) % it.ng, bh = (u / KS::kQ) / it.ng;
        const int r0 = g * G + half * KT;  // first token of this warp's share
        const uint8_t* src = reinterpret_cast<const uint8_t*>(k.x) + ((long long)bh * k.x_bh_stride + r0) * RB +
                             qs * (KS::kCh * 2);
        constexpr int CPR = KS::kNOc;  // 16-byte chunks per token row
#pragma unroll
        for (int i = lane; i < KT * CPR; i += 32) {  // KT rows x CPR chunks
            const int row = i / CPR, col = i % CPR;
            const bool ok = r0 + row < k.n_flush;
            cp_async16(st + (row * CPR + col) * 16, ok ? (const void*)(src + row * RB + col * 16) : (const void*)src,
                       ok);
        }
    } else if (G != 128 || vi_in >= 0) {
        const unsigned vi = vi_in;
        const int t0 = (vi % it.nv) * VS::kRows, bh = vi / it.nv;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(v.x) + ((long long)bh * v.x_bh_stride + t0) * RB;
#pragma unroll
        for (int i = lane; i < 256; i += 32) {  // kRows rows x kCpr chunks
            const int row = i / VS::kCpr, col = i % VS::kCpr;
            const bool ok = t0 + row < v.n_flush;
            // the layout fetch_item_tma leaves: 64-channel pieces kRows * 128 bytes apart, 128-byte rows
            const int off = (col >> 3) * (VS::kRows * 128) + row * 128 + (((col & 7) ^ (row & 7)) << 4);
            cp_async16(st + off, ok ? (const void*)(src + i * 16) : (const void*)src, ok);
        }
    }
}

// Stage item `item` of group size 32 and head dim D by bulk tensor copies
// (called by one lane): a key item is the 32 x 64 box (tokens x channels) at
// channel 64 * (item mod D / 64) of its group, stored as plain 128-byte rows;
// a value item is the D / 64 boxes of its kRows = 2048 / D rows, 64 channels
// each, box j at st + j * kRows * 128 in the 128-byte swizzle (16-byte chunk
// c of row r at c ^ (r & 7); st is 1024-byte aligned, and so is every box).
// Rows past n_flush arrive as zeros.
template <int D>
__device__ __forceinline__ void fetch_item_tma(const CUtensorMap* kmap, const CUtensorMap* vmap, const Items& it,
                                               int item, uint8_t* st, uint32_t bar) {
    constexpr int kQ = D / 64, kRows = ValueShape<D>::kRows;
    const uint32_t dst = smem_u32(st);
    mbar_expect_tx(bar, 4096);
    if (item < it.key_items) {
        const unsigned u = item;
        const int qs = u % kQ, g = (u / kQ) % it.ng, bh = (u / kQ) / it.ng;
        tma_load_3d(dst, kmap, 64 * qs, g * kG, bh, bar);
    } else {
        const int vi = item - it.key_items;
        const int t0 = (vi % it.nv) * kRows, bh = vi / it.nv;
#pragma unroll
        for (int j = 0; j < kQ; ++j) tma_load_3d(dst + j * kRows * 128, vmap, 64 * j, t0, bh, bar);
    }
}

// keys: lane = part * kNOc + oc; part owns the tokens part, part + kNPart, ...
// of the warp's share of the group (kTPP of them), oc owns 8 channels of this
// item's channel slice.
// At G = 128 the warp holds tokens half * 64 .. of the group, and the two
// warps of a pair (warp, warp ^ 1) exchange their column minima and maxima
// through xchg (32 words per warp; named barrier bar_id over the pair's 64
// threads) before the scales; the half-0 warp stores the scales and zeros.
// FAKE: write the fake-quantized fp16 rows to a.fq instead of codes, scales
// and zeros.
template <int BITS, int MODE, int G, int D>
__device__ __forceinline__ void key_item(const FlushArgs& a, const Items& it, int item, int half, uint32_t* xchg,
                                         int warp, const uint8_t* st, int lane) {
    constexpr bool FAKE = (MODE & 1) != 0, HS = (MODE & 2) != 0;  // fake quantization; fp16 scales
    using KS = KeyShape<G, D>;
    const unsigned u = item;
    const int qs = u % KS::kQ, g = (u / KS::kQ) % it.ng, bh = (u / KS::kQ) / it.ng;
    const int oc = lane % KS::kNOc, part = lane / KS::kNOc;
    const int octet = qs * KS::kNOc + oc;
    const int tw = g * G + half * key_warp_tokens(G);  // first token of the warp's share
    const int t0 = tw + part;                           // this lane's first token
    const int nw = a.n_flush - tw;                      // valid tokens of the share (ragged last group)
    const int nv = nw <= part ? 0 : min(KS::kTPP, (nw - part + KS::kNPart - 1) / KS::kNPart);
    constexpr int kStep = KS::kNPart;                   // tokens between a lane's rows
    const uint4* xs = reinterpret_cast<const uint4*>(st) + part * KS::kNOc + oc;  // row i at xs[i * kStep * kNOc]

    const __half2 pinf = __half2half2(__ushort_as_half(0x7c00));
    const __half2 ninf = __half2half2(__ushort_as_half(0xfc00));
    __half2 mn[4] = {pinf, pinf, pinf, pinf};
    __half2 mx[4] = {ninf, ninf, ninf, ninf};
#pragma unroll
    for (int i = 0; i < KS::kTPP; ++i) {
        if (i < nv) {
            const uint4 x = xs[i * kStep * KS::kNOc];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mn[k] = __hmin2(mn[k], u32_as_h2(w[k]));
                mx[k] = __hmax2(mx[k], u32_as_h2(w[k]));
            }
        }
    }
#pragma unroll
    for (int o = KS::kNOc; o < 32; o <<= 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            mn[k] = __hmin2(mn[k], u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mn[k]), o)));
            mx[k] = __hmax2(mx[k], u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(mx[k]), o)));
        }
    }
    if (G == 128) {  // the pair's other half of the group
        uint32_t* mine = xchg + warp * 32 + oc * 8;
        const uint32_t* theirs = xchg + (warp ^ 1) * 32 + oc * 8;
        if (part == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mine[k] = h2_as_u32(mn[k]);
                mine[4 + k] = h2_as_u32(mx[k]);
            }
        }
        if (warp >> 1) named_barrier<2>(64);  // compile-time ids: 3 hardware barriers, not 16
        else named_barrier<1>(64);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            mn[k] = __hmin2(mn[k], u32_as_h2(theirs[k]));
            mx[k] = __hmax2(mx[k], u32_as_h2(theirs[4 + k]));
        }
    }
    float z[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 lo = __half22float2(mn[k]);
        z[2 * k] = canon(lo.x);
        z[2 * k + 1] = canon(lo.y);
    }
    // the part lanes of a column compute its 8 scales: 2 each (4 parts) or 1
    // each (8 parts)
    constexpr int CPP = 8 / KS::kNPart;
    float my_s[CPP], my_r[CPP];
    {
        const int ch0 = part * CPP;  // first channel of the octet this lane scales
        __half2 hx = mx[0], hn = mn[0];                      // the half2 pair holding it (and its neighbour)
#pragma unroll
        for (int k = 1; k < 4; ++k)
            if ((ch0 >> 1) == k) {
                hx = mx[k];
                hn = mn[k];
            }
        const float2 hi = __half22float2(hx), lo = __half22float2(hn);
#pragma unroll
        for (int c = 0; c < CPP; ++c) {
            const bool odd = ((ch0 + c) & 1) != 0;
            my_s[c] = div_levels<BITS>(__fsub_rn(canon(odd ? hi.y : hi.x), canon(odd ? lo.y : lo.x)));
            if (HS) my_s[c] = __half2float(__float2half_rn(my_s[c]));  // the stored fp16 scale
            my_r[c] = my_s[c] == 0.0f ? 0.0f : rcp_1ulp(my_s[c]);
        }
    }
    float s[8], r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int src = (k / CPP) * KS::kNOc + oc;
        s[k] = __shfl_sync(0xffffffffu, my_s[k % CPP], src);
        r[k] = __shfl_sync(0xffffffffu, my_r[k % CPP], src);
    }
    f32x2 z2[4], r2[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        z2[k] = pk(z[2 * k], z[2 * k + 1]);
        r2[k] = pk(r[2 * k], r[2 * k + 1]);
    }
    // every scale of the item was computed by some lane (my_s), so the vote covers them all
    bool small = false;
#pragma unroll
    for (int c = 0; c < CPP; ++c) small |= my_s[c] < kMinNormalF16;
    const bool clip = HS && warp_has_subnormal_scale(small);
    if (FAKE) {
        uint4* frow = reinterpret_cast<uint4*>(a.fq + ((long long)bh * a.fq_bh_stride + t0) * D) + octet;
#pragma unroll 1
        for (int i = 0; i < nv; ++i)
            frow[i * kStep * (D / 8)] = fake8<BITS, HS>(xs[i * kStep * KS::kNOc], z2, r2, s, clip);
        return;
    }
    if (part == 0 && half == 0) {
        const long long m = ((long long)bh * (a.s_cap / G) + a.s_off / G + g) * D + octet * 8;
        store_scales8<HS>(a.scale, m, s);
        uint4 zp;
        zp.x = h2_as_u32(__floats2half2_rn(z[0], z[1]));
        zp.y = h2_as_u32(__floats2half2_rn(z[2], z[3]));
        zp.z = h2_as_u32(__floats2half2_rn(z[4], z[5]));
        zp.w = h2_as_u32(__floats2half2_rn(z[6], z[7]));
        *reinterpret_cast<uint4*>(a.zero + m) = zp;
    }
    constexpr int ROWB = D * BITS / 8;
    uint8_t* crow = a.codes + ((long long)bh * a.s_cap + a.s_off + t0) * ROWB + octet * BITS;
    auto store_row = [&](int i, uint32_t packed) {
        if (BITS == 4) *reinterpret_cast<uint32_t*>(crow + i * kStep * ROWB) = packed;
        else *reinterpret_cast<uint16_t*>(crow + i * kStep * ROWB) = (uint16_t)packed;
    };
#pragma unroll (kKeyUnroll)
    for (int i = 0; i < nv; ++i) store_row(i, quant8<BITS, HS>(xs[i * kStep * KS::kNOc], z2, r2, s, clip));
}

// min and max of the 8 fp16 of each vector of x, as half2 (min and max of fp16
// are exact, so the order is free)
template <int N>
__device__ __forceinline__ void minmax_tree(const uint4 (&x)[N], __half2& m2, __half2& x2) {
    __half2 mk[N], xk[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
        const __half2 a = u32_as_h2(x[k].x), b = u32_as_h2(x[k].y), c = u32_as_h2(x[k].z), d = u32_as_h2(x[k].w);
        mk[k] = __hmin2(__hmin2(a, b), __hmin2(c, d));
        xk[k] = __hmax2(__hmax2(a, b), __hmax2(c, d));
    }
#pragma unroll
    for (int w = 1; w < N; w <<= 1)
#pragma unroll
        for (int k = 0; k + w < N; k += 2 * w) {
            mk[k] = __hmin2(mk[k], mk[k + w]);
            xk[k] = __hmax2(xk[k], xk[k + w]);
        }
    m2 = mk[0];
    x2 = xk[0];
}

// values: lane = kRows jp + row holds 64 channels of row `row` of the item,
// channels 64 jp .. 64 jp + 63: two groups (G = 32), one (G = 64), or half of
// one, whose min/max it shares with its partner lane (lane ^ kRows, the other
// half of the same row's group) (G = 128). Min/max, scale and codes of a
// group stay in its lane(s); one code store per group or half group.
template <int BITS, int MODE, int G, int D>
__device__ __forceinline__ void value_item(const FlushArgs& a, const Items& it, int vi_in, const uint8_t* st,
                                           int lane) {
    constexpr bool FAKE = (MODE & 1) != 0, HS = (MODE & 2) != 0;  // fake quantization; fp16 scales
    using VS = ValueShape<D>;
    static_assert(G <= D, "a value group lies within one token row");
    const unsigned vi = vi_in;
    const int t0 = (vi % it.nv) * VS::kRows, bh = vi / it.nv;
    const int row = lane % VS::kRows, jp = lane / VS::kRows;
    const bool valid = t0 + row < a.n_flush;
    if (G != 128 && !valid) return;  // (G = 128: both lanes of a row leave together below)
    // the stage holds 64-channel pieces kRows * 128 bytes apart in 128-byte
    // rows (the layout fetch_item_tma leaves): this lane's piece jp
    const uint4* xs = reinterpret_cast<const uint4*>(st + jp * (VS::kRows * 128) + row * 128);
    const long long grow = (long long)bh * a.s_cap + a.s_off + t0 + row;
    constexpr int NG = G == 32 ? 2 : 1;      // groups (or half groups) per lane
    constexpr int NVEC = G == 32 ? 4 : 8;    // 16-byte vectors per group (or half group) in this lane
#pragma unroll
    for (int e = 0; e < NG; ++e) {
        const int cv = (64 * jp + (G == 32 ? 32 * e : 0)) / 8;  // first vector of this lane's channels
        const int cl = cv - 8 * jp;                               // ... within the staged row piece
        uint4 x[NVEC];
#pragma unroll
        for (int k = 0; k < NVEC; ++k) x[k] = xs[(cl + k) ^ (row & 7)];
        __half2 m2, x2;
        minmax_tree<NVEC>(x, m2, x2);
        if (G == 128) {  // the other half of the group sits in lane ^ kRows (same row)
            m2 = __hmin2(m2, u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(m2), VS::kRows)));
            x2 = __hmax2(x2, u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(x2), VS::kRows)));
            if (!valid) return;
        }
        const float z = canon(__half2float(__hmin(__low2half(m2), __high2half(m2))));
        float sc = div_levels<BITS>(__fsub_rn(canon(__half2float(__hmax(__low2half(x2), __high2half(x2)))), z));
        if (HS) sc = __half2float(__float2half_rn(sc));  // the stored fp16 scale
        const float rc = sc == 0.0f ? 0.0f : rcp_1ulp(sc);
        const f32x2 z1 = pk(z, z), r1 = pk(rc, rc);
        const f32x2 z2[4] = {z1, z1, z1, z1}, r2[4] = {r1, r1, r1, r1};
        const float sv[8] = {sc, sc, sc, sc, sc, sc, sc, sc};
        const int j = (64 * jp + (G == 32 ? 32 * e : 0)) / G;  // this group's index in the row
        const bool clip = HS && warp_has_subnormal_scale(sc < kMinNormalF16);
        if (FAKE) {
            uint4* frow = reinterpret_cast<uint4*>(a.fq + ((long long)bh * a.fq_bh_stride + t0 + row) * D) + cv;
            #pragma unroll
            for (int k = 0; k < NVEC; ++k) frow[k] = fake8<BITS, HS>(x[k], z2, r2, sv, clip);
        } else {
            uint32_t pq[NVEC];
            #pragma unroll
            for (int k = 0; k < NVEC; ++k) pq[k] = quant8<BITS, HS>(x[k], z2, r2, sv, clip);
            uint8_t* cdst = a.codes + grow * (D * BITS / 8) + cv * BITS;  // 8 channels per vector
            if (BITS == 4) {
#pragma unroll
                for (int k = 0; k < NVEC; k += 4)
                    *reinterpret_cast<uint4*>(cdst + 4 * k) = make_uint4(pq[k], pq[k + 1], pq[k + 2], pq[k + 3]);
            } else {
#pragma unroll
                for (int k = 0; k < NVEC; k += 4)
                    *reinterpret_cast<uint2*>(cdst + 2 * k) =
                        make_uint2(pq[k] | (pq[k + 1] << 16), pq[k + 2] | (pq[k + 3] << 16));
            }
            if (G != 128 || (jp & 1) == 0) {
                store_scale<HS>(a.scale, grow * (D / G) + j, sc);
                a.zero[grow * (D / G) + j] = __float2half_rn(z);
            }
        }
    }
}

// G = 32 keys (the measured fast path, kept as written for that size):
// lane = part * 8 + oc; part owns tokens [8 part, 8 part + 8) of the
// group, oc owns 8 channels of this 64-channel half. FAKE: write the fake-
// quantized fp16 rows to a.fq instead of codes, scales and zeros.
template <int BITS, int MODE>
__device__ __forceinline__ void key_item_g32(const FlushArgs& a, const Items& it, int item, const uint8_t* st, int lane) {
    constexpr bool FAKE = (MODE & 1) != 0, HS = (MODE & 2) != 0;  // fake quantization; fp16 scales
    const int half = item & 1, g = (item >> 1) % it.ng, bh = (item >> 1) / it.ng;
    const int oc = lane & 7, part = lane >> 3;
    const int octet = half * 8 + oc;
    const int t0 = g * kG + part * 8;
    const int nv = min(8, a.n_flush - t0);  // may be <= 0 in a ragged last group
    const uint4* xs = reinterpret_cast<const uint4*>(st) + (part * 8) * 8 + oc;  // row stride 8 vectors

    const __half2 pinf = __half2half2(__ushort_as_half(0x7c00));
    const __half2 ninf = __half2half2(__ushort_as_half(0xfc00));
    __half2 mn[4] = {pinf, pinf, pinf, pinf};
    __half2 mx[4] = {ninf, ninf, ninf, ninf};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < nv) {
            const uint4 x = xs[i * 8];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
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
    float z[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 lo = __half22float2(mn[k]);
        z[2 * k] = canon(lo.x);
        z[2 * k + 1] = canon(lo.y);
    }
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
        my_s[0] = div_levels<BITS>(__fsub_rn(canon(hi.x), canon(lo.x)));
        my_s[1] = div_levels<BITS>(__fsub_rn(canon(hi.y), canon(lo.y)));
        if (HS) {  // the stored fp16 scales
            my_s[0] = __half2float(__float2half_rn(my_s[0]));
            my_s[1] = __half2float(__float2half_rn(my_s[1]));
        }
        my_r[0] = my_s[0] == 0.0f ? 0.0f : rcp_1ulp(my_s[0]);
        my_r[1] = my_s[1] == 0.0f ? 0.0f : rcp_1ulp(my_s[1]);
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
    // every scale of the item was computed by some lane (my_s), so the vote covers them all
    const bool clip = HS && warp_has_subnormal_scale(my_s[0] < kMinNormalF16 || my_s[1] < kMinNormalF16);
    if (FAKE) {
        uint4* frow = reinterpret_cast<uint4*>(a.fq + ((long long)bh * a.fq_bh_stride + t0) * kD) + octet;
#pragma unroll 1
        for (int i = 0; i < nv; ++i) frow[i * (kD / 8)] = fake8<BITS, HS>(xs[i * 8], z2, r2, s, clip);
        return;
    }
    if (part == 0) {
        const long long m = ((long long)bh * (a.s_cap / kG) + a.s_off / kG + g) * kD + octet * 8;
        store_scales8<HS>(a.scale, m, s);
        uint4 zp;
        zp.x = h2_as_u32(__floats2half2_rn(z[0], z[1]));
        zp.y = h2_as_u32(__floats2half2_rn(z[2], z[3]));
        zp.z = h2_as_u32(__floats2half2_rn(z[4], z[5]));
        zp.w = h2_as_u32(__floats2half2_rn(z[6], z[7]));
        *reinterpret_cast<uint4*>(a.zero + m) = zp;
    }
    constexpr int ROWB = kD * BITS / 8;
    uint8_t* crow = a.codes + ((long long)bh * a.s_cap + a.s_off + t0) * ROWB + octet * BITS;
    auto store_row = [&](int i, uint32_t packed) {
        if (BITS == 4) *reinterpret_cast<uint32_t*>(crow + i * ROWB) = packed;
        else *reinterpret_cast<uint16_t*>(crow + i * ROWB) = (uint16_t)packed;
    };
#pragma unroll (kKeyUnroll)
    for (int i = 0; i < nv; ++i) store_row(i, quant8<BITS, HS>(xs[i * 8], z2, r2, s, clip));
}

// G = 32 values: lane = 16 jp + row; the lane quantizes the groups j = 2 jp and
// 2 jp + 1 (32 channels each) of row `row` of the item: min/max, scale and
// codes of a whole group in one lane, no shuffles, one 16-byte code store
// (4-bit) per group. The stage holds the item as fetch_item_tma leaves it
// (channel halves 2 KB apart, swizzled rows), so the 8 lanes of a quarter
// warp read 8 different 16-byte bank groups.
template <int BITS, int MODE>
__device__ __forceinline__ void value_item_g32(const FlushArgs& a, const Items& it, int item, const uint8_t* st,
                                           int lane) {
    constexpr bool FAKE = (MODE & 1) != 0, HS = (MODE & 2) != 0;  // fake quantization; fp16 scales
    const int vi = item - it.key_items;
    const int t0 = (vi % it.nv) * 16, bh = vi / it.nv;
    const int row = lane & 15, jp = lane >> 4;
    if (t0 + row >= a.n_flush) return;
    const uint4* xs = reinterpret_cast<const uint4*>(st + 2048 * jp + row * 128);  // this lane's 64 channels
    const long long grow = (long long)bh * a.s_cap + a.s_off + t0 + row;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int j = 2 * jp + e;
        uint4 x[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = xs[(4 * e + k) ^ (row & 7)];
        // min / max as a tree (min and max of fp16 are exact, so the order is free)
        __half2 mk[4], xk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __half2 a = u32_as_h2(x[k].x), b = u32_as_h2(x[k].y), c = u32_as_h2(x[k].z),
                          d = u32_as_h2(x[k].w);
            mk[k] = __hmin2(__hmin2(a, b), __hmin2(c, d));
            xk[k] = __hmax2(__hmax2(a, b), __hmax2(c, d));
        }
        const __half2 m2 = __hmin2(__hmin2(mk[0], mk[1]), __hmin2(mk[2], mk[3]));
        const __half2 x2 = __hmax2(__hmax2(xk[0], xk[1]), __hmax2(xk[2], xk[3]));
        const float z = canon(__half2float(__hmin(__low2half(m2), __high2half(m2))));
        float sc = div_levels<BITS>(__fsub_rn(canon(__half2float(__hmax(__low2half(x2), __high2half(x2)))), z));
        if (HS) sc = __half2float(__float2half_rn(sc));  // the stored fp16 scale
        const float rc = sc == 0.0f ? 0.0f : rcp_1ulp(sc);
        const f32x2 z1 = pk(z, z), r1 = pk(rc, rc);
        const f32x2 z2[4] = {z1, z1, z1, z1}, r2[4] = {r1, r1, r1, r1};
        const float sv[8] = {sc, sc, sc, sc, sc, sc, sc, sc};
        const bool clip = HS && warp_has_subnormal_scale(sc < kMinNormalF16);
        if (FAKE) {
            uint4* frow = reinterpret_cast<uint4*>(a.fq + ((long long)bh * a.fq_bh_stride + t0 + row) * kD + 32 * j);
            #pragma unroll
            for (int k = 0; k < 4; ++k) frow[k] = fake8<BITS, HS>(x[k], z2, r2, sv, clip);
        } else {
            auto store_group = [&](const uint32_t (&pq)[4]) {
                if (BITS == 4) {
                    *reinterpret_cast<uint4*>(a.codes + grow * 64 + 16 * j) = make_uint4(pq[0], pq[1], pq[2], pq[3]);
                } else {
                    *reinterpret_cast<uint2*>(a.codes + grow * 32 + 8 * j) =
                        make_uint2(pq[0] | (pq[1] << 16), pq[2] | (pq[3] << 16));
                }
            };
            uint32_t pq[4];
            #pragma unroll
            for (int k = 0; k < 4; ++k) pq[k] = quant8<BITS, HS>(x[k], z2, r2, sv, clip);
            store_group(pq);
            store_scale<HS>(a.scale, grow * (kD / kG) + j, sc);
            a.zero[grow * (kD / kG) + j] = __float2half_rn(z);
        }
    }
}

// Keys, values, or both: warp w of the grid handles items w, w + W, ... of the
// list [key items | value items] (W = total warps). At G = 128 the unit is a
// warp pair (warps 2p, 2p + 1 of a CTA): pair w of the grid handles units
// w, w + W, ... of the list [key items | value item pairs]; both warps of a
// pair walk the same units, so they meet at the same key-item barriers.
// TMA (G = 32 only): the stages are filled by bulk tensor copies (kmap: the
// keys, boxes of 32 tokens x 64 channels; vmap: the values, boxes of
// 2048 / D tokens x 64 channels, 128-byte swizzle), each completing on its
// stage's shared-memory barrier; otherwise they are filled with cp.async
// (the maps are unused).
template <int BITS, int MODE, int G, int D, bool TMA>
__global__ void __launch_bounds__(kThreads, blocks_per_sm<TMA>())
    flush_kernel(FlushArgs k, FlushArgs v, Items it, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap) {
    static_assert(!TMA || G == 32, "bulk copies stage the items of group size 32 only");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    constexpr bool kTma = TMA;
    // the swizzled value boxes want 1024-byte aligned stages
    uint8_t* const smem = kTma ? smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u) : smem_raw;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kStageBytes = Stage<G>::kBytes;
    uint8_t* const base = smem + warp * 2 * kStageBytes;
    // kTma: this warp's two stage barriers (8 bytes each) after all stages
    const uint32_t bar0 = smem_u32(smem + (kThreads / 32) * 2 * kStageBytes) + warp * 16;
    if (kTma) {
        if (threadIdx.x == 0) {  // the maps this launch uses, while the previous kernel may still run
            if (it.key_items > 0) prefetch_map(&kmap);
            if (it.val_items > 0) prefetch_map(&vmap);
        }
        if (lane == 0) {
            mbar_init(bar0);
            mbar_init(bar0 + 8);
            mbar_init_fence();
        }
        __syncwarp();
    }
    constexpr bool kPair = G == 128;
    const int half = kPair ? warp & 1 : 0;
    const int per_cta = kPair ? kThreads / 64 : kThreads / 32;        // units a CTA walks at a time
    const int unit0 = blockIdx.x * per_cta + (kPair ? warp >> 1 : warp);
    const int total = it.key_items + (kPair ? (it.val_items + 1) / 2 : it.val_items);
    const int stride = gridDim.x * per_cta;
    uint32_t* const xchg = reinterpret_cast<uint32_t*>(smem + (kThreads / 32) * 2 * kStageBytes);
    // value item of unit u for this warp, or -1 (a pair's second warp past the last value item)
    auto value_of = [&](int u) {
        if (!kPair) return u - it.key_items;
        const int vi = 2 * (u - it.key_items) + half;
        return vi < it.val_items ? vi : -1;
    };
    int item = unit0;
    pdl_wait();
    if (kTma) {
        if (lane == 0) {
            if (item < total) fetch_item_tma<D>(&kmap, &vmap, it, item, base, bar0);
            if (item + stride < total)
                fetch_item_tma<D>(&kmap, &vmap, it, item + stride, base + kStageBytes, bar0 + 8);
        }
    } else {
        if (item < total) fetch_item<G, D>(k, v, it, item, half, value_of(item), base, lane);
        cp_async_commit();
        if (item + stride < total) fetch_item<G, D>(k, v, it, item + stride, half, value_of(item + stride),
                                                    base + kStageBytes, lane);
        cp_async_commit();
    }
    pdl_trigger();
    for (int n = 0; item < total; item += stride, ++n) {
        uint8_t* S = base + (n & 1) * kStageBytes;  // stage n mod 2
        if (kTma) {
            // use n >> 1 of this stage's barrier completes its phase of parity (n >> 1) & 1
            if (!mbar_wait(bar0 + 8 * (n & 1), (n >> 1) & 1)) {
                // gave up on this copy: count it, wait (bounded) for this and
                // the other stage's copy, and stop
                if (lane == 0) atomicAdd(&g_wait_timeouts, 1u);
                mbar_wait(bar0 + 8 * (n & 1), (n >> 1) & 1);
                if (item + stride < total) mbar_wait(bar0 + 8 * ((n + 1) & 1), ((n + 1) >> 1) & 1);
                return;
            }
        } else {
            cp_async_wait1();
        }
        __syncwarp();
        if (G == 32 && D == kD) {  // the generic item code at G = 32 measured 0.7 % slower than this form
            if (item < it.key_items) key_item_g32<BITS, MODE>(k, it, item, S, lane);
            else value_item_g32<BITS, MODE>(v, it, item, S, lane);
        } else {
            if (item < it.key_items) {
                key_item<BITS, MODE, G, D>(k, it, item, half, xchg + (n & 1) * (kThreads / 32) * 32, warp, S, lane);
            } else {
                const int vi = value_of(item);
                if (!kPair || vi >= 0) value_item<BITS, MODE, G, D>(v, it, vi, S, lane);
            }
        }
        __syncwarp();
        if (kTma) {
            // every lane has read stage S: refill it
            if (lane == 0 && item + 2 * stride < total)
                fetch_item_tma<D>(&kmap, &vmap, it, item + 2 * stride, S, bar0 + 8 * (n & 1));
        } else {
            if (item + 2 * stride < total)
                fetch_item<G, D>(k, v, it, item + 2 * stride, half, value_of(item + 2 * stride), S, lane);
            cp_async_commit();
        }
    }
}

// cuTensorMapEncodeTiled from the driver (looked up once; null if the driver
// has none)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiledFn) nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The tensor map of the flush input a.x ([BH, x_bh_stride, D] fp16, tokens
// [0, n_flush) of each head; rows past n_flush read as zeros) with boxes of
// `rows` tokens x `cols` channels (cols * 2 bytes a multiple of 16). a.x is
// 16-byte aligned and the row and head strides (2D and 2D x_bh_stride bytes)
// are multiples of 16, as the copy needs.
cudaError_t encode_rows_map(CUtensorMap* m, const FlushArgs& a, unsigned cols, unsigned rows,
                            CUtensorMapSwizzle swizzle) {
    const EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)a.D, (cuuint64_t)a.n_flush, (cuuint64_t)a.BH};
    const cuuint64_t strides[2] = {(cuuint64_t)a.D * 2, (cuuint64_t)a.x_bh_stride * a.D * 2};
    const cuuint32_t box[3] = {cols, rows, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(a.x), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// TMA: kmap and vmap describe k.x and v.x (encode_rows_map); otherwise unused.
template <int BITS, int MODE, int G, int D, bool TMA>
cudaError_t launch_items_t(const FlushArgs& k, const FlushArgs& v, const Items& it, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, cudaStream_t stream) {
    static int grid_cap = 0;
    static bool configured = false;  // benign race: every caller sets the same values
    constexpr bool kTma = TMA;
    // kTma: two stage barriers per warp and room to align the stages to 1024 bytes
    const int smem = (kThreads / 32) * 2 * Stage<G>::kBytes + (G == 128 ? kXchgBytes : 0) +
                     (kTma ? (kThreads / 32) * 16 + 1024 : 0);
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(flush_kernel<BITS, MODE, G, D, TMA>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        grid_cap = sm_count() * blocks_per_sm<TMA>();
        configured = true;
    }
    // units: items, or at G = 128 key items and value item pairs, each for a warp pair
    const long long total = (long long)it.key_items + (G == 128 ? (it.val_items + 1) / 2 : it.val_items);
    if (total <= 0) return cudaSuccess;
    const int per_cta = G == 128 ? kThreads / 64 : kThreads / 32;
    long long blocks = (total + per_cta - 1) / per_cta;
    if (blocks > grid_cap) blocks = grid_cap;
    return launch_pdl(flush_kernel<BITS, MODE, G, D, TMA>, dim3((unsigned)blocks), kThreads, smem, stream, k, v, it,
                      kmap, vmap);
}

// The bulk-copy kernel takes flushes (not fake quantization) of G = 32 with
// more items than one wave of the cp.async grid: measured on the long 2-bit
// flush 29.5 us against 31.2 (D = 128), 28.3 against 30.8 (D = 64) and 29.6
// against 31.1 (D = 256). The cp.async kernel keeps fake
// quantization (54.7 us against 56.1 at 4 and 60.9 at 6 CTAs per SM),
// launches of at most one item per warp (the qwen8b flush, 5.7 against
// 6.1 us: one item's latency) and the other group sizes (bulk copies of the
// 64 x 32 key boxes measured 34.2 against 32.5 us at G = 64, and 36.0
// against 36.0 at G = 128, whose warp pairs' exchange sets the pace). The
// bulk copies need the driver's tensor-map encoder: where it is missing, or
// rejects a map, the cp.async kernel runs instead (the same results).
template <int BITS, int MODE, int G, int D>
cudaError_t launch_items(const FlushArgs& k, const FlushArgs& v, const Items& it, cudaStream_t stream) {
    CUtensorMap kmap{}, vmap{};
    constexpr bool kCanTma = G == 32 && (MODE & 1) == 0;
    if constexpr (kCanTma) {
        const long long units = (long long)it.key_items + it.val_items;
        if (units > (long long)sm_count() * blocks_per_sm<false>() * (kThreads / 32) &&
            (it.key_items == 0 || encode_rows_map(&kmap, k, 64, kG, CU_TENSOR_MAP_SWIZZLE_NONE) == cudaSuccess) &&
            (it.val_items == 0 ||
             encode_rows_map(&vmap, v, 64, ValueShape<D>::kRows, CU_TENSOR_MAP_SWIZZLE_128B) == cudaSuccess))
            return launch_items_t<BITS, MODE, G, D, true>(k, v, it, kmap, vmap, stream);
    }
    return launch_items_t<BITS, MODE, G, D, false>(k, v, it, kmap, vmap, stream);
}

// Pointers of heads [h0, h0 + nh) of a flush.
FlushArgs head_slice(const FlushArgs& a, int h0, int nh, int bits, int axis) {
    FlushArgs s = a;
    s.BH = nh;
    s.x += (long long)h0 * a.x_bh_stride * a.D;
    if (a.fq) {
        s.fq += (long long)h0 * a.fq_bh_stride * a.D;
        return s;
    }
    s.codes += (long long)h0 * a.s_cap * (a.D * bits / 8);
    const long long meta = axis == 0 ? (long long)(a.s_cap / a.G) * a.D : (long long)a.s_cap * (a.D / a.G);
    s.scale = a.scale_f16 ? reinterpret_cast<float*>(reinterpret_cast<__half*>(a.scale) + h0 * meta)
                          : a.scale + h0 * meta;
    s.zero += h0 * meta;
    return s;
}

// (G, D) pairs: G in {32, 64, 128}, D in {64, 128, 256}, G <= D
template <int BITS, int MODE>
cudaError_t launch_items_g(const FlushArgs& k, const FlushArgs& v, const Items& it, int G, int D,
                           cudaStream_t stream) {
    switch (G * 1000 + D) {
        case 32064: return launch_items<BITS, MODE, 32, 64>(k, v, it, stream);
        case 32128: return launch_items<BITS, MODE, 32, 128>(k, v, it, stream);
        case 32256: return launch_items<BITS, MODE, 32, 256>(k, v, it, stream);
        case 64064: return launch_items<BITS, MODE, 64, 64>(k, v, it, stream);
        case 64128: return launch_items<BITS, MODE, 64, 128>(k, v, it, stream);
        case 64256: return launch_items<BITS, MODE, 64, 256>(k, v, it, stream);
        case 128128: return launch_items<BITS, MODE, 128, 128>(k, v, it, stream);
        case 128256: return launch_items<BITS, MODE, 128, 256>(k, v, it, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Item counts must fit in an int; inputs beyond that are split by heads.
cudaError_t launch_flush_impl(const FlushArgs& k, const FlushArgs& v, bool do_k, bool do_v, int bits,
                              cudaStream_t stream) {
    const FlushArgs& a = do_k ? k : v;
    if (a.n_flush <= 0 || a.BH <= 0) return cudaSuccess;
    const int G = a.G, D = a.D;
    const int rows = 2048 / D;  // token rows per value item
    const int ng = (a.n_flush + G - 1) / G, nv = (a.n_flush + rows - 1) / rows;
    const int kq = D / key_item_channels(G);  // key items per group
    const int per_head = (do_k ? kq * ng : 0) + (do_v ? nv : 0);
    const int max_heads = (int)(0x3fffffff / per_head) > 0 ? (int)(0x3fffffff / per_head) : 1;
    for (int h0 = 0; h0 < a.BH; h0 += max_heads) {
        const int nh = a.BH - h0 < max_heads ? a.BH - h0 : max_heads;
        FlushArgs ks = k, vs = v;
        if (do_k) ks = head_slice(k, h0, nh, bits, 0);
        if (do_v) vs = head_slice(v, h0, nh, bits, 1);
        Items it;
        it.ng = ng;
        it.nv = nv;
        it.key_items = do_k ? nh * kq * ng : 0;
        it.val_items = do_v ? nh * nv : 0;
        // MODE bit 0: fake quantization; bit 1: fp16 scales
        const int mode = (a.fq != nullptr ? 1 : 0) | (a.scale_f16 ? 2 : 0);
        cudaError_t e = cudaErrorInvalidValue;
        switch (bits * 10 + mode) {
            case 40: e = launch_items_g<4, 0>(ks, vs, it, G, D, stream); break;
            case 41: e = launch_items_g<4, 1>(ks, vs, it, G, D, stream); break;
            case 42: e = launch_items_g<4, 2>(ks, vs, it, G, D, stream); break;
            case 43: e = launch_items_g<4, 3>(ks, vs, it, G, D, stream); break;
            case 20: e = launch_items_g<2, 0>(ks, vs, it, G, D, stream); break;
            case 21: e = launch_items_g<2, 1>(ks, vs, it, G, D, stream); break;
            case 22: e = launch_items_g<2, 2>(ks, vs, it, G, D, stream); break;
            case 23: e = launch_items_g<2, 3>(ks, vs, it, G, D, stream); break;
            default: break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_flush(int axis, const FlushArgs& a, int bits, cudaStream_t stream) {
    return launch_flush_impl(a, a, axis == 0, axis == 1, bits, stream);
}

cudaError_t launch_flush_kv(const FlushArgs& k, const FlushArgs& v, int bits, cudaStream_t stream) {
    return launch_flush_impl(k, v, true, true, bits, stream);
}

cudaError_t launch_fake_quant(const FlushArgs& k, const FlushArgs& v, bool do_k, bool do_v, int bits,
                              cudaStream_t stream) {
    return launch_flush_impl(k, v, do_k, do_v, bits, stream);
}

cudaError_t read_wait_timeouts(unsigned int* count, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(unsigned int));
    if (e == cudaSuccess && reset) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace kivi

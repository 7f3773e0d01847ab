/*
 * kivi_oracle.c -- plain, slow CPU reference for KIVI (asymmetric 2/4-bit
 * KV-cache quantization with an fp16 residual window).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the CPU
 * baseline leg of the benchmark. It shares nothing with the CUDA path.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math (never -ffast-math), default
 * FE_TONEAREST rounding. Every fp32 step below is one IEEE binary32 operation
 * rounded to nearest-even, written as separate statements so that no step is
 * fused or reassociated.
 *
 * Citation tags (page title, section):
 *  [F]  VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly 0%
 *       Faster" (the fused KIVI post)
 *  [Q]  VeloxQuant-MLX blog, "A Kernel That Wasn't There"
 *  [R]  VeloxQuant-MLX benchmarks page, "KV-Cache Kernel Roofline"
 *
 * Readings where the pages are silent (all listed in the design notes):
 *  - quantizer arithmetic is fp32 after widening the fp16 inputs;
 *  - scale is stored as fp32, zero as fp16 (lossless: zero is an fp16 input);
 *    with the ORC_SCALE_F16 option bit set in `bits`, scale is stored as
 *    binary16 (round to nearest even) and the codes are computed with that
 *    stored scale, so a dequant reproduces exactly what the flush used;
 *  - min and max of -0.0 are taken as +0.0, so the stored zero and scale
 *    never carry a negative sign whatever order equal values are met in;
 *  - max == min gives scale 0, every code 0, recon == min;
 *  - codes are packed along D inside each token row, low bits first;
 *  - the decode reads store tokens as their fp32 reconstruction.
 */
#include "kivi_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary32                                           */
/* ------------------------------------------------------------------------ */

/* value = (-1)^s * 2^(e-15) * (1 + m/1024) for 0 < e < 31,
 *         (-1)^s * 2^-14 * (m/1024)          for e == 0 (zero, subnormal),
 *         +-inf / NaN                         for e == 31.                  */
float orc_half_to_float(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    float mag;
    if (e == 0)
        mag = ldexpf((float)m, -24);
    else if (e == 31)
        mag = m ? NAN : INFINITY;
    else
        mag = ldexpf((float)(1024 + m), e - 25);
    return s ? -mag : mag;
}

/* Round |f| to the binary16 grid of its binade (quantum 2^(E-10), with the
 * subnormal quantum 2^-24 below 2^-14), ties to even; carry into the next
 * binade when the significand rounds up to 2048; overflow to infinity. */
uint16_t orc_float_to_half(float f)
{
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f))
        return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)f);
    if (isinf(a))
        return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;         /* a in [2^E, 2^(E+1)) */
    if (E < -14)
        E = -14;            /* subnormal range shares the 2^-24 quantum */
    double n = rint(a / ldexp(1.0, E - 10)); /* exact scaling, then RNE */
    if (n >= 2048.0) {
        n = n / 2.0;
        E += 1;
    }
    if (E > 15)
        return (uint16_t)(sign | 0x7c00u);
    if (n < 1024.0)         /* only reachable with E == -14: subnormal */
        return (uint16_t)(sign | (uint16_t)n);
    return (uint16_t)(sign | (uint16_t)(((E + 15) << 10) | ((int)n - 1024)));
}

void orc_half_to_float_n(const uint16_t* h, float* f, long n)
{
    for (long i = 0; i < n; ++i)
        f[i] = orc_half_to_float(h[i]);
}

void orc_float_to_half_n(const float* f, uint16_t* h, long n)
{
    for (long i = 0; i < n; ++i)
        h[i] = orc_float_to_half(f[i]);
}

/* ------------------------------------------------------------------------ */
/* Flush plan                                                               */
/* ------------------------------------------------------------------------ */

/* [F] "What we're actually optimizing": the newest residual_length tokens stay
 * in fp16; once enough fresh tokens accumulate they are quantized as a batch.
 * Reading (checked against the flush/layer column of [F] "The full end-to-end
 * record", Generation 1: 559 -> 512, 2059 -> 2016, 8209 -> 8160 at R = G = 32
 * with 2048-token prefill chunks): a window of n_res tokens flushes whole
 * groups while it holds at least R + G tokens, leaving R <= n_res < R + G.
 * residual_length == 0 means "quantize everything", a ragged last group
 * included. */
int orc_flush_count(int n_res, int residual_length, int group_size)
{
    if (n_res <= 0)
        return 0;
    if (residual_length == 0)
        return n_res;
    int over = n_res - residual_length;
    if (over < group_size)
        return 0;
    return (over / group_size) * group_size;
}

/* ------------------------------------------------------------------------ */
/* One quantization group                                                   */
/* ------------------------------------------------------------------------ */

/* [F] "What we're actually optimizing" gives the textbook asymmetric min/max
 * quantizer:
 *     zero  = min(group)
 *     scale = (max(group) - min(group)) / (2^bits - 1)
 *     q     = round((x - zero) / scale)          then clip to [0, 2^bits-1]
 * and [F] "Three ways to be off by one bit" #2 fixes the rounding to
 * half-to-even (rint). Each line is one fp32 operation.
 * `bits` is the bit width, optionally ORed with ORC_SCALE_F16: the scale is
 * then rounded to binary16 before any code is computed (the stored scale is
 * the one the codes use). The fp16 scale can be 0 for a range far below the
 * fp16 grid (every code 0), and a subnormal fp16 scale can leave a quotient
 * past 2^bits - 1, which the clip catches. *scale receives the scale used. */
void orc_quantize_group(const float* v, int n, int bits,
                        uint8_t* codes, float* scale, float* zero)
{
    int f16_scale = (bits & ORC_SCALE_F16) != 0;
    bits &= ORC_BITS_MASK;
    float mn = v[0];
    float mx = v[0];
    for (int i = 1; i < n; ++i) {
        if (v[i] < mn) mn = v[i];
        if (v[i] > mx) mx = v[i];
    }
    mn = mn + 0.0f;                          /* -0.0 -> +0.0: canonical zero */
    mx = mx + 0.0f;                          /* and canonical range sign */
    float levels = (float)((1 << bits) - 1); /* 2^bits - 1 */
    float range = mx - mn;
    float s = range / levels;
    if (f16_scale)
        s = orc_half_to_float(orc_float_to_half(s)); /* the stored binary16 scale */
    for (int i = 0; i < n; ++i) {
        int q = 0;
        if (s != 0.0f) {                     /* max == min: every code 0 */
            float a = v[i] - mn;
            float t = a / s;
            float r = rintf(t);
            if (r < 0.0f) r = 0.0f;
            if (r > levels) r = levels;
            q = (int)r;
        }
        codes[i] = (uint8_t)q;
    }
    *scale = s;
    *zero = mn;
}

/* A stored scale: fp32, or binary16 under ORC_SCALE_F16 (element m of the
 * array either way). */
static void store_scale(void* scale, long m, float s, int bits)
{
    if (bits & ORC_SCALE_F16)
        ((uint16_t*)scale)[m] = orc_float_to_half(s);
    else
        ((float*)scale)[m] = s;
}

static float load_scale(const void* scale, long m, int bits)
{
    if (bits & ORC_SCALE_F16)
        return orc_half_to_float(((const uint16_t*)scale)[m]);
    return ((const float*)scale)[m];
}

/* [F] "Three ways to be off by one bit" #1: the reconstruction is a multiply
 * followed by a separate add (two roundings, no fused multiply-add). */
static float recon_one(int q, float s, float z)
{
    float prod = (float)q * s;
    float out = prod + z;
    return out;
}

/* ------------------------------------------------------------------------ */
/* Packing                                                                  */
/* ------------------------------------------------------------------------ */

/* Element i of a row goes to byte (i*bits)/8 at bit offset (i*bits)%8. */
void orc_pack_codes(const uint8_t* codes, int n, int bits, uint8_t* packed)
{
    int nbytes = n * bits / 8;
    memset(packed, 0, (size_t)nbytes);
    for (int i = 0; i < n; ++i) {
        int bit = i * bits;
        packed[bit / 8] |= (uint8_t)((codes[i] & ((1 << bits) - 1)) << (bit % 8));
    }
}

void orc_unpack_codes(const uint8_t* packed, int n, int bits, uint8_t* codes)
{
    for (int i = 0; i < n; ++i) {
        int bit = i * bits;
        codes[i] = (uint8_t)((packed[bit / 8] >> (bit % 8)) & ((1 << bits) - 1));
    }
}

/* ------------------------------------------------------------------------ */
/* Flush                                                                    */
/* ------------------------------------------------------------------------ */

/* Gather the group into a buffer of G slots. A ragged group (fewer than G
 * real elements) is padded by repeating its last real element, as [F] "Three
 * ways to be off by one bit" #3 describes for the reference's reshape; the pad
 * slots never change min or max and their codes are discarded. */
static int fill_group(float* buf, int G, const float* real, int n_real)
{
    for (int i = 0; i < n_real; ++i)
        buf[i] = real[i];
    for (int i = n_real; i < G; ++i)
        buf[i] = real[n_real - 1];
    return G;
}

/* [F] "The layout problem that shapes everything" and "Kernel A": keys are
 * [BH, S, D] row-contiguous, and a key group is G consecutive tokens of one
 * channel d (stride D apart in memory). One scale and zero per
 * (head, group, channel). */
void orc_flush_keys(const uint16_t* x, int BH, int x_bh_stride, int n_flush,
                    int D, int G, int bits,
                    uint8_t* codes, void* kscale, uint16_t* kzero,
                    int s_off, int s_cap)
{
    int width = bits & ORC_BITS_MASK;
    int row_bytes = D * width / 8;
    int ng_cap = s_cap / G;
    int ng = (n_flush + G - 1) / G;
    float* real = (float*)malloc(sizeof(float) * (size_t)G);
    float* buf = (float*)malloc(sizeof(float) * (size_t)G);
    uint8_t* q = (uint8_t*)malloc((size_t)G);
    uint8_t* rows = (uint8_t*)malloc((size_t)n_flush * (size_t)D + 1);
    for (int bh = 0; bh < BH; ++bh) {
        const uint16_t* xb = x + (long)bh * x_bh_stride * D;
        for (int g = 0; g < ng; ++g) {
            int t0 = g * G;
            int t1 = t0 + G < n_flush ? t0 + G : n_flush;
            for (int d = 0; d < D; ++d) {
                for (int t = t0; t < t1; ++t)
                    real[t - t0] = orc_half_to_float(xb[(long)t * D + d]);
                int n = fill_group(buf, G, real, t1 - t0);
                float s, z;
                orc_quantize_group(buf, n, bits, q, &s, &z);
                for (int t = t0; t < t1; ++t)
                    rows[(long)t * D + d] = q[t - t0];
                long m = ((long)bh * ng_cap + (s_off / G + g)) * D + d;
                store_scale(kscale, m, s, bits);
                kzero[m] = orc_float_to_half(z);
            }
        }
        for (int t = 0; t < n_flush; ++t)
            orc_pack_codes(rows + (long)t * D, D, width,
                           codes + ((long)bh * s_cap + s_off + t) * row_bytes);
    }
    free(real);
    free(buf);
    free(q);
    free(rows);
}

/* [F] "The layout problem" and "Kernel B": a value group is G consecutive
 * channels of one token (the contiguous axis). One scale and zero per
 * (head, token, group). */
void orc_flush_values(const uint16_t* x, int BH, int x_bh_stride, int n_flush,
                      int D, int G, int bits,
                      uint8_t* codes, void* vscale, uint16_t* vzero,
                      int s_off, int s_cap)
{
    int width = bits & ORC_BITS_MASK;
    int row_bytes = D * width / 8;
    int ngd = (D + G - 1) / G;
    float* real = (float*)malloc(sizeof(float) * (size_t)G);
    float* buf = (float*)malloc(sizeof(float) * (size_t)G);
    uint8_t* q = (uint8_t*)malloc((size_t)G);
    uint8_t* row = (uint8_t*)malloc((size_t)D);
    for (int bh = 0; bh < BH; ++bh) {
        const uint16_t* xb = x + (long)bh * x_bh_stride * D;
        for (int t = 0; t < n_flush; ++t) {
            for (int j = 0; j < ngd; ++j) {
                int d0 = j * G;
                int d1 = d0 + G < D ? d0 + G : D;
                for (int d = d0; d < d1; ++d)
                    real[d - d0] = orc_half_to_float(xb[(long)t * D + d]);
                int n = fill_group(buf, G, real, d1 - d0);
                float s, z;
                orc_quantize_group(buf, n, bits, q, &s, &z);
                for (int d = d0; d < d1; ++d)
                    row[d] = q[d - d0];
                long m = ((long)bh * s_cap + s_off + t) * ngd + j;
                store_scale(vscale, m, s, bits);
                vzero[m] = orc_float_to_half(z);
            }
            orc_pack_codes(row, D, width,
                           codes + ((long)bh * s_cap + s_off + t) * row_bytes);
        }
    }
    free(real);
    free(buf);
    free(q);
    free(row);
}

/* ------------------------------------------------------------------------ */
/* Dequantize                                                               */
/* ------------------------------------------------------------------------ */

/* recon = q * scale + zero (two roundings), per element, with the scale and
 * zero of the element's group: keys by (token group, channel), values by
 * (token, channel group). */
void orc_recon_f32(int axis, const uint8_t* codes, const void* scale,
                   const uint16_t* zero, int BH, int S, int D, int G, int bits,
                   int s_cap, float* out)
{
    int width = bits & ORC_BITS_MASK;
    int row_bytes = D * width / 8;
    int ng_cap = s_cap / G;
    int ngd = (D + G - 1) / G;
    uint8_t* row = (uint8_t*)malloc((size_t)D);
    for (int bh = 0; bh < BH; ++bh) {
        for (int t = 0; t < S; ++t) {
            orc_unpack_codes(codes + ((long)bh * s_cap + t) * row_bytes, D, width, row);
            for (int d = 0; d < D; ++d) {
                long m;
                if (axis == 0)
                    m = ((long)bh * ng_cap + t / G) * D + d;
                else
                    m = ((long)bh * s_cap + t) * ngd + d / G;
                float z = orc_half_to_float(zero[m]);
                out[((long)bh * S + t) * D + d] = recon_one(row[d], load_scale(scale, m, bits), z);
            }
        }
    }
    free(row);
}

void orc_dequant(int axis, const uint8_t* codes, const void* scale,
                 const uint16_t* zero, int BH, int S, int D, int G, int bits,
                 int s_cap, uint16_t* out)
{
    long n = (long)BH * S * D;
    float* f = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    orc_recon_f32(axis, codes, scale, zero, BH, S, D, G, bits, s_cap, f);
    orc_float_to_half_n(f, out, n);
    free(f);
}

/* ------------------------------------------------------------------------ */
/* fp16 residual window                                                     */
/* ------------------------------------------------------------------------ */

void orc_residual_append(uint16_t* res, int BH, int res_cap, int D, int n_res,
                         const uint16_t* src, int src_bh_stride, int n_new)
{
    for (int bh = 0; bh < BH; ++bh)
        for (int t = 0; t < n_new; ++t)
            for (int d = 0; d < D; ++d)
                res[((long)bh * res_cap + n_res + t) * D + d] =
                    src[((long)bh * src_bh_stride + t) * D + d];
}

void orc_residual_compact(uint16_t* res, int BH, int res_cap, int D, int n_res,
                          int n_drop)
{
    for (int bh = 0; bh < BH; ++bh)
        for (int t = 0; t + n_drop < n_res; ++t)
            for (int d = 0; d < D; ++d)
                res[((long)bh * res_cap + t) * D + d] =
                    res[((long)bh * res_cap + t + n_drop) * D + d];
}

/* ------------------------------------------------------------------------ */
/* Single-token decode-attend                                               */
/* ------------------------------------------------------------------------ */

/* [F] "So why does the kernel ship?" (dequant-in-SDPA) and [R] "KV-Cache
 * Kernel Roofline" (fused decode+attend, one query token): plain softmax
 * attention of one query token per head over the S_q quantized store tokens
 * followed by the n_res fp16 residual tokens:
 *     score_t = sm_scale * sum_d q[d] * K[t][d]
 *     out[d]  = sum_t softmax(score)_t * V[t][d]
 * Store rows are the fp32 reconstruction; query head h reads KV head
 * h / (Hq / Hkv) (grouped-query attention, [Q] "Picking a model"). No mask:
 * the single query sees every cached token. Computed in float64. */
void orc_decode_attend(const uint16_t* q,
                       const uint8_t* kcodes, const void* kscale, const uint16_t* kzero,
                       const uint8_t* vcodes, const void* vscale, const uint16_t* vzero,
                       int S_q, int s_cap,
                       const uint16_t* k_res, const uint16_t* v_res, int n_res, int res_cap,
                       int B, int Hq, int Hkv, int D, int G, int bits, double sm_scale,
                       double* out)
{
    int T = S_q + n_res;
    int group = Hq / Hkv;
    float* kf = (float*)malloc(sizeof(float) * (size_t)(S_q > 0 ? S_q : 1) * D);
    float* vf = (float*)malloc(sizeof(float) * (size_t)(S_q > 0 ? S_q : 1) * D);
    double* K = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * D);
    double* V = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * D);
    double* score = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    int row_bytes = D * (bits & ORC_BITS_MASK) / 8;
    int ng_cap = s_cap / G;
    int ngd = (D + G - 1) / G;
    long esz = (bits & ORC_SCALE_F16) ? 2 : 4; /* bytes per stored scale */
    for (int b = 0; b < B; ++b) {
        for (int hk = 0; hk < Hkv; ++hk) {
            int bh = b * Hkv + hk;
            /* Gather this KV head's rows: store (fp32 recon) then residual. */
            if (S_q > 0) {
                long off_codes = (long)bh * s_cap * row_bytes;
                orc_recon_f32(0, kcodes + off_codes, (const char*)kscale + (long)bh * ng_cap * D * esz,
                              kzero + (long)bh * ng_cap * D, 1, S_q, D, G, bits, s_cap, kf);
                orc_recon_f32(1, vcodes + off_codes, (const char*)vscale + (long)bh * s_cap * ngd * esz,
                              vzero + (long)bh * s_cap * ngd, 1, S_q, D, G, bits, s_cap, vf);
            }
            for (int t = 0; t < S_q; ++t)
                for (int d = 0; d < D; ++d) {
                    K[(long)t * D + d] = (double)kf[(long)t * D + d];
                    V[(long)t * D + d] = (double)vf[(long)t * D + d];
                }
            for (int t = 0; t < n_res; ++t)
                for (int d = 0; d < D; ++d) {
                    long src = ((long)bh * res_cap + t) * D + d;
                    K[(long)(S_q + t) * D + d] = (double)orc_half_to_float(k_res[src]);
                    V[(long)(S_q + t) * D + d] = (double)orc_half_to_float(v_res[src]);
                }
            for (int h = hk * group; h < (hk + 1) * group; ++h) {
                const uint16_t* qh = q + ((long)b * Hq + h) * D;
                double* oh = out + ((long)b * Hq + h) * D;
                double mx = -INFINITY;
                for (int t = 0; t < T; ++t) {
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d)
                        acc += (double)orc_half_to_float(qh[d]) * K[(long)t * D + d];
                    score[t] = sm_scale * acc;
                    if (score[t] > mx) mx = score[t];
                }
                double denom = 0.0;
                for (int t = 0; t < T; ++t) {
                    score[t] = exp(score[t] - mx);
                    denom += score[t];
                }
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int t = 0; t < T; ++t)
                        acc += score[t] * V[(long)t * D + d];
                    oh[d] = T > 0 ? acc / denom : 0.0;
                }
            }
        }
    }
    free(kf);
    free(vf);
    free(K);
    free(V);
    free(score);
}

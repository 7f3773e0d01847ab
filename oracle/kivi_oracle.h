/*
 * kivi_oracle.h -- plain, slow CPU reference for KIVI's flush, dequantize and
 * single-token decode-attend.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library. The CUDA product path
 * shares no code, header, table or helper with it, and it never calls into
 * the CUDA path.
 *
 * Sources (see oracle/kivi_oracle.c for the step-by-step citations):
 *  [F] VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly 0%
 *      Faster" (fused KIVI post): sections "What we're actually optimizing",
 *      "The layout problem that shapes everything", "Kernel A", "Kernel B",
 *      "Three ways to be off by one bit", "The full end-to-end record",
 *      "So why does the kernel ship?".
 *  [Q] VeloxQuant-MLX blog, "A Kernel That Wasn't There" (Qwen3-8B on M4).
 *  [R] VeloxQuant-MLX benchmarks page, "KV-Cache Kernel Roofline".
 *
 * Every array is plain host memory owned by the caller. fp16 values are
 * passed as their IEEE binary16 bit patterns (uint16_t).
 */
#ifndef KIVI_ORACLE_H
#define KIVI_ORACLE_H

#include <stdint.h>

/* `bits` arguments: the bit width (2 or 4) in the low byte, optionally ORed
 * with ORC_SCALE_F16 to store every scale as binary16 instead of fp32 (the
 * codes are then computed with the stored binary16 scale). Scale arrays are
 * float32 or uint16 (binary16 bit patterns) accordingly. */
#define ORC_SCALE_F16 0x100
#define ORC_BITS_MASK 0xff

#ifdef __cplusplus
extern "C" {
#endif

/* binary16 <-> binary32, written from the IEEE 754 definitions. */
float    orc_half_to_float(uint16_t h);
uint16_t orc_float_to_half(float f); /* round to nearest, ties to even */
void     orc_half_to_float_n(const uint16_t* h, float* f, long n);
void     orc_float_to_half_n(const float* f, uint16_t* h, long n);

/* Tokens moved from the fp16 residual window into the quantized store when
 * the window holds n_res tokens. */
int orc_flush_count(int n_res, int residual_length, int group_size);

/* Quantize one group of n values (already widened to fp32). codes[i] is the
 * integer code of v[i]; *scale and *zero receive the group's parameters. */
void orc_quantize_group(const float* v, int n, int bits,
                        uint8_t* codes, float* scale, float* zero);

/* Pack / unpack n codes (n * bits a multiple of 8), low bits first. */
void orc_pack_codes(const uint8_t* codes, int n, int bits, uint8_t* packed);
void orc_unpack_codes(const uint8_t* packed, int n, int bits, uint8_t* codes);

/* Key flush: per-channel groups of G tokens. x is [BH, *, D] fp16 with
 * x_bh_stride tokens between heads; tokens [0, n_flush) are quantized and
 * written at store token offset s_off of a store with capacity s_cap. */
void orc_flush_keys(const uint16_t* x, int BH, int x_bh_stride, int n_flush,
                    int D, int G, int bits,
                    uint8_t* codes, void* kscale, uint16_t* kzero,
                    int s_off, int s_cap);

/* Value flush: per-token groups of G channels. Same arguments as above;
 * vscale / vzero are [BH, s_cap, D/G]. */
void orc_flush_values(const uint16_t* x, int BH, int x_bh_stride, int n_flush,
                      int D, int G, int bits,
                      uint8_t* codes, void* vscale, uint16_t* vzero,
                      int s_off, int s_cap);

/* Reconstruction of tokens [0, S) of the store, in fp32 (before the final
 * fp16 rounding) and in fp16. axis 0 = keys, 1 = values. out is [BH, S, D]. */
void orc_recon_f32(int axis, const uint8_t* codes, const void* scale,
                   const uint16_t* zero, int BH, int S, int D, int G, int bits,
                   int s_cap, float* out);
void orc_dequant(int axis, const uint8_t* codes, const void* scale,
                 const uint16_t* zero, int BH, int S, int D, int G, int bits,
                 int s_cap, uint16_t* out);

/* fp16 residual window [BH, res_cap, D]: append n_new tokens of src (with
 * src_bh_stride tokens between heads) at position n_res; drop the oldest
 * n_drop of n_res tokens, moving the rest to the front. */
void orc_residual_append(uint16_t* res, int BH, int res_cap, int D, int n_res,
                         const uint16_t* src, int src_bh_stride, int n_new);
void orc_residual_compact(uint16_t* res, int BH, int res_cap, int D, int n_res,
                          int n_drop);

/* Single-token decode over S_q store tokens followed by n_res residual
 * tokens, in float64. q [B, Hq, D] fp16; out [B, Hq, D] float64. */
void orc_decode_attend(const uint16_t* q,
                       const uint8_t* kcodes, const void* kscale, const uint16_t* kzero,
                       const uint8_t* vcodes, const void* vscale, const uint16_t* vzero,
                       int S_q, int s_cap,
                       const uint16_t* k_res, const uint16_t* v_res, int n_res, int res_cap,
                       int B, int Hq, int Hkv, int D, int G, int bits, double sm_scale,
                       double* out);

#ifdef __cplusplus
}
#endif
#endif

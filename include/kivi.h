/*
 * kivi.h -- C ABI of the GB300 (sm_103a) KIVI KV-cache library, libkivi_gb300.so.
 *
 * KIVI keeps a KV cache as asymmetric min/max 2- or 4-bit codes: keys are
 * quantized per channel (each group runs along the token axis), values per
 * token (each group runs along head_dim), and the newest residual_length
 * tokens stay in fp16. This library implements, as hand-written CUDA kernels:
 *   - the flush (quantize + bit-pack) of keys and of values,
 *   - the dequantize of the packed store back to fp16,
 *   - the fp16 residual window's append / compact,
 *   - a fused dequantize-and-attend single-token decode over the packed store
 *     plus the residual window (split over the cached tokens; the splits are
 *     merged by a log-sum-exp combine inside the same launch),
 *   - fake quantization: the quantize-then-dequantize fp16 tensor in one pass.
 *
 * Sources (page title, section):
 *   [F] VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly 0%
 *       Faster" -- the fused KIVI post.
 *   [Q] VeloxQuant-MLX blog, "A Kernel That Wasn't There" (Qwen3-8B on M4).
 *   [R] VeloxQuant-MLX benchmarks page, "KV-Cache Kernel Roofline".
 *
 * Conventions shared by every entry point
 *   - Ownership: the caller owns every buffer. The library never allocates
 *     device memory and keeps no state between calls (it caches the device's
 *     SM count per device for the split heuristic).
 *   - Pointers: device pointers (CUDA global memory), 16-byte aligned, unless
 *     stated otherwise. Scalars and *_out arguments are host values/pointers.
 *   - Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL
 *     is the legacy default stream). Results are ready when the stream is.
 *   - Errors: argument checks happen on the host before any launch; a failed
 *     check returns its status and launches nothing. A launch failure returns
 *     KIVI_ERR_CUDA (from cudaGetLastError). No call aborts, throws, traps or
 *     spins on the device.
 *   - Numbers: fp16 is IEEE binary16 passed as raw 16-bit words. Inputs must
 *     be finite; NaN/Inf inputs give unspecified codes but every access stays
 *     in bounds.
 *   - Supported shapes: bits in {2, 4}; group_size G in {32, 64, 128};
 *     head_dim D in {64, 128, 256} with G <= D (a value group lies within one
 *     token row), for every entry point. Other values return
 *     KIVI_ERR_UNSUPPORTED.
 *
 * Store layout (one store per tensor, keys and values separately):
 *   codes  uint8   [BH, s_cap, D*bits/8]  codes packed along D inside each
 *                                          token row, element i at bit offset
 *                                          i*bits, low bits first
 *   keys:   scale float32 [BH, s_cap/G, D]  zero fp16 [BH, s_cap/G, D]
 *   values: scale float32 [BH, s_cap, D/G]  zero fp16 [BH, s_cap, D/G]
 * with s_cap (the store's token capacity) a multiple of G. zero is the group
 * minimum (an fp16 input, so fp16 storage is lossless); scale is the fp32
 * value the codes were computed with.
 *
 * fp16 scale storage (KIVI_SCALE_F16): every `bits` argument may be ORed
 * with KIVI_SCALE_F16. The scale arrays then hold fp16 values (same shapes,
 * 2 bytes per element; pass them through the float* parameters by a pointer
 * cast). The flush rounds each fp32 scale (max - min) / (2^bits - 1) to the
 * nearest fp16 and computes the codes with that stored scale, so dequant and
 * decode reproduce exactly what the flush used: 4 instead of 6 bytes of
 * metadata per group. Consequences of the rounding: a group whose range is
 * below about 2^-25 * (2^bits - 1) stores scale 0 (every code 0, recon = min);
 * a subnormal fp16 scale can clip the largest codes at 2^bits - 1; and a
 * scale rounded up can reconstruct the group maximum past 65504 (fp16 inf in
 * a dequant) for inputs within one step of the fp16 range. A store is read
 * with the same option it was flushed with.
 */
#ifndef KIVI_GB300_H
#define KIVI_GB300_H

#include <stddef.h>

/* Option bit of every `bits` argument: scales stored as fp16 (see above). */
#define KIVI_SCALE_F16 0x100
/* Option bit of the decode's `bits` argument (kivi_decode_attend and
 * kivi_decode_attend_noalloc): the caller states that the kernel preceding
 * this call on `stream` does not write the store (codes, scales, zeros) the
 * decode reads -- e.g. the store was last flushed before that kernel, or
 * that kernel is an append to the residual window, a projection or another
 * layer's decode. The decode then requests its first store tiles before
 * waiting for that kernel to finish (the library launches every kernel with
 * programmatic dependent launch), so its first DRAM round trip overlaps the
 * preceding kernel's tail. q, the residual window and the workspace are
 * still read only after the wait. Results are identical with and without the
 * option; setting it when the preceding kernel does write the store (a flush
 * launched directly before the decode on the same stream) gives undefined
 * results. */
#define KIVI_DECODE_STORE_READY 0x200

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* kivi_stream_t;

typedef enum {
    KIVI_OK = 0,
    KIVI_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad offset/capacity */
    KIVI_ERR_UNSUPPORTED = 2,  /* D, G, bits or Hq/Hkv outside the compiled set */
    KIVI_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    KIVI_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    KIVI_ERR_ALIGNMENT = 5     /* a pointer is not 16-byte aligned */
} kivi_status;

typedef enum { KIVI_AXIS_KEYS = 0, KIVI_AXIS_VALUES = 1 } kivi_axis;

/* Human-readable name of a status. Never NULL; host only. */
const char* kivi_status_string(kivi_status status);

/* Library ABI version (major*100 + minor). */
int kivi_version(void);

/*
 * Waits that ran out. The flush stages its items of group size 32 and head
 * dim 128 with bulk tensor copies, each completing on a shared-memory
 * barrier that the warp polls a bounded number of times (well over a
 * second). A poll that runs out adds one to a device-wide count, and that
 * warp leaves its remaining items undone (their outputs are unspecified).
 * *count (host pointer) receives the count; reset != 0 sets it back to zero.
 * It is zero in correct operation. Synchronizes the device. Errors:
 * INVALID_ARG if count is NULL; CUDA if the device copy fails.
 */
kivi_status kivi_wait_timeouts(unsigned int* count, int reset);

/*
 * Flush plan ([F] "What we're actually optimizing": the newest
 * residual_length tokens stay fp16 and fresh tokens are quantized in a batch
 * once enough accumulate). Given a residual window holding n_res tokens,
 * returns how many of its oldest tokens to flush:
 *   residual_length == 0  -> n_res (quantize everything, ragged tail allowed)
 *   n_res - R <  G        -> 0
 *   otherwise             -> floor((n_res - R) / G) * G
 * so that afterwards R <= n_res < R + G. This reproduces the flush counts
 * printed in [F] "The full end-to-end record" (559 -> 512, 2059 -> 2016,
 * 8209 -> 8160 at R = G = 32 with 2048-token prefill chunks). Host only;
 * returns -1 for negative n_res, negative R or G <= 0.
 */
int kivi_flush_count(int n_res, int residual_length, int group_size);

/*
 * Key flush ([F] "The layout problem that shapes everything", "Kernel A",
 * "Three ways to be off by one bit"). x is fp16 [BH, S, D] row-major with
 * x_bh_stride tokens between consecutive heads (x_bh_stride >= S; pass S for a
 * dense tensor, or the capacity of a larger cache to flush a view of it).
 * n_flush = kivi_flush_count(S, residual_length, group_size) of the oldest
 * tokens [0, n_flush) are quantized per channel in groups of G consecutive
 * tokens (a ragged last group, possible only when residual_length == 0, uses
 * min/max over its real tokens):
 *     zero = min, scale = RN32(RN32(max - min) / (2^bits - 1)),
 *     q = clamp(rint(RN32(RN32(x - zero) / scale)), 0, 2^bits - 1)
 * (IEEE fp32 division, round half to even; scale == 0 gives q = 0), and
 * written at store token offset s_off (a multiple of G) of a key store of
 * capacity s_cap: codes[BH, s_cap, D*bits/8], scale f32 (fp16 with
 * KIVI_SCALE_F16) / zero fp16 [BH, s_cap/G, D]. Bit-exact with the CPU
 * oracle.
 * *n_flushed (host pointer, may be NULL) receives n_flush.
 * Errors: INVALID_ARG if S < 0, BH <= 0, x_bh_stride < S, s_cap % G != 0,
 * s_off % G != 0 or s_off + n_flush > s_cap; ALIGNMENT if a pointer is not
 * 16-byte aligned. n_flush == 0 returns KIVI_OK without a launch.
 */
kivi_status kivi_flush_keys(const void* x_f16, int BH, int S, int x_bh_stride, int D,
                            int group_size, int bits, int residual_length,
                            void* codes_u8, float* scale, void* zero_f16,
                            int s_off, int s_cap, int* n_flushed, kivi_stream_t stream);

/*
 * Value flush ([F] "The layout problem", "Kernel B"): as kivi_flush_keys,
 * but each group is G consecutive channels of one token; scale f32 (fp16
 * with KIVI_SCALE_F16) and zero fp16 are [BH, s_cap, D/G]. s_off need not be
 * a multiple of G here, but must satisfy s_off + n_flush <= s_cap.
 */
kivi_status kivi_flush_values(const void* x_f16, int BH, int S, int x_bh_stride, int D,
                              int group_size, int bits, int residual_length,
                              void* codes_u8, float* scale, void* zero_f16,
                              int s_off, int s_cap, int* n_flushed, kivi_stream_t stream);

/*
 * Key and value flush of the same tokens in one launch (both as above, same
 * n_flush). k and v share x_bh_stride. Bit-exact with the two calls above.
 */
kivi_status kivi_flush_kv(const void* k_f16, const void* v_f16, int BH, int S, int x_bh_stride,
                          int D, int group_size, int bits, int residual_length,
                          void* kcodes_u8, float* kscale, void* kzero_f16,
                          void* vcodes_u8, float* vscale, void* vzero_f16,
                          int s_off, int s_cap, int* n_flushed, kivi_stream_t stream);

/*
 * Dequantize ([F] "What we're actually optimizing" recon = q*scale + zero;
 * "Three ways to be off by one bit" #1: a multiply then a separate add, two
 * roundings, no FMA): tokens [0, S) of a store of capacity s_cap to fp16
 * out[BH, S, D]:  out = fp16_rn(RN32(RN32(q * scale) + zero)).
 * axis selects the key or value metadata layout; bits carries
 * KIVI_SCALE_F16 when the store holds fp16 scales. Bit-exact with the oracle.
 * Errors: INVALID_ARG if S < 0, S > s_cap or s_cap % G != 0.
 */
kivi_status kivi_dequant(kivi_axis axis, const void* codes_u8, const float* scale,
                         const void* zero_f16, int BH, int S, int D, int group_size, int bits,
                         int s_cap, void* out_f16, kivi_stream_t stream);

/*
 * Key and value dequantize in one launch (both as kivi_dequant, same S and
 * s_cap): kout from the key store, vout from the value store. Bit-exact with
 * two kivi_dequant calls.
 */
kivi_status kivi_dequant_kv(const void* kcodes_u8, const float* kscale, const void* kzero_f16,
                            const void* vcodes_u8, const float* vscale, const void* vzero_f16,
                            int BH, int S, int D, int group_size, int bits, int s_cap,
                            void* kout_f16, void* vout_f16, kivi_stream_t stream);

/*
 * fp16 residual window res[BH, res_cap, D] ([F] "What we're actually
 * optimizing": the newest tokens stay fp16).
 * append:  copies src[bh, t, :] (src_bh_stride tokens between heads) for
 *          t < n_new to res[bh, n_res + t, :]. INVALID_ARG if
 *          n_res + n_new > res_cap or src_bh_stride < n_new.
 * compact: drops the oldest n_drop of n_res tokens and moves the other
 *          n_res - n_drop to the front (overlap-safe). INVALID_ARG if
 *          n_drop > n_res or n_res > res_cap.
 * UNSUPPORTED unless D is 64, 128 or 256.
 */
kivi_status kivi_residual_append(const void* src_f16, int src_bh_stride, int n_new,
                                 void* res_f16, int BH, int res_cap, int D, int n_res,
                                 kivi_stream_t stream);
kivi_status kivi_residual_compact(void* res_f16, int BH, int res_cap, int D, int n_res,
                                  int n_drop, kivi_stream_t stream);

/* The same two operations on a key window and a value window of equal
 * geometry, in one launch each. */
kivi_status kivi_residual_append_kv(const void* k_src_f16, const void* v_src_f16, int src_bh_stride,
                                    int n_new, void* k_res_f16, void* v_res_f16, int BH, int res_cap,
                                    int D, int n_res, kivi_stream_t stream);
kivi_status kivi_residual_compact_kv(void* k_res_f16, void* v_res_f16, int BH, int res_cap, int D,
                                     int n_res, int n_drop, kivi_stream_t stream);

/*
 * Fake quantization ([F] "What we're actually optimizing": the pages' kernels
 * write the quantize-then-dequantize fp16 tensor; "So why does the kernel
 * ship?"). For the tokens a flush would quantize, n = kivi_flush_count(S,
 * residual_length, group_size), out[bh, t, :] = fp16(RN(RN(q * scale) + zero))
 * with q, scale and zero exactly those of kivi_flush_keys (per-channel
 * groups along the tokens) or kivi_flush_values (per-token groups along D):
 * bit-identical to kivi_dequant of the flushed store. Tokens [n, S) are copied
 * unchanged. Nothing else is written: no codes, scales or zeros.
 * x: fp16 [BH, S, D] with a head stride of x_bh_stride tokens; out: fp16
 * [BH, S, D] with a head stride of out_bh_stride tokens. out may be x itself
 * (in place, same stride); otherwise it must not overlap x.
 * Errors: as kivi_flush_keys; INVALID_ARG if out == x with another stride.
 * *n_quantized (may be NULL) receives n.
 */
kivi_status kivi_fake_quant_keys(const void* x_f16, int BH, int S, int x_bh_stride, int D,
                                 int group_size, int bits, int residual_length, void* out_f16,
                                 int out_bh_stride, int* n_quantized, kivi_stream_t stream);
kivi_status kivi_fake_quant_values(const void* x_f16, int BH, int S, int x_bh_stride, int D,
                                   int group_size, int bits, int residual_length, void* out_f16,
                                   int out_bh_stride, int* n_quantized, kivi_stream_t stream);
/* Keys and values of equal geometry in one launch (plus one for the copies). */
kivi_status kivi_fake_quant_kv(const void* k_f16, const void* v_f16, int BH, int S, int x_bh_stride,
                               int D, int group_size, int bits, int residual_length,
                               void* k_out_f16, void* v_out_f16, int out_bh_stride,
                               int* n_quantized, kivi_stream_t stream);

/*
 * Bytes of device workspace kivi_decode_attend needs for these sizes on the
 * current device, for any bit width, group size and scale storage (the
 * split count depends on the device's SM count, the bit width and the kernel
 * these select; the partials hold D floats per split). Returns
 * 0 when the decode runs as a single split per (batch, KV head) and needs no
 * workspace, and 0 for invalid sizes. Host only (reads the device's SM count
 * once).
 *
 * Workspace layout: the first KIVI_DECODE_COUNTER_BYTES bytes hold the merge
 * counters of the split decode, one per head group (batch, KV head, and
 * sub-group of up to 4 query heads when Hq/Hkv is not 1, 2 or 4); the split partials
 * follow. The counters must be zero before a workspace's first use
 * (kivi_decode_workspace_init, or any zero fill), and every completed call
 * leaves them zero again, whatever its sizes. The rest of the workspace is
 * scratch whose contents on entry are ignored. One workspace serves one call
 * at a time: calls whose kernels may overlap need distinct workspaces.
 */
#define KIVI_DECODE_COUNTER_BYTES 32768u
size_t kivi_decode_workspace_size(int B, int Hq, int Hkv, int S_q, int n_res, int D);

/*
 * The split plan kivi_decode_attend takes for these arguments (bits may carry
 * KIVI_SCALE_F16), for inspection and capacity planning. Host only; reads the
 * device's SM count once. info (host, 7 ints) receives:
 *   [0] kernel: 0 one warp per tile, 1 warp pairs (small batches; group size
 *       32, head dim 128, fp32 scales, 1, 2 or 4 query heads per KV head)
 *   [1] n_split: CTAs per head group, merged in the same launch
 *   [2] tiles per warp (per warp pair for the pair kernel)
 *   [3] warps per CTA (2, 4 or 8; the pair kernel: 8, four pairs)
 *   [4] query sub-groups per KV head (1, or ceil(Hq/Hkv / 4))
 *   [5] tiles per head group: ceil(S_q / 32) store + ceil(n_res / 16) residual
 *   [6] tiles per split
 * Errors: as kivi_decode_attend's argument checks (no pointers but info).
 */
kivi_status kivi_decode_plan_info(int B, int Hq, int Hkv, int S_q, int n_res, int D, int group_size, int bits,
                                  int* info);

/*
 * Zero the merge counters of a fresh decode workspace: the first
 * min(workspace_bytes, KIVI_DECODE_COUNTER_BYTES) bytes, by an asynchronous
 * memset on `stream`. Needed once per workspace, before its first decode.
 * INVALID_ARG if workspace is NULL and workspace_bytes > 0.
 */
kivi_status kivi_decode_workspace_init(void* workspace, size_t workspace_bytes, kivi_stream_t stream);

/*
 * Fused dequantize-and-attend single-token decode ([F] "So why does the kernel
 * ship?": attention reads the packed codes and expands them in registers;
 * [R] "KV-Cache Kernel Roofline": one query token per head). For each batch
 * b and query head h, with KV head hk = h / (Hq / Hkv) (grouped-query
 * attention, query heads of a group contiguous -- [Q] "Picking a model"):
 *     K_t = fp32 recon of store token t (t < S_q), else k_res[t - S_q]
 *     score_t = sm_scale * sum_d q[b,h,d] * K_t[d]
 *     out[b,h,:] = sum_t softmax(score)_t * V_t[:]
 * over all S_q + n_res tokens (no mask). Stores are those of
 * kivi_flush_keys / kivi_flush_values with BH = B*Hkv and capacity s_cap;
 * residuals are fp16 [B*Hkv, res_cap, D]. q fp16 [B, Hq, D]; out f32
 * [B, Hq, D]. Accumulation is fp32; max-abs error against the float64 oracle
 * is well below 2e-3 for inputs of unit scale.
 * workspace: device memory of at least kivi_decode_workspace_size(...) bytes,
 * laid out and initialised as described there (may be NULL when that size is
 * 0).
 * Errors: INVALID_ARG if S_q + n_res == 0, S_q > s_cap, n_res > res_cap or
 * Hq % Hkv != 0; UNSUPPORTED if Hq/Hkv > 64, or D, group_size or bits as for
 * the flush; WORKSPACE if the workspace is NULL or too small. Stores of
 * every supported group size (32, 64, 128) are read; their key groups align
 * with the kernels' 32-token tiles.
 */
kivi_status kivi_decode_attend(const void* q_f16,
                               const void* kcodes_u8, const float* kscale, const void* kzero_f16,
                               const void* vcodes_u8, const float* vscale, const void* vzero_f16,
                               int S_q, int s_cap,
                               const void* k_res_f16, const void* v_res_f16, int n_res, int res_cap,
                               int B, int Hq, int Hkv, int D, int group_size, int bits,
                               float sm_scale, float* out_f32,
                               void* workspace, size_t workspace_bytes, kivi_stream_t stream);

/*
 * One attention layer's KIVI cache ([F] "What we're actually optimizing":
 * the newest residual_length tokens stay fp16, and the oldest whole groups
 * are quantized into the packed store once enough accumulate; [F] "Four
 * benchmarks that lied", Lie #2, counts those flushes per decode run). The
 * struct holds the geometry, the caller-owned device buffers and two host
 * counters; the calls below sequence the library's kernels and update the
 * counters. The caller owns the struct and every buffer.
 *   stores:  as kivi_flush_keys / kivi_flush_values, BH heads, capacity s_cap
 *            (a multiple of group_size) tokens;
 *   windows: fp16 [BH, res_cap, D] for keys and for values, with
 *            res_cap >= residual_length + group_size;
 *   S_q:     tokens in the stores (set 0 for an empty cache);
 *   n_res:   tokens in the windows, oldest first (set 0 for an empty cache);
 *   res_off: the window's first row: its tokens are rows res_off ..
 *            res_off + n_res - 1 of each head (set 0 for an empty cache).
 * Invariant kept by the calls: after each call, n_res < residual_length +
 * group_size (a window that reaches R + G tokens flushes its oldest
 * floor((n_res - R) / G) * G tokens into the stores at offset S_q; the
 * window then starts that many rows later). The window moves back to row 0
 * only when new tokens would not fit behind it, so with res_cap = R + kG
 * the remaining tokens are copied once per about k - 1 flushes instead of
 * after every flush.
 * Errors: every argument check (geometry, counters, pointers and alignment,
 * store capacity for every flush the call will make) runs before the call's
 * first launch; a failed check returns its status, launches nothing and
 * leaves the counters unchanged. After a KIVI_ERR_CUDA the counters describe
 * the launches that succeeded.
 */
typedef struct {
    int BH;               /* sequences times KV heads */
    int D;                /* head dim: 64, 128 or 256 */
    int group_size;       /* 32, 64 or 128 (<= D) */
    int bits;             /* 2 or 4, optionally ORed with KIVI_SCALE_F16 */
    int residual_length;  /* R: fp16 tokens kept after a flush */
    int s_cap;            /* store capacity in tokens */
    int res_cap;          /* window capacity in tokens */
    void* kcodes;         /* key store */
    float* kscale;
    void* kzero;
    void* vcodes;         /* value store */
    float* vscale;
    void* vzero;
    void* k_res;          /* fp16 windows */
    void* v_res;
    int S_q;              /* tokens in the stores */
    int n_res;            /* tokens in the windows */
    int store_written;    /* 1 when the cache's latest launch wrote the stores (set 0 for an empty cache) */
    int res_off;          /* first window row in use (set 0 for an empty cache) */
} kivi_cache;

/*
 * Prefill into a cache whose windows are empty (n_res == 0): of the S tokens
 * of k and v ([BH, S, D] fp16, x_bh_stride tokens between heads), the oldest
 * n = kivi_flush_count(S, residual_length, group_size) are flushed straight
 * from k and v into the stores at offset S_q (one launch), and the other
 * S - n are copied into rows 0 .. S - n - 1 of the windows. S_q += n,
 * n_res = S - n, res_off = 0; *n_flushed
 * (may be NULL) receives n. With residual_length 0 and S not a multiple of
 * group_size the last key group is ragged and the cache takes no further
 * flushes (their store offset would not be a multiple of group_size).
 * Errors: INVALID_ARG if n_res != 0, S < 0, x_bh_stride < S, the stores
 * lack room, or a flush would start at an offset that is not a multiple of
 * group_size.
 */
kivi_status kivi_cache_prefill(kivi_cache* cache, const void* k_f16, const void* v_f16, int x_bh_stride, int S,
                               int* n_flushed, kivi_stream_t stream);

/*
 * Append n_new tokens (k, v: [BH, n_new, D] fp16, src_bh_stride tokens
 * between heads) to the windows, oldest first, flushing as the rule above
 * says. The tokens enter in pieces that fit the windows, each followed by
 * the flush it triggers (one piece when res_cap >= residual_length +
 * group_size + n_new). *n_flushed (may be NULL) receives the tokens flushed.
 * One decode step of a serving loop is kivi_cache_append of one token
 * followed by kivi_cache_decode.
 * Errors: INVALID_ARG if n_new < 0, src_bh_stride < n_new, or a flush would
 * overrun the stores or start at an offset that is not a multiple of
 * group_size.
 */
kivi_status kivi_cache_append(kivi_cache* cache, const void* k_f16, const void* v_f16, int src_bh_stride,
                              int n_new, int* n_flushed, kivi_stream_t stream);

/*
 * kivi_decode_attend over the cache's S_q store tokens and n_res window
 * tokens, for B sequences with Hkv KV heads (B * Hkv == BH) and Hq query
 * heads; every other argument, check and result is that of
 * kivi_decode_attend. The counters are not changed. Unless the cache's
 * latest launch wrote the stores (store_written: a flush that no window
 * append or move followed), the decode takes KIVI_DECODE_STORE_READY: the calls
 * on one cache are meant to be issued on one stream, and a flush followed by
 * any other kernel has finished before the decode's first loads.
 */
kivi_status kivi_cache_decode(const kivi_cache* cache, const void* q_f16, int B, int Hq, int Hkv, float sm_scale,
                              float* out_f32, void* workspace, size_t workspace_bytes, kivi_stream_t stream);

/*
 * kivi_decode_attend_noalloc -- the same decode as kivi_decode_attend, for
 * callers that cannot allocate device memory when they decode: serving
 * runtimes that hand out all of HBM to weights and KV-cache pages at start-up
 * and forbid later allocations (a late cudaMalloc may fail, or synchronise the
 * whole device), and C callers that only receive device pointers from a
 * framework owning the memory pool. The pages have no counterpart; this is an
 * interface addition of this library.
 *
 * Instead of a workspace argument it uses one library-owned device array of
 * KIVI_NOALLOC_SCRATCH_BYTES (8 MiB) per device, reserved when the library's
 * device code is loaded and kept until the process exits. It allocates
 * nothing itself.
 *   - Size limit: if the workspace of the split plan this call takes (for
 *     its bit width, group size and scale storage) exceeds
 *     KIVI_NOALLOC_SCRATCH_BYTES, it returns KIVI_ERR_WORKSPACE and launches
 *     nothing. The plan's split count grows with the device's SM count; on a
 *     152-SM GB300 with the library's default planner settings no supported
 *     shape needs more than about 6.1 MB (head dim 256), 3.1 MB (128) or
 *     1.6 MB (64). A device with more SMs may reject the widest shapes.
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's contents. Calls whose kernels overlap on the GPU (two
 *     unordered streams) race and give wrong results; order them.
 *   - Its merge counters start at zero (the array is zero-initialised when
 *     the device code loads) and every completed call leaves them zero.
 *   - Address: host code cannot use the array's name as a device address, so
 *     every call made outside stream capture looks it up with
 *     cudaGetSymbolAddress (the current device must be the one the pointers
 *     belong to); after cudaDeviceReset the reloaded array is found at its
 *     new address. A call made while `stream` is being captured uses the
 *     address the last uncaptured call on that device found, so make one call
 *     per device before capturing any stream (the first call may also load
 *     the library's device code). KIVI_ERR_CUDA if no address is known or the
 *     lookup fails.
 * Every other argument, check, status and result is that of
 * kivi_decode_attend.
 */
#define KIVI_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
kivi_status kivi_decode_attend_noalloc(const void* q_f16,
                                       const void* kcodes_u8, const float* kscale, const void* kzero_f16,
                                       const void* vcodes_u8, const float* vscale, const void* vzero_f16,
                                       int S_q, int s_cap,
                                       const void* k_res_f16, const void* v_res_f16, int n_res, int res_cap,
                                       int B, int Hq, int Hkv, int D, int group_size, int bits,
                                       float sm_scale, float* out_f32, kivi_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* KIVI_GB300_H */

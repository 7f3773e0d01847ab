// kivi_launch.h -- internal launch interface between the C ABI (kivi_api.cu)
// and the kernels. Arguments are validated by the caller; launchers only
// pick a grid and launch on the given stream.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kivi {

constexpr int kD = 128;  // head dim of the decode (the flush, dequant and residual also take 64 and 256)
constexpr int kG = 32;   // the default group size

struct FlushArgs {
    const __half* x;      // [BH, x_bh_stride, D], tokens [0, n_flush) used
    long long x_bh_stride;
    int BH;
    int n_flush;
    uint8_t* codes;       // [BH, s_cap, D*bits/8]
    float* scale;         // keys [BH, s_cap/G, D]; values [BH, s_cap, D/G]; __half elements if scale_f16
    __half* zero;
    int s_off;
    int s_cap;
    __half* fq = nullptr;      // fake quantization: fp16 reconstructions [BH, fq_bh_stride, D] instead of a store
    long long fq_bh_stride = 0;
    int G = kG;                // group size: 32, 64 or 128
    int D = kD;                // head dim: 64, 128 or 256 (G <= D)
    bool scale_f16 = false;    // scales stored as fp16 (codes computed with the stored scale)
};

struct DequantArgs {
    const uint8_t* codes;
    const float* scale;
    const __half* zero;
    int BH;
    int S;
    int s_cap;
    __half* out;          // [BH, S, D]
    int G = kG;           // group size: 32, 64 or 128
    int D = kD;           // head dim: 64, 128 or 256 (G <= D)
    bool scale_f16 = false;  // scales stored as fp16
};

struct DecodeArgs {
    const __half* q;      // [B, Hq, D]
    const uint8_t* kcodes;
    const float* kscale;
    const __half* kzero;
    const uint8_t* vcodes;
    const float* vscale;
    const __half* vzero;
    int S_q;
    int s_cap;
    int g_shift;          // log2(G / 32): the store's group size is 32, 64 or 128
    int D = kD;           // head dim: 64, 128 or 256 (the warp-pair kernel: 128)
    int scale_f16 = 0;    // 1: scales stored as fp16 (the warp-pair kernel: fp32 only)
    const __half* k_res;  // [B*Hkv, res_cap, D]
    const __half* v_res;
    int n_res;
    int res_cap;
    int B;
    int Hq;
    int Hkv;
    float score_scale;    // sm_scale * log2(e): scores live in the exp2 domain
    int n_split;
    int tiles_per_split;  // planned tiles per split (the kernels spread n_tiles evenly)
    int tiles_per_warp;   // planned tiles per warp of the one-warp-per-tile kernel
    int warps_per_cta;    // one-warp-per-tile kernel: 2 (head dim 128 only), 4 or 8
    int pair_kernel;      // 1: groups of 1, 2 or 4 heads run the warp-pair kernel
    int n_store_tiles;
    int n_tiles;
    int q_sub;            // one-warp-per-tile kernel: query sub-groups of up to 4 heads per KV head
    int store_ready = 0;  // 1: the store is not written by the preceding kernel on the stream, so its first
                          // tiles may be requested before griddepcontrol.wait
    unsigned int* counters;  // [B*Hkv*q_sub] merge tickets, zero between calls (n_split > 1)
    float* part_o;        // [B, Hq, n_split, D]
    float* part_ml;       // [B, Hq, n_split, 2]  (running max, running sum)
    float* out;           // [B, Hq, D]
};

struct DecodePlan {
    int n_split;
    int tiles_per_split;
    int tiles_per_warp;
    int warps_per_cta;
    int pair_kernel;
    int n_store_tiles;
    int n_tiles;
    int q_sub;
};

// Tokens per residual tile of the decode kernels.
constexpr int kResTileTokensMma = 16;
constexpr int kMergeCounters = 8192;    // (batch, KV head, sub-group) CTA groups that can take split merges
constexpr int kMaxClusterSplits = 16;   // splits of one head merged inside a thread-block cluster
#ifndef KIVI_PAIRS_PER_CTA
#define KIVI_PAIRS_PER_CTA 4
#endif
constexpr int kPairsPerCta = KIVI_PAIRS_PER_CTA;  // warp pairs per CTA of the warp-pair kernel

// Launch with programmatic stream serialization allowed: the kernel may start
// while the previous kernel on the stream finishes; it must (and every kernel
// of this library does) execute griddepcontrol.wait before touching memory.
template <typename... Exp, typename... Act>
inline cudaError_t launch_pdl(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Act&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Act&&>(args)...);
}

// The same launch with the grid's x dimension cut into thread-block clusters
// of cluster_x CTAs.
template <typename... Exp, typename... Act>
inline cudaError_t launch_pdl_cluster(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t stream, unsigned cluster_x, Act&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Act&&>(args)...);
}

// KIVI_OK (0), or KIVI_ERR_UNSUPPORTED for a head dim, group size or bit
// width (bits may carry KIVI_SCALE_F16) outside the compiled set.
int shape_status(int D, int group_size, int bits);

// Streaming multiprocessors of the current device (152 when no device is
// visible), read once per device.
int sm_count();

// Workspace bytes of the exact plan kivi_decode_attend takes for these
// arguments (bits may carry KIVI_SCALE_F16); 0 for a single-split plan or
// for arguments the decode rejects. kivi_decode_workspace_size is the
// largest of these over bit widths, group sizes and scale storage.
size_t decode_workspace_need(int B, int Hq, int Hkv, int S_q, int n_res, int D, int group_size, int bits);

cudaError_t launch_flush(int axis, const FlushArgs& a, int bits, cudaStream_t stream);
cudaError_t launch_flush_kv(const FlushArgs& k, const FlushArgs& v, int bits, cudaStream_t stream);
// fake quantization (k.fq / v.fq set): the first n_flush tokens of x become
// their KIVI reconstructions in fq; keys if do_k, values if do_v, one launch
cudaError_t launch_fake_quant(const FlushArgs& k, const FlushArgs& v, bool do_k, bool do_v, int bits,
                              cudaStream_t stream);
// The count of bounded waits on a bulk copy that ran out (flush.cu), and
// optionally reset it. Synchronous.
cudaError_t read_wait_timeouts(unsigned int* count, bool reset);
cudaError_t launch_dequant(int axis, const DequantArgs& a, int bits, cudaStream_t stream);
cudaError_t launch_dequant_kv(const DequantArgs& k, const DequantArgs& v, int bits, cudaStream_t stream);
// src1/res1 may be null (one tensor); otherwise both pairs are handled in one launch
cudaError_t launch_residual_append(const __half* src0, const __half* src1, long long src_bh_stride,
                                   int n_new, __half* res0, __half* res1, int BH, int res_cap, int n_res, int D,
                                   cudaStream_t stream);
cudaError_t launch_residual_compact(__half* res0, __half* res1, int BH, int res_cap, int n_res, int n_drop, int D,
                                    cudaStream_t stream);
// Fused decodes; each merges its own splits in the same launch.
// One warp per tile: gq in {1, 2, 4}, or any other gq in a.q_sub sub-groups of
// up to 4 query heads; stores of group size 32, 64 or 128; head dim a.D of 64,
// 128 or 256, fp32 or fp16 scales (the suffixed forms serve one head dim and
// scale storage each).
cudaError_t launch_decode_mma(const DecodeArgs& a, int bits, int gq, cudaStream_t stream);
cudaError_t launch_decode_mma_d128_f16s(const DecodeArgs& a, int bits, int gq, cudaStream_t stream);
cudaError_t launch_decode_mma_d64(const DecodeArgs& a, int bits, int gq, cudaStream_t stream);
cudaError_t launch_decode_mma_d256(const DecodeArgs& a, int bits, int gq, cudaStream_t stream);
cudaError_t launch_decode_mma_d256_f16s(const DecodeArgs& a, int bits, int gq, cudaStream_t stream);
// gq in {1, 2, 4}: two warps per tile, 4 warp pairs per CTA (small batches);
// stores of group size 32 only.
cudaError_t launch_decode_pair(const DecodeArgs& a, int bits, int gq, cudaStream_t stream);

}  // namespace kivi

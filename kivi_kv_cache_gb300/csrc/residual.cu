// residual.cu -- the fp16 residual window of the newest tokens (VeloxQuant-MLX
// blog, "A 5.65x Metal Kernel That Made My LLM Exactly 0% Faster", "What
// we're actually optimizing": the most recent residual_length tokens stay in
// fp16 until a flush folds the oldest whole groups into the packed store).
//
// append:  16-byte vector copy of new token rows behind the n_res live ones.
// compact: after a flush of the oldest n_drop tokens, move the rest to the
//          front. Source and destination overlap inside one head's window,
//          so one CTA per head moves it in chunks: every chunk is read into
//          registers, the CTA synchronises, then the chunk is written. Later
//          chunks only read addresses above everything written so far.
#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi {

namespace {

constexpr int kThreads = 256;

// vpr = 16-byte vectors per fp16 token row (D / 8).
// blockIdx.y = head, blockIdx.z = tensor (0: first, 1: second of a K/V pair)
__global__ void __launch_bounds__(kThreads) residual_append_kernel(
    const uint4* __restrict__ src0, const uint4* __restrict__ src1, long long src_bh_stride, int n_new,
    uint4* __restrict__ res0, uint4* __restrict__ res1, int res_cap, int n_res, int vpr) {
    pdl_wait();
    const int bh = blockIdx.y;
    const uint4* src = blockIdx.z ? src1 : src0;
    uint4* res = blockIdx.z ? res1 : res0;
    const int total = n_new * vpr;
    const uint4* s = src + (long long)bh * src_bh_stride * vpr;
    uint4* d = res + ((long long)bh * res_cap + n_res) * vpr;
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < total; i += gridDim.x * kThreads) d[i] = __ldg(s + i);
    pdl_trigger();
}

constexpr int kChunkVec = kThreads * 4;  // vectors moved per chunk (64 token rows at D = 128)

// blockIdx.x = head, blockIdx.y = tensor of a K/V pair
__global__ void __launch_bounds__(kThreads) residual_compact_kernel(
    uint4* res0, uint4* res1, int res_cap, int n_res, int n_drop, int vpr) {
    pdl_wait();
    const int bh = blockIdx.x;
    uint4* base = (blockIdx.y ? res1 : res0) + (long long)bh * res_cap * vpr;
    const int total = (n_res - n_drop) * vpr;
    const int from = n_drop * vpr;
    for (int c0 = 0; c0 < total; c0 += kChunkVec) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = c0 + k * kThreads + threadIdx.x;
            if (i < total) v[k] = base[from + i];
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = c0 + k * kThreads + threadIdx.x;
            if (i < total) base[i] = v[k];
        }
    }
}

}  // namespace

cudaError_t launch_residual_append(const __half* src0, const __half* src1, long long src_bh_stride,
                                   int n_new, __half* res0, __half* res1, int BH, int res_cap, int n_res, int D,
                                   cudaStream_t stream) {
    if (n_new <= 0 || BH <= 0) return cudaSuccess;
    const int vpr = D / 8;
    const int total = n_new * vpr;
    const int bx = (total + kThreads - 1) / kThreads < 64 ? (total + kThreads - 1) / kThreads : 64;
    const int nt = src1 ? 2 : 1;
    for (int h0 = 0; h0 < BH; h0 += 65535) {
        const int nh = BH - h0 < 65535 ? BH - h0 : 65535;
        const long long so = (long long)h0 * src_bh_stride * D, ro = (long long)h0 * res_cap * D;
        cudaError_t e = launch_pdl(residual_append_kernel, dim3(bx, nh, nt), kThreads, 0, stream,
                                   reinterpret_cast<const uint4*>(src0 + so),
                                   reinterpret_cast<const uint4*>(src1 ? src1 + so : src0 + so),
                                   src_bh_stride, n_new, reinterpret_cast<uint4*>(res0 + ro),
                                   reinterpret_cast<uint4*>(res1 ? res1 + ro : res0 + ro), res_cap, n_res, vpr);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_residual_compact(__half* res0, __half* res1, int BH, int res_cap, int n_res, int n_drop, int D,
                                    cudaStream_t stream) {
    if (n_drop == 0 || n_res - n_drop <= 0 || BH <= 0) return cudaSuccess;
    const int nt = res1 ? 2 : 1;
    for (int h0 = 0; h0 < BH; h0 += 65535) {
        const int nh = BH - h0 < 65535 ? BH - h0 : 65535;
        const long long ro = (long long)h0 * res_cap * D;
        cudaError_t e = launch_pdl(residual_compact_kernel, dim3(nh, nt), kThreads, 0, stream,
                                   reinterpret_cast<uint4*>(res0 + ro),
                                   reinterpret_cast<uint4*>(res1 ? res1 + ro : res0 + ro), res_cap, n_res,
                                   n_drop, D / 8);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace kivi

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
constexpr int kVecPerRow = kD / 8;  // 16-byte vectors per fp16 token row

__global__ void __launch_bounds__(kThreads) residual_append_kernel(
    const uint4* __restrict__ src, long long src_bh_stride, int n_new,
    uint4* __restrict__ res, int BH, int res_cap, int n_res) {
    const long long total = (long long)BH * n_new * kVecPerRow;
    for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < total;
         i += (long long)gridDim.x * kThreads) {
        const int c = (int)(i % kVecPerRow);
        const long long r = i / kVecPerRow;
        const int bh = (int)(r / n_new);
        const int t = (int)(r - (long long)bh * n_new);
        res[((long long)bh * res_cap + n_res + t) * kVecPerRow + c] =
            __ldg(src + ((long long)bh * src_bh_stride + t) * kVecPerRow + c);
    }
}

constexpr int kChunkVec = kThreads * 4;  // vectors moved per chunk (64 token rows)

__global__ void __launch_bounds__(kThreads) residual_compact_kernel(
    uint4* res, int res_cap, int n_res, int n_drop) {
    const int bh = blockIdx.x;
    uint4* base = res + (long long)bh * res_cap * kVecPerRow;
    const int total = (n_res - n_drop) * kVecPerRow;
    const int from = n_drop * kVecPerRow;
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

cudaError_t launch_residual_append(const __half* src, long long src_bh_stride, int n_new,
                                   __half* res, int BH, int res_cap, int n_res, cudaStream_t stream) {
    const long long total = (long long)BH * n_new * kVecPerRow;
    if (total <= 0) return cudaSuccess;
    long long blocks = (total + kThreads - 1) / kThreads;
    if (blocks > 65535LL * 16) blocks = 65535LL * 16;
    residual_append_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(src), src_bh_stride, n_new,
        reinterpret_cast<uint4*>(res), BH, res_cap, n_res);
    return cudaGetLastError();
}

cudaError_t launch_residual_compact(__half* res, int BH, int res_cap, int n_res, int n_drop,
                                    cudaStream_t stream) {
    if (n_drop == 0 || n_res - n_drop <= 0 || BH <= 0) return cudaSuccess;
    residual_compact_kernel<<<BH, kThreads, 0, stream>>>(reinterpret_cast<uint4*>(res), res_cap,
                                                         n_res, n_drop);
    return cudaGetLastError();
}

}  // namespace kivi

// decode_mma_d64.cu -- the one-warp-per-tile fused decode at head dim 64
// (fp32 or fp16 scales).
#include "decode_mma.cuh"

namespace kivi {

cudaError_t launch_decode_mma_d64(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    return a.scale_f16 ? launch_decode_mma_impl<64, true>(a, bits, gq, stream)
                       : launch_decode_mma_impl<64, false>(a, bits, gq, stream);
}

}  // namespace kivi

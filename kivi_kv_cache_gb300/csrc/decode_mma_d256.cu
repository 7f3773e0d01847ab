// decode_mma_d256.cu -- the one-warp-per-tile fused decode at head dim 256
// with fp32 scales.
#include "decode_mma.cuh"

namespace kivi {

cudaError_t launch_decode_mma_d256(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    return launch_decode_mma_impl<256, false>(a, bits, gq, stream);
}

}  // namespace kivi

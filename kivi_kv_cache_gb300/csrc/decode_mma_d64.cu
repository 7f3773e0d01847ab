// decode_mma_d64.cu -- the one-warp-per-tile fused decode at head dim 64.
#include "decode_mma.cuh"

namespace kivi {

cudaError_t launch_decode_mma_d64(const DecodeArgs& a, int bits, int gq, cudaStream_t stream) {
    return launch_decode_mma_impl<64>(a, bits, gq, stream);
}

}  // namespace kivi
